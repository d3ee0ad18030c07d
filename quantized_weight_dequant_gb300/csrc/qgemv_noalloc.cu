// qgemv_run_noalloc: the split-K streaming GEMV for callers that cannot allocate device
// memory, with its scratch (column sums and per-range counters) in fixed file-scope device
// arrays instead of a handle's workspace.  See include/qgemv.h.  No error word: the kernel
// writes one only for the stall test hook, which this entry point never sets.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "../../include/qgemv.h"
#include "qgemv_stream.cuh"

namespace qg {
const void* stream_kernel_q4k(int R, int D);
const void* stream_kernel_q5k(int R, int D);
const void* stream_kernel_q6k(int R, int D);
const void* stream_kernel_q80(int R, int D);
const void* stream_kernel_tq10(int R, int D);
const void* stream_kernel_nvfp4(int R, int D);
}  // namespace qg

namespace {

using namespace qg;

constexpr int kMaxDevices = 64;
constexpr int kMaxRanges = 1024;
constexpr int kMaxWarps = 16;

// The scratch.  Every GPU that loads the library holds these arrays until the process
// exits; every call on a device shares them.
static __device__ __align__(256) float g_noalloc_ws[QGEMV_NOALLOC_MAX_COLUMN_SUMS];
static __device__ __align__(256) int g_noalloc_cnt[kMaxRanges];

struct DeviceSetup {
  bool ready = false;
  int sms = 0;
  size_t dyn_smem_max[6][3][3] = {};  // [format][R 1/2/4][D 2/3/4]
  float* ws = nullptr;                 // device addresses of the arrays above
  int* cnt = nullptr;
};

std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];

const void* kernel_for(int f, int R, int D) {
  switch (f) {
    case F_Q4K: return stream_kernel_q4k(R, D);
    case F_Q5K: return stream_kernel_q5k(R, D);
    case F_Q6K: return stream_kernel_q6k(R, D);
    case F_Q80: return stream_kernel_q80(R, D);
    case F_TQ10: return stream_kernel_tq10(R, D);
    case F_NVFP4: return stream_kernel_nvfp4(R, D);
  }
  return nullptr;
}

int sb_bytes(int f) {
  switch (f) {
    case F_Q4K: return 144;
    case F_Q5K: return 176;
    case F_Q6K: return 210;
    case F_Q80: return 272;
    case F_TQ10: return 54;
    case F_NVFP4: return 128;
  }
  return 0;
}

// Once per device, with that device current: kernel attributes and the device addresses of
// the scratch arrays (host code cannot use the arrays' names as device pointers).
qgemv_status_t setup(int dev, DeviceSetup** out) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  DeviceSetup& s = g_setup[dev];
  if (!s.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return QGEMV_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return QGEMV_ERR_NO_DEVICE;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&s.ws), g_noalloc_ws) != cudaSuccess ||
        cudaGetSymbolAddress(reinterpret_cast<void**>(&s.cnt), g_noalloc_cnt) != cudaSuccess) {
      cudaGetLastError();
      return QGEMV_ERR_CUDA;
    }
    const int Rs[3] = {1, 2, 4};
    for (int f = 0; f <= 5; ++f)
      for (int ri = 0; ri < 3; ++ri)
        for (int D = 2; D <= 4; ++D) {
          const void* fn = kernel_for(f, Rs[ri], D);
          cudaFuncAttributes fa;
          if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) {
            cudaGetLastError();
            return QGEMV_ERR_CUDA;
          }
          const size_t mx = prop.sharedMemPerBlockOptin - std::min(prop.sharedMemPerBlockOptin, fa.sharedSizeBytes);
          if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(mx)) !=
              cudaSuccess) {
            cudaGetLastError();
            return QGEMV_ERR_CUDA;
          }
          s.dyn_smem_max[f][ri][D - 2] = mx;
        }
    s.sms = prop.multiProcessorCount;
    s.ready = true;
  }
  *out = &s;
  return QGEMV_OK;
}

}  // namespace

extern "C" qgemv_status_t qgemv_run_noalloc(qgemv_format_t fmt, const void* x, const void* packed_W, int64_t N,
                                            int64_t K, float* y, cudaStream_t stream) {
  const int f = static_cast<int>(fmt);
  if (f < 0 || f > 5) return QGEMV_ERR_UNSUPPORTED_FORMAT;
  if (!x || !packed_W || !y) return QGEMV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(packed_W) | reinterpret_cast<uintptr_t>(y)) & 15)
    return QGEMV_ERR_MISALIGNED;
  // The streaming kernel's shape rule: whole 256-element superblocks, rows a multiple of
  // 16 bytes, at most 16 K-columns of 2048.
  if (N < 1 || K < 256 || K % 256 || K > 32768) return QGEMV_ERR_BAD_SHAPE;
  const int64_t nsb = K / 256;
  const int64_t rb1 = (f == F_NVFP4) ? K / 2 : nsb * sb_bytes(f);
  const int64_t rb2 = (f == F_NVFP4) ? K / 16 : 0;
  if (rb1 % 16 || rb2 % 16) return QGEMV_ERR_BAD_SHAPE;
  const int Wk = static_cast<int>((nsb + 7) / 8);
  if (Wk > 1 && N * Wk > QGEMV_NOALLOC_MAX_COLUMN_SUMS) return QGEMV_ERR_TOO_LARGE;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return QGEMV_ERR_NO_DEVICE;
  }
  DeviceSetup* s = nullptr;
  const qgemv_status_t st = setup(dev, &s);
  if (st != QGEMV_OK) return st;

  // Split plan: CTA = one K-column of a row range, all warps on it.
  const int cps = (Wk <= kMaxWarps / 2) ? 2 : 1;
  const int P = kMaxWarps / cps;
  int64_t ranges = std::min<int64_t>(std::max(1, (s->sms * cps) / Wk), (N + P - 1) / P);
  ranges = std::max<int64_t>(1, std::min<int64_t>(ranges, kMaxRanges));
  if (N / ranges >= 0x7ffffffe) return QGEMV_ERR_TOO_LARGE;
  const int Kx = static_cast<int>(std::min<int64_t>(K, 2048));
  const int slice = 8 * sb_bytes(f) + (f == F_NVFP4 ? 8 * 16 : 0);
  int R = Wk > 1 ? 4 : 2, D = Wk > 1 ? 2 : 4;
  const size_t cap = static_cast<size_t>((228 * 1024) / cps - 1024);
  auto rix = [](int r) { return r == 1 ? 0 : r == 2 ? 1 : 2; };
  auto limit = [&](int d, int r) { return std::min(s->dyn_smem_max[f][rix(r)][d - 2], cap); };
  const int coef = f == F_TQ10 ? DecTQ10::kCoefSB : f == F_NVFP4 ? DecNVFP4::kCoefSB : 0;
  auto smem_of = [&](int d, int r) { return stream_smem(P, d, r, slice, Wk, 0, Kx, coef).total; };
  while (smem_of(D, R) > limit(D, R) && (D > 2 || R > 1)) {
    if (D > 2)
      --D;
    else
      R >>= 1, D = 4;
  }
  if (smem_of(D, R) > limit(D, R)) return QGEMV_ERR_BAD_SHAPE;

  StreamArgs a{};
  a.W = static_cast<const uint8_t*>(packed_W);
  a.W2 = (f == F_NVFP4) ? a.W + N * (K / 2) : nullptr;
  a.x = static_cast<const uint16_t*>(x);
  a.y = y;
  a.N = N;
  a.rows_q = static_cast<int>(N / ranges);
  a.rows_rem = static_cast<int>(N % ranges);
  a.row_bytes = rb1;
  a.row_bytes2 = rb2;
  a.nsb = static_cast<int>(nsb);
  a.Wk = Wk;
  a.P = P;
  a.red_rows = 0;
  a.err = nullptr;  // written only under the stall test hook (test_stall = 0 here)
  a.spin_ns = 1000000000ull;
  a.test_stall = 0;
  a.pdl = 0;
  a.split = 1;
  a.ws = s->ws;
  a.cnt = s->cnt;

  // The counters must start at zero; a completed launch leaves them so, but the arrays keep
  // whatever an earlier call left, so clear them (no allocation: a memset of the array).
  if (Wk > 1 && cudaMemsetAsync(s->cnt, 0, sizeof(int) * ranges, stream) != cudaSuccess) {
    cudaGetLastError();
    return QGEMV_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ranges * Wk), 1, 1);
  cfg.blockDim = dim3(32 * P, 1, 1);
  cfg.dynamicSmemBytes = smem_of(D, R);
  cfg.stream = stream;
  void* args[] = {&a};
  if (cudaLaunchKernelExC(&cfg, kernel_for(f, R, D), args) != cudaSuccess) {
    cudaGetLastError();
    return QGEMV_ERR_CUDA;
  }
  return QGEMV_OK;
}
