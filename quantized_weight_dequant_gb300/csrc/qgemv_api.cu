// C-ABI of libqgemv: validation, launch planning and launches.  See include/qgemv.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <new>

#include "../../include/qgemv.h"
#include "qgemv_kernels.cuh"

#ifndef QGEMV_BUILD_ID
#define QGEMV_BUILD_ID "unversioned"
#endif

namespace {

using namespace qg;

constexpr size_t kWorkspaceBytes = 64ull << 20;  // split-K partials (fp32)
constexpr int kMaxWarpsPerCta = 16;
constexpr size_t kSmemBudget = 200 * 1024;       // ring + barriers + reduction buffer per CTA
constexpr size_t kRedBudget = 16 * 1024;

struct Handle {
  int device = 0;
  int sms = 0;
  int l2_bytes = 0;
  size_t smem_optin = 0;
  float* ws = nullptr;
  int* err = nullptr;
  int force_path = 0;
  int force_splitk = 0;
  int ring_depth = 0;
  int rows_per_stage = 0;
  uint64_t spin_ns = 1000000000ull;
  int pdl = 0;
  int test_stall = 0;
};

bool fmt_ok(int f) { return f >= 0 && f <= 5; }

int k_multiple(int f) {
  switch (f) {
    case F_Q80: return 32;
    case F_NVFP4: return 16;
    default: return 256;
  }
}

// Bytes per superblock (256 elements) of stream 1 / stream 2.
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
int sb_bytes2(int f) { return f == F_NVFP4 ? 16 : 0; }

size_t packed_bytes(int f, int64_t N, int64_t K) {
  if (!fmt_ok(f) || N < 1 || K < 1 || K % k_multiple(f)) return 0;
  if (f == F_NVFP4) return static_cast<size_t>(N) * (K / 2) + static_cast<size_t>(N) * (K / 16);
  if (f == F_Q80) return static_cast<size_t>(N) * (K / 32) * 34;
  return static_cast<size_t>(N) * (K / 256) * sb_bytes(f);
}

int group_size(int f) {
  switch (f) {
    case F_Q4K: case F_Q5K: case F_Q80: return 32;
    case F_Q6K: case F_NVFP4: return 16;
    case F_TQ10: return 256;
  }
  return 0;
}

struct Plan {
  int path = 2;  // 1 streaming kernels, 2 warp-per-row kernels
  StreamArgs sa{};
  int threads = 0, grid_x = 0, S = 1;
  size_t smem = 0;
  int rw_grid = 0, rw_block = 256;
};

template <class Dec>
const void* stream_fn() {
  return reinterpret_cast<const void*>(&stream_kernel<Dec>);
}

const void* stream_kernel_for(int f) {
  switch (f) {
    case F_Q4K: return stream_fn<DecQ4K>();
    case F_Q5K: return stream_fn<DecQ5K>();
    case F_Q6K: return stream_fn<DecQ6K>();
    case F_Q80: return stream_fn<DecQ80>();
    case F_TQ10: return stream_fn<DecTQ10>();
    case F_NVFP4: return stream_fn<DecNVFP4>();
  }
  return nullptr;
}

qgemv_status_t make_plan(const Handle& h, int f, int64_t N, int64_t K, Plan& pl) {
  const int64_t nsb = K / 256;
  int64_t rb1 = 0, rb2 = 0;
  if (K % 256 == 0) {
    rb1 = (f == F_NVFP4) ? K / 2 : nsb * sb_bytes(f);
    rb2 = (f == F_NVFP4) ? K / 16 : 0;
  }
  const bool fast_ok = (K % 256 == 0) && rb1 % 16 == 0 && rb2 % 16 == 0 && nsb <= (int64_t{1} << 30);
  int path = fast_ok ? 1 : 2;
  if (h.force_path == 2) path = 2;
  pl.path = path;
  if (path == 2) {
    pl.rw_block = 256;
    const int64_t want = (N + 7) / 8;
    pl.rw_grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, int64_t{h.sms} * 8)));
    return QGEMV_OK;
  }
  const int wk_full = static_cast<int>((nsb + 7) / 8);
  int S = (wk_full + kMaxWarpsPerCta - 1) / kMaxWarpsPerCta;
  if (h.force_splitk > 0) S = std::min<int>(h.force_splitk, static_cast<int>(nsb));
  const int sb_per_split = 8 * static_cast<int>(((nsb + S - 1) / S + 7) / 8);
  S = static_cast<int>((nsb + sb_per_split - 1) / sb_per_split);
  const int Wk = sb_per_split / 8;
  const int P = std::max(1, kMaxWarpsPerCta / Wk);
  const int warps = P * Wk;
  const int slice = 8 * sb_bytes(f) + 8 * sb_bytes2(f);  // multiple of 16 for every format
  int R = h.rows_per_stage > 0 ? h.rows_per_stage : 2;
  int D = h.ring_depth;
  if (D == 0) {
    D = static_cast<int>(kSmemBudget / (static_cast<size_t>(warps) * R * slice + 8));
    D = std::min(8, D);
    if (D < 2 && R > 1) {
      R = 1;
      D = std::min<int>(8, static_cast<int>(kSmemBudget / (static_cast<size_t>(warps) * slice + 8)));
    }
    D = std::max(2, D);
  }
  // Grid: one wave of CTAs over the rows, enough CTAs that the reduction buffer fits.
  const int64_t sms = h.sms;
  int64_t grid = std::min<int64_t>((N + P - 1) / P, std::max<int64_t>(1, sms / S));
  if (Wk > 1) {
    const int64_t max_rows = static_cast<int64_t>(kRedBudget / (4 * static_cast<size_t>(Wk)));
    grid = std::max<int64_t>(grid, (N + max_rows - 1) / max_rows);
  }
  grid = std::max<int64_t>(1, std::min<int64_t>(grid, 0x7fffffff));
  if (static_cast<int64_t>(S) * N * 4 > static_cast<int64_t>(kWorkspaceBytes) && S > 1) {
    pl.path = 2;  // would not fit the handle's workspace: plain path instead
    pl.rw_block = 256;
    pl.rw_grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((N + 7) / 8, int64_t{h.sms} * 8)));
    return QGEMV_OK;
  }
  const int red_rows = static_cast<int>((N + grid - 1) / grid + 1);
  // Forced ring shapes are upper bounds: shrink depth, then rows per stage, to fit.
  size_t smem = stream_smem_bytes(warps, D, R * slice, Wk, red_rows);
  while (smem > h.smem_optin && (D > 2 || R > 1)) {
    if (D > 2)
      --D;
    else
      --R;
    smem = stream_smem_bytes(warps, D, R * slice, Wk, red_rows);
  }
  if (smem > h.smem_optin) return QGEMV_ERR_BAD_SHAPE;

  StreamArgs& a = pl.sa;
  a.N = N;
  a.row_bytes = rb1;
  a.row_bytes2 = rb2;
  a.nsb = static_cast<int>(nsb);
  a.sb_per_split = sb_per_split;
  a.Wk = Wk;
  a.P = P;
  a.R = R;
  a.D = D;
  a.slot_bytes = R * slice;
  a.slice_stride = slice;
  a.red_rows = red_rows;
  a.err = h.err;
  a.spin_ns = h.spin_ns;
  a.test_stall = h.test_stall;
  a.pdl = h.pdl;
  pl.threads = 32 * warps;
  pl.grid_x = static_cast<int>(grid);
  pl.S = S;
  pl.smem = smem;
  return QGEMV_OK;
}

qgemv_status_t validate_shape(const Handle* h, int f, int64_t N, int64_t K) {
  if (!h) return QGEMV_ERR_INVALID_ARG;
  if (!fmt_ok(f)) return QGEMV_ERR_UNSUPPORTED_FORMAT;
  if (N < 1 || K < 1 || K % k_multiple(f)) return QGEMV_ERR_BAD_SHAPE;
  return QGEMV_OK;
}

qgemv_status_t validate(const Handle* h, int f, const void* W, int64_t N, int64_t K) {
  const qgemv_status_t st = validate_shape(h, f, N, K);
  if (st != QGEMV_OK) return st;
  if (!W) return QGEMV_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(W) & 15) return QGEMV_ERR_MISALIGNED;
  return QGEMV_OK;
}

template <int F>
void launch_rowwarp(const Plan& pl, const RowArgs& ra, cudaStream_t s) {
  rowwarp_kernel<F><<<pl.rw_grid, pl.rw_block, 0, s>>>(ra);
}

void launch_rowwarp_any(int f, const Plan& pl, const RowArgs& ra, cudaStream_t s) {
  switch (f) {
    case F_Q4K: launch_rowwarp<F_Q4K>(pl, ra, s); break;
    case F_Q5K: launch_rowwarp<F_Q5K>(pl, ra, s); break;
    case F_Q6K: launch_rowwarp<F_Q6K>(pl, ra, s); break;
    case F_Q80: launch_rowwarp<F_Q80>(pl, ra, s); break;
    case F_TQ10: launch_rowwarp<F_TQ10>(pl, ra, s); break;
    case F_NVFP4: launch_rowwarp<F_NVFP4>(pl, ra, s); break;
  }
}

template <int F>
void launch_unpack(const UnpackArgs& ua, int grid, cudaStream_t s) {
  unpack_kernel<F><<<grid, 256, 0, s>>>(ua);
}

}  // namespace

extern "C" {

const char* qgemv_build_marker(void) { return "qgemv-build:" QGEMV_BUILD_ID; }

const char* qgemv_status_string(qgemv_status_t s) {
  switch (s) {
    case QGEMV_OK: return "ok";
    case QGEMV_ERR_INVALID_ARG: return "invalid argument";
    case QGEMV_ERR_UNSUPPORTED_FORMAT: return "unsupported format";
    case QGEMV_ERR_BAD_SHAPE: return "bad shape";
    case QGEMV_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case QGEMV_ERR_CUDA: return "CUDA error";
    case QGEMV_ERR_TIMEOUT: return "kernel wait timed out";
    case QGEMV_ERR_OOM: return "out of device memory";
    case QGEMV_ERR_NO_DEVICE: return "no usable sm_103 device";
  }
  return "unknown status";
}

size_t qgemv_packed_bytes(qgemv_format_t fmt, int64_t N, int64_t K) { return packed_bytes(fmt, N, K); }

int qgemv_group_size(qgemv_format_t fmt) { return fmt_ok(fmt) ? group_size(fmt) : 0; }

qgemv_status_t qgemv_create(qgemv_handle_t* out, int device) {
  if (!out) return QGEMV_ERR_INVALID_ARG;
  *out = nullptr;
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || device < 0 || device >= n) {
    cudaGetLastError();
    return QGEMV_ERR_NO_DEVICE;
  }
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return QGEMV_ERR_NO_DEVICE;
  if (prop.major != 10 || prop.minor != 3) return QGEMV_ERR_NO_DEVICE;
  if (cudaSetDevice(device) != cudaSuccess) return QGEMV_ERR_CUDA;
  Handle* h = new (std::nothrow) Handle();
  if (!h) return QGEMV_ERR_OOM;
  h->device = device;
  h->sms = prop.multiProcessorCount;
  h->l2_bytes = prop.l2CacheSize;
  h->smem_optin = prop.sharedMemPerBlockOptin;
  if (cudaMalloc(&h->ws, kWorkspaceBytes) != cudaSuccess || cudaMalloc(&h->err, sizeof(int)) != cudaSuccess ||
      cudaMemset(h->err, 0, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->ws);
    cudaFree(h->err);
    delete h;
    return QGEMV_ERR_OOM;
  }
  for (int f = 0; f <= 5; ++f) {
    if (cudaFuncSetAttribute(stream_kernel_for(f), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(h->smem_optin)) != cudaSuccess) {
      cudaGetLastError();
      cudaFree(h->ws);
      cudaFree(h->err);
      delete h;
      return QGEMV_ERR_CUDA;
    }
  }
  *out = reinterpret_cast<qgemv_handle_t>(h);
  return QGEMV_OK;
}

qgemv_status_t qgemv_destroy(qgemv_handle_t hh) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return QGEMV_OK;
  cudaFree(h->ws);
  cudaFree(h->err);
  delete h;
  return QGEMV_OK;
}

qgemv_status_t qgemv_set_option(qgemv_handle_t hh, qgemv_option_t opt, int64_t v) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return QGEMV_ERR_INVALID_ARG;
  switch (opt) {
    case QGEMV_OPT_FORCE_PATH:
      if (v < 0 || v > 2) return QGEMV_ERR_INVALID_ARG;
      h->force_path = static_cast<int>(v);
      return QGEMV_OK;
    case QGEMV_OPT_FORCE_SPLITK:
      if (v < 0 || v > 4096) return QGEMV_ERR_INVALID_ARG;
      h->force_splitk = static_cast<int>(v);
      return QGEMV_OK;
    case QGEMV_OPT_RING_DEPTH:
      if (v != 0 && (v < 2 || v > 8)) return QGEMV_ERR_INVALID_ARG;
      h->ring_depth = static_cast<int>(v);
      return QGEMV_OK;
    case QGEMV_OPT_ROWS_PER_STAGE:
      if (v < 0 || v > 8) return QGEMV_ERR_INVALID_ARG;
      h->rows_per_stage = static_cast<int>(v);
      return QGEMV_OK;
    case QGEMV_OPT_SPIN_LIMIT_NS:
      if (v < 0) return QGEMV_ERR_INVALID_ARG;
      h->spin_ns = static_cast<uint64_t>(v);
      return QGEMV_OK;
    case QGEMV_OPT_PDL:
      if (v < 0 || v > 1) return QGEMV_ERR_INVALID_ARG;
      h->pdl = static_cast<int>(v);
      return QGEMV_OK;
    case QGEMV_OPT_TEST_STALL:
      if (v < 0 || v > 1) return QGEMV_ERR_INVALID_ARG;
      h->test_stall = static_cast<int>(v);
      return QGEMV_OK;
  }
  return QGEMV_ERR_INVALID_ARG;
}

qgemv_status_t qgemv_describe(qgemv_handle_t hh, qgemv_format_t fmt, int64_t N, int64_t K, char* buf, size_t len) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  qgemv_status_t st = validate_shape(h, fmt, N, K);
  if (st != QGEMV_OK) return st;
  Plan pl;
  st = make_plan(*h, fmt, N, K, pl);
  if (st != QGEMV_OK) return st;
  if (buf && len) {
    if (pl.path == 1)
      snprintf(buf, len,
               "path=stream grid=%dx%d block=%d warps_per_row=%d row_groups=%d rows_per_stage=%d ring=%d "
               "splitk=%d smem=%zu pdl=%d",
               pl.grid_x, pl.S, pl.threads, pl.sa.Wk, pl.sa.P, pl.sa.R, pl.sa.D, pl.S, pl.smem, pl.sa.pdl);
    else
      snprintf(buf, len, "path=rowwarp grid=%d block=%d", pl.rw_grid, pl.rw_block);
  }
  return QGEMV_OK;
}

qgemv_status_t qgemv_run(qgemv_handle_t hh, qgemv_format_t fmt, const void* x, const void* W, int64_t N, int64_t K,
                         float* y, cudaStream_t stream) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  qgemv_status_t st = validate(h, fmt, W, N, K);
  if (st != QGEMV_OK) return st;
  if (!x || !y) return QGEMV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15) return QGEMV_ERR_MISALIGNED;
  Plan pl;
  st = make_plan(*h, fmt, N, K, pl);
  if (st != QGEMV_OK) return st;
  const uint8_t* Wb = static_cast<const uint8_t*>(W);
  if (pl.path == 2) {
    RowArgs ra{Wb, static_cast<const uint16_t*>(x), y, N, K};
    launch_rowwarp_any(fmt, pl, ra, stream);
    return cudaGetLastError() == cudaSuccess ? QGEMV_OK : QGEMV_ERR_CUDA;
  }
  StreamArgs a = pl.sa;
  a.W = Wb;
  a.W2 = (fmt == QGEMV_NVFP4) ? Wb + N * (K / 2) : nullptr;
  a.x = static_cast<const uint16_t*>(x);
  a.out = (pl.S > 1) ? h->ws : y;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid_x, pl.S, 1);
  cfg.blockDim = dim3(pl.threads, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (h->pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  void* args[] = {&a};
  if (cudaLaunchKernelExC(&cfg, stream_kernel_for(fmt), args) != cudaSuccess) {
    cudaGetLastError();
    return QGEMV_ERR_CUDA;
  }
  if (pl.S > 1) {
    const int grid = static_cast<int>(std::min<int64_t>((N + 255) / 256, int64_t{h->sms} * 4));
    splitk_reduce<<<grid, 256, 0, stream>>>(h->ws, y, N, pl.S);
    if (cudaGetLastError() != cudaSuccess) return QGEMV_ERR_CUDA;
  }
  return QGEMV_OK;
}

qgemv_status_t qgemv_unpack(qgemv_handle_t hh, qgemv_format_t fmt, const void* W, int64_t N, int64_t K, int8_t* codes,
                            float* scales, float* mins, cudaStream_t stream) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  qgemv_status_t st = validate(h, fmt, W, N, K);
  if (st != QGEMV_OK) return st;
  if (!codes || !scales) return QGEMV_ERR_INVALID_ARG;
  UnpackArgs ua{static_cast<const uint8_t*>(W), codes, scales, mins, N, K, group_size(fmt)};
  const int64_t total = N * (K / ua.G);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, int64_t{h->sms} * 16)));
  switch (fmt) {
    case QGEMV_Q4_K: launch_unpack<F_Q4K>(ua, grid, stream); break;
    case QGEMV_Q5_K: launch_unpack<F_Q5K>(ua, grid, stream); break;
    case QGEMV_Q6_K: launch_unpack<F_Q6K>(ua, grid, stream); break;
    case QGEMV_Q8_0: launch_unpack<F_Q80>(ua, grid, stream); break;
    case QGEMV_TQ1_0: launch_unpack<F_TQ10>(ua, grid, stream); break;
    case QGEMV_NVFP4: launch_unpack<F_NVFP4>(ua, grid, stream); break;
  }
  return cudaGetLastError() == cudaSuccess ? QGEMV_OK : QGEMV_ERR_CUDA;
}

qgemv_status_t qgemv_check_error(qgemv_handle_t hh, cudaStream_t stream) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return QGEMV_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return QGEMV_ERR_CUDA;
  }
  int e = 0;
  if (cudaMemcpy(&e, h->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return QGEMV_ERR_CUDA;
  if (e != 0 && cudaMemset(h->err, 0, sizeof(int)) != cudaSuccess) return QGEMV_ERR_CUDA;
  return (e & kDevErrTimeout) ? QGEMV_ERR_TIMEOUT : QGEMV_OK;
}

}  // extern "C"
