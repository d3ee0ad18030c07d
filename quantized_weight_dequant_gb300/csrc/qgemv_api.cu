// C-ABI of libqgemv: validation, launch planning and launches.  See include/qgemv.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <new>

#include "../../include/qgemv.h"
#include "qgemv_simple.cuh"
#include "qgemv_stream.cuh"

#ifndef QGEMV_BUILD_ID
#define QGEMV_BUILD_ID "unversioned"
#endif

namespace {

using namespace qg;

constexpr int kMaxWarps = 16;                    // per CTA (launch bound 512 threads)
constexpr size_t kRedBudget = 16 * 1024;         // cross-warp reduction buffer per CTA
constexpr size_t kWsFloats = size_t{4} << 20;    // split-K column sums: N * K-columns <= 4 Mi
constexpr int kMaxRanges = 1024;                 // split-K row ranges (one counter each)

struct Handle {
  int device = 0;
  int sms = 0;
  int l2_bytes = 0;
  size_t smem_optin = 0;
  int* err = nullptr;
  float* ws = nullptr;  // split-K column sums
  int* cnt = nullptr;   // split-K per-range arrival counts, zero between launches
  int ctas_per_sm = 2;
  int ksplit = 0;       // 0: split K-columns over CTAs when the workspace holds them; 1: never
  int grid_per_sm = 0;  // CTAs launched per SM (0: as many as fit, ctas_per_sm)
  size_t dyn_smem_max[6][3][3] = {};  // [format][R 1/2/4][D 2/3/4]
  int force_path = 0;
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
  int path = 2;  // 1 streaming kernel, 2 warp-per-row kernel
  StreamArgs sa{};
  int grid = 0, threads = 0, R = 2, D = 4;
  size_t smem = 0;
  int rw_grid = 0, rw_block = 256;
};

}  // namespace

namespace qg {
const void* stream_kernel_q4k(int R, int D);
const void* stream_kernel_q5k(int R, int D);
const void* stream_kernel_q6k(int R, int D);
const void* stream_kernel_q80(int R, int D);
const void* stream_kernel_tq10(int R, int D);
const void* stream_kernel_nvfp4(int R, int D);
}  // namespace qg

namespace {

const void* stream_kernel_for(int f, int R, int D) {
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

int r_index(int R) { return R == 1 ? 0 : R == 2 ? 1 : 2; }
int d_index(int D) { return D - 2; }

void rowwarp_plan(const Handle& h, int64_t N, Plan& pl) {
  pl.path = 2;
  pl.rw_block = 256;
  pl.rw_grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((N + 7) / 8, int64_t{h.sms} * 8)));
}

int slice_of(int f) { return 8 * sb_bytes(f) + 8 * sb_bytes2(f); }

qgemv_status_t make_plan(const Handle& h, int f, int64_t N, int64_t K, Plan& pl) {
  const int64_t nsb = K / 256;
  int64_t rb1 = 0, rb2 = 0;
  if (K % 256 == 0) {
    rb1 = (f == F_NVFP4) ? K / 2 : nsb * sb_bytes(f);
    rb2 = (f == F_NVFP4) ? K / 16 : 0;
  }
  const int64_t Wk64 = (nsb + 7) / 8;
  const bool fast_ok = (K % 256 == 0) && rb1 % 16 == 0 && rb2 % 16 == 0 && Wk64 >= 1 && Wk64 <= kMaxWarps;
  if (!fast_ok || h.force_path == 2) {
    rowwarp_plan(h, N, pl);
    return QGEMV_OK;
  }
  const int Wk = static_cast<int>(Wk64);
  const int cps = (Wk <= kMaxWarps / 2) ? h.ctas_per_sm : 1;  // CTAs per SM
  // Split mode: a CTA takes one K-column of a row range with all its warps, so it stages only
  // that column of x; column sums meet in the workspace.  Fused mode: a CTA covers all
  // K-columns of its rows and adds the column sums in shared memory.
  // Two columns are faster fused (their x is small); from three on the split pays.
  const bool split = Wk == 1 || (h.ksplit == 0 && Wk >= 3 && static_cast<double>(N) * Wk <= static_cast<double>(kWsFloats));
  const int P = split ? kMaxWarps / cps : std::max(1, (kMaxWarps / cps) / Wk);
  const int warps = split ? P : P * Wk;
  // Under programmatic dependent launch a fused launch with few rows per warp (at most 16
  // with every slot filled) takes one CTA per SM: the next launch's CTAs then fit beside it
  // and fetch their first stages while this one finishes.
  const bool short_pdl = h.pdl && !split && cps == 2 && N <= int64_t{16} * h.sms * cps * P;
  const int gps = h.grid_per_sm > 0 ? std::min(h.grid_per_sm, cps) : (short_pdl ? 1 : cps);
  int64_t ranges, grid;
  if (split) {
    ranges = std::min<int64_t>(std::max(1, (h.sms * gps) / Wk), (N + P - 1) / P);
    ranges = std::max<int64_t>(1, std::min<int64_t>(ranges, kMaxRanges));
    grid = ranges * Wk;
  } else {
    grid = std::min<int64_t>(int64_t{h.sms} * gps, (N + P - 1) / P);
    if (Wk > 1) grid = std::max<int64_t>(grid, (N + (kRedBudget / (4 * Wk)) - 2) / (kRedBudget / (4 * Wk) - 1));
    grid = std::max<int64_t>(1, std::min<int64_t>(grid, 0x7fffffff));
    ranges = grid;
  }
  if (N / ranges >= 0x7ffffffe) {  // per-CTA row counts are 32-bit in the kernel
    rowwarp_plan(h, N, pl);
    return QGEMV_OK;
  }
  const int red_rows = split ? 0 : static_cast<int>((N + grid - 1) / grid + 1);
  const int Kx = split ? static_cast<int>(std::min<int64_t>(K, 2048)) : static_cast<int>(K);
  const int slice = slice_of(f);
  // Defaults: 2 rows per stage, 4 stages; split launches (long K): 4 rows, 2 stages.
  const bool long_k = split && Wk > 1;
  const bool half = gps < cps;  // one CTA per SM of a two-per-SM layout
  int R = h.rows_per_stage > 0 ? (h.rows_per_stage >= 4 ? 4 : h.rows_per_stage >= 2 ? 2 : 1) : (long_k || half ? 4 : 2);
  int D = h.ring_depth > 0 ? std::min(h.ring_depth, 4) : (long_k ? 2 : half ? 3 : 4);
  const size_t cap = static_cast<size_t>((228 * 1024) / cps - 1024);
  auto limit = [&](int d, int r) { return std::min(h.dyn_smem_max[f][r_index(r)][d_index(d)], cap); };
  auto smem_of = [&](int d, int r) { return stream_smem(warps, d, r, slice, Wk, red_rows, Kx).total; };
  while (smem_of(D, R) > limit(D, R) && (D > 2 || R > 1)) {
    if (D > 2)
      --D;
    else
      R >>= 1, D = 4;
  }
  const size_t smem = smem_of(D, R);
  if (smem > limit(D, R)) {
    rowwarp_plan(h, N, pl);
    return QGEMV_OK;
  }
  StreamArgs& a = pl.sa;
  a.N = N;
  a.rows_q = static_cast<int>(N / ranges);
  a.rows_rem = static_cast<int>(N % ranges);
  a.row_bytes = rb1;
  a.row_bytes2 = rb2;
  a.nsb = static_cast<int>(nsb);
  a.Wk = Wk;
  a.P = P;
  a.red_rows = red_rows;
  a.err = h.err;
  a.spin_ns = h.spin_ns;
  a.test_stall = h.test_stall;
  // Under programmatic dependent launch, a launch that leaves room on each SM for the next
  // one requests its first weight stages before waiting for the previous kernel (kernel mode
  // 1); one that fills the SMs cannot overlap much, and takes x first (mode 2), so x is not
  // queued behind its own weight stages.
  a.pdl = !h.pdl ? 0 : (gps < cps ? 1 : 2);
  a.split = split ? 1 : 0;
  a.ws = h.ws;
  a.cnt = h.cnt;
  pl.path = 1;
  pl.grid = static_cast<int>(grid);
  pl.threads = 32 * warps;
  pl.R = R;
  pl.D = D;
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
    case QGEMV_ERR_TOO_LARGE: return "shape exceeds the fixed scratch of qgemv_run_noalloc";
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
  auto release = [h]() {
    cudaGetLastError();
    cudaFree(h->err);
    cudaFree(h->ws);
    cudaFree(h->cnt);
    delete h;
  };
  if (cudaMalloc(&h->err, sizeof(int)) != cudaSuccess || cudaMalloc(&h->ws, kWsFloats * sizeof(float)) != cudaSuccess ||
      cudaMalloc(&h->cnt, kMaxRanges * sizeof(int)) != cudaSuccess) {
    release();
    return QGEMV_ERR_OOM;
  }
  if (cudaMemset(h->err, 0, sizeof(int)) != cudaSuccess || cudaMemset(h->cnt, 0, kMaxRanges * sizeof(int)) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    release();
    return QGEMV_ERR_CUDA;
  }
  for (int f = 0; f <= 5; ++f)
    for (int R : {1, 2, 4})
      for (int D : {2, 3, 4}) {
      cudaFuncAttributes fa;
      const void* fn = stream_kernel_for(f, R, D);
      if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) {
        release();
        return QGEMV_ERR_CUDA;
      }
      size_t& mx = h->dyn_smem_max[f][r_index(R)][d_index(D)];
      mx = h->smem_optin - std::min(h->smem_optin, fa.sharedSizeBytes);
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(mx)) != cudaSuccess) {
        release();
        return QGEMV_ERR_CUDA;
      }
    }
  *out = reinterpret_cast<qgemv_handle_t>(h);
  return QGEMV_OK;
}

qgemv_status_t qgemv_destroy(qgemv_handle_t hh) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return QGEMV_OK;
  cudaFree(h->err);
  cudaFree(h->ws);
  cudaFree(h->cnt);
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
    case QGEMV_OPT_CTAS_PER_SM:
      if (v < 1 || v > 2) return QGEMV_ERR_INVALID_ARG;
      h->ctas_per_sm = static_cast<int>(v);
      return QGEMV_OK;
    case QGEMV_OPT_GRID_PER_SM:
      if (v < 0 || v > 2) return QGEMV_ERR_INVALID_ARG;
      h->grid_per_sm = static_cast<int>(v);
      return QGEMV_OK;
    case QGEMV_OPT_KSPLIT:
      if (v < 0 || v > 1) return QGEMV_ERR_INVALID_ARG;
      h->ksplit = static_cast<int>(v);
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
               "path=stream grid=%d block=%d kcols=%d split=%d row_groups=%d rows_per_stage=%d ring=%d smem=%zu "
               "pdl=%d",
               pl.grid, pl.threads, pl.sa.Wk, pl.sa.split, pl.sa.P, pl.R, pl.D, pl.smem, h->pdl);
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
  a.y = y;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid, 1, 1);
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
  if (cudaLaunchKernelExC(&cfg, stream_kernel_for(fmt, pl.R, pl.D), args) != cudaSuccess) {
    cudaGetLastError();
    return QGEMV_ERR_CUDA;
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
