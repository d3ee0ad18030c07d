// C-ABI of libqgemv: validation, launch planning and launches.  See include/qgemv.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <new>

#include "../../include/qgemv.h"
#include "qgemm_tc.cuh"
#include "qgemv_batch.cuh"
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
  size_t group_smem_max[2][3] = {};   // mixed-format grouped kernel [R 2/4][D 2/3/4]
  size_t group1_smem_max[6][2][2][3] = {};  // one-format grouped kernels [format][pairs][R 2/4][D 2/3/4]
  size_t batch_smem_max[6][2] = {};          // small-batch kernels [format][D 2/3]
  void* encode_tiled = nullptr;              // the driver's cuTensorMapEncodeTiled (null: no TMA path)
  int tc_cluster_max[3] = {1, 1, 1};         // largest cluster (K splits) the GEMM kernels can run [BT 64/128/256]
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

// One matrix of a launch as the planner sees it.
struct Problem {
  int f = 0;
  const void* W = nullptr;
  const void* WB = nullptr;  // SwiGLU up matrix
  int64_t N = 0;             // outputs
  void* y = nullptr;
  float alpha = 1.f, beta = 0.f;
  int ydt = 0, pair = 0;
};

struct Plan {
  int path = 2;  // 1 streaming kernel, 2 warp-per-row kernel
  StreamArgs sa{};
  int grid = 0, threads = 0, R = 2, D = 4;
  size_t smem = 0;
  int rw_grid = 0, rw_block = 256;
};

// A streaming launch over several matrices sharing x: the CTAs of matrix i are
// [cta_end[i-1], cta_end[i]).
struct GroupPlan {
  GroupArgs ga{};
  int fmt = -1;  // the one format of the launch, or -1 for mixed formats
  bool pairs = false;  // one format, every matrix a SwiGLU pair
  int grid = 0, threads = 0, R = 2, D = 4;
  size_t smem = 0;
};
static_assert(kMaxGroup == QGEMV_MAX_GROUP, "grouped launch capacity");

}  // namespace

namespace qg {
const void* stream_kernel_q4k(int R, int D);
const void* stream_kernel_q5k(int R, int D);
const void* stream_kernel_q6k(int R, int D);
const void* stream_kernel_q80(int R, int D);
const void* stream_kernel_tq10(int R, int D);
const void* stream_kernel_nvfp4(int R, int D);
const void* group_kernel_r2(int D);
const void* group_kernel_r4(int D);
const void* group_kernel_q4k(int R, int D);
const void* group_kernel_q5k(int R, int D);
const void* group_kernel_q6k(int R, int D);
const void* group_kernel_q80(int R, int D);
const void* group_kernel_tq10(int R, int D);
const void* group_kernel_nvfp4(int R, int D);
const void* group_kernel_pair_q4k(int R, int D);
const void* group_kernel_pair_q5k(int R, int D);
const void* group_kernel_pair_q6k(int R, int D);
const void* group_kernel_pair_q80(int R, int D);
const void* group_kernel_pair_tq10(int R, int D);
const void* group_kernel_pair_nvfp4(int R, int D);
const void* batch_kernel_for(int f, int D);
size_t batch_smem_bytes(int f, int warps, int D);
const void* tc_kernel_for(int BT);
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

// Grouped kernel for ring shape (R, D): the one-format kernel of format f (with the SwiGLU
// pairing compiled in when every matrix is a pair), or (f < 0) the mixed-format one.
const void* group_kernel_for(int f, int R, int D, bool pairs = false) {
  if (pairs) {
    switch (f) {
      case F_Q4K: return group_kernel_pair_q4k(R, D);
      case F_Q5K: return group_kernel_pair_q5k(R, D);
      case F_Q6K: return group_kernel_pair_q6k(R, D);
      case F_Q80: return group_kernel_pair_q80(R, D);
      case F_TQ10: return group_kernel_pair_tq10(R, D);
      case F_NVFP4: return group_kernel_pair_nvfp4(R, D);
    }
  }
  switch (f) {
    case F_Q4K: return group_kernel_q4k(R, D);
    case F_Q5K: return group_kernel_q5k(R, D);
    case F_Q6K: return group_kernel_q6k(R, D);
    case F_Q80: return group_kernel_q80(R, D);
    case F_TQ10: return group_kernel_tq10(R, D);
    case F_NVFP4: return group_kernel_nvfp4(R, D);
  }
  return R >= 4 ? group_kernel_r4(D) : group_kernel_r2(D);
}

int r_index(int R) { return R == 1 ? 0 : R == 2 ? 1 : 2; }
int d_index(int D) { return D - 2; }

void rowwarp_plan(const Handle& h, int64_t N, Plan& pl) {
  pl.path = 2;
  pl.rw_block = 256;
  pl.rw_grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((N + 7) / 8, int64_t{h.sms} * 8)));
}

int slice_of(int f) { return 8 * sb_bytes(f) + 8 * sb_bytes2(f); }
// Decoder area bytes per staged superblock (TQ1_0's x in its own per-superblock slots,
// NVFP4's residuals); must equal the decoder's kCoefSB.
int coef_of(int f) { return f == F_TQ10 ? DecTQ10::kCoefSB : f == F_NVFP4 ? DecNVFP4::kCoefSB : 0; }

// Packed row bytes of stream 1 / 2, or false when the streaming kernel cannot take the
// shape (rows must be whole superblocks and 16-byte multiples, at most 16 K-columns).
bool stream_rows(int f, int64_t K, int64_t& rb1, int64_t& rb2) {
  if (K % 256) return false;
  const int64_t nsb = K / 256;
  rb1 = (f == F_NVFP4) ? K / 2 : nsb * sb_bytes(f);
  rb2 = (f == F_NVFP4) ? K / 16 : 0;
  const int64_t Wk = (nsb + 7) / 8;
  return rb1 % 16 == 0 && rb2 % 16 == 0 && Wk >= 1 && Wk <= kMaxWarps;
}

// The streaming launch over the matrices `ps[0..n)` (all of them streaming-eligible, one K).
// Every matrix gets CTAs in proportion to its bytes; the launch-wide choices (K-columns per
// CTA, split or fused, ring shape) follow from K and the largest shared-memory need.
// `general` selects the grouped kernel (epilogue, pairs, several formats), whose ring shapes
// are R in {2, 4}.  Returns false when no ring shape fits (the caller falls back).
bool plan_stream(const Handle& h, const Problem* ps, int n, int64_t K, bool general, GroupPlan& gp) {
  int gf = ps[0].f;  // the one format of a grouped launch, or -1 for mixed formats
  bool all_pairs = true;
  for (int i = 0; i < n; ++i) {
    if (ps[i].f != gf) gf = -1;
    all_pairs = all_pairs && ps[i].pair;
  }
  const bool pairs = gf >= 0 && all_pairs;
  const int64_t nsb = K / 256;
  const int Wk = static_cast<int>((nsb + 7) / 8);
  const int cps = (Wk <= kMaxWarps / 2) ? h.ctas_per_sm : 1;  // CTAs per SM
  int64_t V[kMaxGroup], U[kMaxGroup], rb1[kMaxGroup], rb2[kMaxGroup];
  int64_t Vsum = 0;
  double Bsum = 0;
  bool any_pair = false;
  for (int i = 0; i < n; ++i) {
    stream_rows(ps[i].f, K, rb1[i], rb2[i]);
    U[i] = ps[i].N;
    V[i] = ps[i].pair ? 2 * ps[i].N : ps[i].N;  // virtual rows
    Vsum += V[i];
    Bsum += static_cast<double>(V[i]) * static_cast<double>(rb1[i] + rb2[i]);
    any_pair = any_pair || ps[i].pair;
  }
  // Split mode: a CTA takes one K-column of a row range with all its warps, so it stages only
  // that column of x; column sums meet in the workspace.  Fused mode: a CTA covers all
  // K-columns of its rows and adds the column sums in shared memory.
  // Two columns are faster fused (their x is small); from three on the split pays.
  const bool split = Wk == 1 || (h.ksplit == 0 && Wk >= 3 && static_cast<double>(Vsum) * Wk <= static_cast<double>(kWsFloats));
  const int P = split ? kMaxWarps / cps : std::max(1, (kMaxWarps / cps) / Wk);
  const int warps = split ? P : P * Wk;
  // Under programmatic dependent launch a fused launch with few rows per warp (at most 16
  // with every slot filled) takes one CTA per SM: the next launch's CTAs then fit beside it
  // and fetch their first stages while this one finishes.
  const bool short_pdl = h.pdl && !split && cps == 2 && Vsum <= int64_t{16} * h.sms * cps * P;
  const int gps = h.grid_per_sm > 0 ? std::min(h.grid_per_sm, cps) : (short_pdl ? 1 : cps);
  const int64_t T = int64_t{h.sms} * gps;  // CTAs that fit at once
  int64_t ranges[kMaxGroup], grid[kMaxGroup];
  int red_rows[kMaxGroup] = {};
  int64_t total_ranges = 0, total_grid = 0, ws_need = 0;
  for (int i = 0; i < n; ++i) {
    const double share = (static_cast<double>(V[i]) * static_cast<double>(rb1[i] + rb2[i])) / Bsum;
    const int64_t units_max = (U[i] + P - 1) / P;  // at least one unit per row group
    if (split) {
      ranges[i] = std::min<int64_t>(std::max<int64_t>(1, static_cast<int64_t>(static_cast<double>(T / Wk) * share)), units_max);
      ranges[i] = std::max<int64_t>(1, ranges[i]);
      grid[i] = ranges[i] * Wk;
    } else {
      grid[i] = std::min<int64_t>(std::max<int64_t>(1, static_cast<int64_t>(static_cast<double>(T) * share)), units_max);
      if (Wk > 1) {  // the reduction buffer holds every row of a CTA
        const int64_t per = (static_cast<int64_t>(kRedBudget / (4 * Wk)) - 1) / (ps[i].pair ? 2 : 1);
        if (per < 1) return false;
        grid[i] = std::max<int64_t>(grid[i], (U[i] + per - 1) / per);
      }
      grid[i] = std::max<int64_t>(1, grid[i]);
      ranges[i] = grid[i];
      red_rows[i] = static_cast<int>((ps[i].pair ? 2 : 1) * ((U[i] + grid[i] - 1) / grid[i]) + 1);
    }
    if (U[i] / ranges[i] >= 0x3ffffffe) return false;  // per-CTA row counts are 32-bit in the kernel
    if (split && (Wk > 1 || ps[i].pair)) {  // sums through the workspace, one counter per range
      total_ranges += ranges[i];
      ws_need += V[i] * Wk;
    }
    total_grid += grid[i];
  }
  if (total_ranges > kMaxRanges || ws_need > static_cast<int64_t>(kWsFloats)) return false;
  if (total_grid > 0x7fffffff) return false;
  const int Kx = split ? static_cast<int>(std::min<int64_t>(K, 2048)) : static_cast<int>(K);
  // Ring shape.  Defaults: 4 rows per stage, 2 stages (measured on the 28672 x 4096 decode
  // shape: fewer stage turns per row than 2 rows x 4 stages for the same bytes in flight);
  // a one-CTA-per-SM launch of a two-per-SM layout: 4 rows, 3 stages (split launches keep 2);
  // one K-column (K <= 2048): 2 rows, 4 stages.
  const bool half = gps < cps;
  const bool one_col = Wk == 1 && !half;
  int64_t rpw = INT64_MAX;  // fewest rows per warp over the launch's matrices
  for (int i = 0; i < n; ++i) rpw = std::min<int64_t>(rpw, V[i] / std::max<int64_t>(1, ranges[i] * P));
  // one K-column with fewer than 4 rows per warp (e.g. 1024 x 1024): one row per stage.  One
  // CTA per SM: as deep a ring as fits (below; measured: TQ1_0 4096 x 4096 4.40 -> 4.14 µs,
  // the other small launches unchanged).
  const int Rdef = one_col ? (rpw < 4 ? 1 : 2) : 4, Ddef = one_col ? 4 : (half && !(split && Wk > 1)) ? 4 : 2;
  int R = h.rows_per_stage > 0 ? (h.rows_per_stage >= 4 ? 4 : h.rows_per_stage >= 2 ? 2 : 1) : Rdef;
  int D = h.ring_depth > 0 ? std::min(h.ring_depth, 4) : Ddef;
  const int Rmin = general ? 2 : 1;
  if (R < Rmin) R = Rmin;
  const size_t cap = static_cast<size_t>((228 * 1024) / cps - 1024);
  auto limit = [&](int d, int r) {
    size_t m = cap;
    for (int i = 0; i < n; ++i)
      m = std::min(m, !general ? h.dyn_smem_max[ps[i].f][r_index(r)][d_index(d)]
                      : gf >= 0 ? h.group1_smem_max[gf][pairs ? 1 : 0][r >= 4 ? 1 : 0][d_index(d)]
                                : h.group_smem_max[r >= 4 ? 1 : 0][d_index(d)]);
    return m;
  };
  auto smem_of = [&](int d, int r) {
    size_t m = 0;
    for (int i = 0; i < n; ++i) m = std::max(m, stream_smem(warps, d, r, slice_of(ps[i].f), Wk, red_rows[i], Kx, coef_of(ps[i].f)).total);
    return m;
  };
  while (smem_of(D, R) > limit(D, R) && (D > 2 || R > Rmin)) {
    if (D > 2)
      --D;
    else
      R >>= 1, D = 4;
  }
  if (smem_of(D, R) > limit(D, R)) return false;
  (void)any_pair;
  gp.fmt = gf;
  gp.pairs = pairs;
  gp.grid = static_cast<int>(total_grid);
  gp.threads = 32 * warps;
  gp.R = R;
  gp.D = D;
  gp.smem = smem_of(D, R);
  gp.ga.count = n;
  int64_t cta = 0, rng = 0, ws_off = 0;
  for (int i = 0; i < n; ++i) {
    const Problem& q = ps[i];
    StreamArgs& a = gp.ga.p[i];
    a = StreamArgs{};
    a.W = static_cast<const uint8_t*>(q.W);
    a.W2 = (q.f == F_NVFP4) ? a.W + q.N * (K / 2) : nullptr;
    a.WB = q.pair ? static_cast<const uint8_t*>(q.WB) : nullptr;
    a.WB2 = (q.pair && q.f == F_NVFP4) ? a.WB + q.N * (K / 2) : nullptr;
    a.y = q.y;
    a.N = V[i];
    a.rows_q = static_cast<int>(U[i] / ranges[i]);
    a.rows_rem = static_cast<int>(U[i] % ranges[i]);
    a.row_bytes = rb1[i];
    a.row_bytes2 = rb2[i];
    a.nsb = static_cast<int>(nsb);
    a.Wk = Wk;
    a.P = P;
    a.red_rows = red_rows[i];
    a.err = h.err;
    a.spin_ns = h.spin_ns;
    a.test_stall = i == 0 ? h.test_stall : 0;
    // Under programmatic dependent launch every launch requests its first weight stages before
    // waiting for the previous kernel (kernel mode 1; measured faster than taking x first, mode
    // 2, also on launches that fill the SMs: CTAs that start as the previous kernel's leave
    // their SM have their first weights in flight while the rest of it finishes).
    a.pdl = !h.pdl ? 0 : 1;
    a.split = split ? 1 : 0;
    a.ws = h.ws + ws_off;
    a.cnt = h.cnt + rng;
    a.alpha = q.alpha;
    a.beta = q.beta;
    a.ydt = q.ydt;
    a.pair = q.pair;
    gp.ga.fmt[i] = q.f;
    cta += grid[i];
    gp.ga.cta_end[i] = static_cast<int>(cta);
    if (split && (Wk > 1 || q.pair)) {
      rng += ranges[i];
      ws_off += V[i] * Wk;
    }
  }
  return true;
}

// The single-matrix plan of qgemv_run / qgemv_describe.
qgemv_status_t make_plan(const Handle& h, int f, int64_t N, int64_t K, Plan& pl) {
  int64_t rb1 = 0, rb2 = 0;
  if (!stream_rows(f, K, rb1, rb2) || h.force_path == 2) {
    rowwarp_plan(h, N, pl);
    return QGEMV_OK;
  }
  Problem p;
  p.f = f;
  p.N = N;
  GroupPlan gp;
  if (!plan_stream(h, &p, 1, K, false, gp)) {
    rowwarp_plan(h, N, pl);
    return QGEMV_OK;
  }
  pl.path = 1;
  pl.sa = gp.ga.p[0];
  pl.grid = gp.grid;
  pl.threads = gp.threads;
  pl.R = gp.R;
  pl.D = gp.D;
  pl.smem = gp.smem;
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

// One single-vector GEMV on validated arguments (x 16-byte aligned; y needs no alignment).
qgemv_status_t launch_single(const Handle& hr, int fmt, const void* x, const void* W, int64_t N, int64_t K, float* y,
                             cudaStream_t stream) {
  const Handle* h = &hr;
  Plan pl;
  qgemv_status_t st = make_plan(*h, fmt, N, K, pl);
  if (st != QGEMV_OK) return st;
  const uint8_t* Wb = static_cast<const uint8_t*>(W);
  if (pl.path == 2) {
    RowArgs ra{Wb, static_cast<const uint16_t*>(x), y, N, K, 1.f, 0.f, 0, 0, nullptr};
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
  for (int f = -1; f <= 5; ++f)
    for (int pr = 0; pr < (f < 0 ? 1 : 2); ++pr)
      for (int R : {2, 4})
        for (int D : {2, 3, 4}) {
          cudaFuncAttributes fa;
          const void* fn = group_kernel_for(f, R, D, pr == 1);
          if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) {
            release();
            return QGEMV_ERR_CUDA;
          }
          size_t& mx = f < 0 ? h->group_smem_max[R >= 4 ? 1 : 0][d_index(D)]
                             : h->group1_smem_max[f][pr][R >= 4 ? 1 : 0][d_index(D)];
          mx = h->smem_optin - std::min(h->smem_optin, fa.sharedSizeBytes);
          if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(mx)) != cudaSuccess) {
            release();
            return QGEMV_ERR_CUDA;
          }
        }
  for (int f = 0; f < 6; ++f)
    for (int D : {2, 3}) {
      cudaFuncAttributes fa;
      const void* fn = batch_kernel_for(f, D);
      if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) {
        release();
        return QGEMV_ERR_CUDA;
      }
      size_t& mx = h->batch_smem_max[f][D - 2];
      mx = h->smem_optin - std::min(h->smem_optin, fa.sharedSizeBytes);
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(mx)) != cudaSuccess) {
        release();
        return QGEMV_ERR_CUDA;
      }
    }
  // The tensor-core GEMM needs TMA descriptors, encoded by the driver; without the entry point
  // qgemv_run_gemm keeps to the batch path.
  {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      h->encode_tiled = fn;
    cudaGetLastError();
  }
  for (int BT : {64, 128, 256}) {
    if (cudaFuncSetAttribute(tc_kernel_for(BT), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(tc_smem_bytes(BT))) != cudaSuccess) {
      release();
      return QGEMV_ERR_CUDA;
    }
    for (int cs : {8, 4, 2}) {  // the largest cluster of these CTAs that the GPU can place
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(cs), 1, 1);
      cfg.blockDim = dim3(kTcThreads, 1, 1);
      cfg.dynamicSmemBytes = tc_smem_bytes(BT);
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = static_cast<unsigned>(cs);
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int nc = 0;
      if (cudaOccupancyMaxActiveClusters(&nc, tc_kernel_for(BT), &cfg) == cudaSuccess && nc >= 1) {
        h->tc_cluster_max[BT > 128 ? 2 : BT > 64 ? 1 : 0] = cs;
        break;
      }
      cudaGetLastError();
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
  return launch_single(*h, fmt, x, W, N, K, y, stream);
}

qgemv_status_t qgemv_run_batch(qgemv_handle_t hh, qgemv_format_t fmt, const void* x, int M, const void* W, int64_t N,
                               int64_t K, float* y, cudaStream_t stream) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  qgemv_status_t st = validate(h, fmt, W, N, K);
  if (st != QGEMV_OK) return st;
  if (!x || !y || M < 1 || M > QGEMV_MAX_BATCH) return QGEMV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15) return QGEMV_ERR_MISALIGNED;
  const int f = static_cast<int>(fmt);
  int64_t rb1 = 0, rb2 = 0;
  const int64_t Wk = (K / 256 + kBatchColSB - 1) / kBatchColSB;
  // The batch kernel: two or more vectors, rows whose byte length is a multiple of 16, its
  // column sums in the workspace.  Otherwise each vector runs the single-vector path (which
  // is also the faster one for a single vector).
  const int warps = kBatchThreads / 32;
  const bool fmt_ok_b = f >= 0 && f < 6;
  int D = 3;
  while (fmt_ok_b && D > 2 && batch_smem_bytes(f, warps, D) > h->batch_smem_max[f][D - 2]) --D;
  // Below 4096 rows a warp's 16-row tiles hold a row or two, and the kernel's latency (a few
  // dependent copy rounds plus the column reduction) exceeds two or three short launches.
  const bool worth = M >= 4 || N >= 4096 || h->force_path == 1;
  const bool batch = M > 1 && worth && fmt_ok_b && h->force_path != 2 && stream_rows(f, K, rb1, rb2) &&
                     batch_smem_bytes(f, warps, D) <= h->batch_smem_max[f][D - 2] &&
                     (Wk == 1 || static_cast<double>(M) * N * Wk <= static_cast<double>(kWsFloats));
  if (!batch) {
    for (int m = 0; m < M; ++m) {
      st = launch_single(*h, f, static_cast<const uint16_t*>(x) + m * K, W, N, K, y + m * N, stream);
      if (st != QGEMV_OK) return st;
    }
    return QGEMV_OK;
  }
  int64_t ranges = std::max<int64_t>(1, h->sms / Wk);
  ranges = std::min<int64_t>(ranges, (N + kBatchRows - 1) / kBatchRows);
  ranges = std::max<int64_t>(1, std::min<int64_t>(ranges, kMaxRanges));
  if (N / ranges >= 0x7ffffffe) return QGEMV_ERR_BAD_SHAPE;
  const size_t smem = batch_smem_bytes(f, warps, D);
  BatchArgs a{};
  a.W = static_cast<const uint8_t*>(W);
  a.W2 = (f == F_NVFP4) ? a.W + N * (K / 2) : nullptr;
  a.x = static_cast<const uint16_t*>(x);
  a.y = y;
  a.N = N;
  a.M = M;
  a.K = static_cast<int>(K);
  a.nsb = static_cast<int>(K / 256);
  a.Wk = static_cast<int>(Wk);
  a.rows_q = static_cast<int>(N / ranges);
  a.rows_rem = static_cast<int>(N % ranges);
  a.row_bytes = rb1;
  a.row_bytes2 = rb2;
  a.ws = h->ws;
  a.cnt = h->cnt;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ranges * Wk), 1, 1);
  cfg.blockDim = dim3(32 * warps, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (h->pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  void* args[] = {&a};
  if (cudaLaunchKernelExC(&cfg, batch_kernel_for(f, D), args) != cudaSuccess) {
    cudaGetLastError();
    return QGEMV_ERR_CUDA;
  }
  return QGEMV_OK;
}

qgemv_status_t qgemv_run_gemm(qgemv_handle_t hh, qgemv_format_t fmt, const void* x, int64_t M, const void* W, int64_t N,
                              int64_t K, float* y, cudaStream_t stream) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  qgemv_status_t st = validate(h, fmt, W, N, K);
  if (st != QGEMV_OK) return st;
  if (!x || !y || M < 1) return QGEMV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15) return QGEMV_ERR_MISALIGNED;
  const int f = static_cast<int>(fmt);
  const int BT = M > 128 ? 256 : M > 64 ? 128 : 64;
  const int BK = tc_bk(BT);
  const bool tc = f == F_NVFP4 && M > QGEMV_MAX_BATCH && K % BK == 0 && h->encode_tiled && h->force_path != 2 &&
                  tc_smem_bytes(BT) <= h->smem_optin;
  if (!tc) {
    for (int64_t m0 = 0; m0 < M; m0 += QGEMV_MAX_BATCH) {
      const int mb = static_cast<int>(std::min<int64_t>(QGEMV_MAX_BATCH, M - m0));
      st = qgemv_run_batch(hh, fmt, static_cast<const uint16_t*>(x) + m0 * K, mb, W, N, K, y + m0 * N, stream);
      if (st != QGEMV_OK) return st;
    }
    return QGEMV_OK;
  }
  if (M > 0x7fffffff || K > 0x7fffffff) return QGEMV_ERR_BAD_SHAPE;
  const int64_t ntt = (M + BT - 1) / BT, nwt = (N + kTcRows - 1) / kTcRows;
  if (ntt * nwt > 0x7fffffff) return QGEMV_ERR_BAD_SHAPE;
  // X as a 2-D tensor (K innermost, M rows), read in boxes of 64 x BT with the 128-byte swizzle
  CUtensorMap map;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(BT)};  // one 128-byte swizzle row
  const cuuint32_t estr[2] = {1, 1};
  using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*, const cuuint64_t*,
                                const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  if (reinterpret_cast<EncodeFn>(h->encode_tiled)(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims,
                                                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return QGEMV_ERR_CUDA;
  // Split K over the CTAs of a cluster when the tiles fill fewer than all SMs: as many splits
  // as whole waves of tiles fit, at least four K-blocks each, at most the largest cluster.
  const int64_t tiles = ntt * nwt, nk = K / BK;
  int64_t ks = 1;
  if (tiles < h->sms)
    ks = std::min<int64_t>({h->sms / tiles, std::max<int64_t>(1, nk / 4), h->tc_cluster_max[BT > 128 ? 2 : BT > 64 ? 1 : 0]});
  int64_t kb_per = (nk + ks - 1) / ks;
  while (ks > 1 && (ks - 1) * kb_per >= nk) --ks;  // every split gets at least one K-block
  TcArgs a{};
  a.W = static_cast<const uint8_t*>(W);
  a.S = a.W + N * (K / 2);
  a.y = y;
  a.N = N;
  a.T = static_cast<int>(M);
  a.K = static_cast<int>(K);
  a.n_ttiles = static_cast<int>(ntt);
  a.ks = static_cast<int>(ks);
  a.kb_per = static_cast<int>(kb_per);
  a.err = h->err;
  a.spin_ns = h->spin_ns;
  a.stall = h->test_stall;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * ks), 1, 1);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = tc_smem_bytes(BT);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(ks);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&map, &a};
  if (cudaLaunchKernelExC(&cfg, tc_kernel_for(BT), args) != cudaSuccess) {
    cudaGetLastError();
    return QGEMV_ERR_CUDA;
  }
  return QGEMV_OK;
}

qgemv_status_t qgemv_run_group(qgemv_handle_t hh, const void* x, int64_t K, int count, const qgemv_problem_t* probs,
                               cudaStream_t stream) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h || !probs || !x || count < 1 || count > kMaxGroup) return QGEMV_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(x) & 15) return QGEMV_ERR_MISALIGNED;
  Problem ps[kMaxGroup];
  int nvfp4 = 0;
  for (int i = 0; i < count; ++i) {
    const qgemv_problem_t& q = probs[i];
    const int f = static_cast<int>(q.fmt);
    qgemv_status_t st = validate(h, f, q.packed_W, q.N, K);
    if (st != QGEMV_OK) return st;
    if (!q.y || q.swiglu < 0 || q.swiglu > 1 || q.out < QGEMV_OUT_F32 || q.out > QGEMV_OUT_BF16)
      return QGEMV_ERR_INVALID_ARG;
    if (q.swiglu && !q.packed_W_up) return QGEMV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q.y) | reinterpret_cast<uintptr_t>(q.packed_W_up)) & 15) return QGEMV_ERR_MISALIGNED;
    nvfp4 += f == F_NVFP4;
    ps[i].f = f;
    ps[i].W = q.packed_W;
    ps[i].WB = q.swiglu ? q.packed_W_up : nullptr;
    ps[i].N = q.N;
    ps[i].y = q.y;
    ps[i].alpha = q.alpha;
    ps[i].beta = q.beta;
    ps[i].ydt = static_cast<int>(q.out);
    ps[i].pair = q.swiglu;
  }
  if (nvfp4 != 0 && nvfp4 != count) return QGEMV_ERR_INVALID_ARG;  // one x: bf16 for NVFP4, fp16 otherwise
  // Streaming-eligible matrices share one launch; the rest run warp per row.
  Problem sp[kMaxGroup];
  int ns = 0, nr = 0, rw[kMaxGroup];
  for (int i = 0; i < count; ++i) {
    int64_t rb1, rb2;
    if (h->force_path != 2 && stream_rows(ps[i].f, K, rb1, rb2))
      sp[ns++] = ps[i];
    else
      rw[nr++] = i;
  }
  GroupPlan gp;
  if (ns > 0 && !plan_stream(*h, sp, ns, K, true, gp)) {
    for (int i = 0; i < count; ++i) rw[i] = i;  // no ring shape fits: everything warp per row
    nr = count;
    ns = 0;
  }
  if (ns > 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gp.grid, 1, 1);
    cfg.blockDim = dim3(gp.threads, 1, 1);
    cfg.dynamicSmemBytes = gp.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (h->pdl) {
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
    }
    for (int i = 0; i < ns; ++i) gp.ga.p[i].x = static_cast<const uint16_t*>(x);
    void* args[] = {&gp.ga};
    if (cudaLaunchKernelExC(&cfg, group_kernel_for(gp.fmt, gp.R, gp.D, gp.pairs), args) != cudaSuccess) {
      cudaGetLastError();
      return QGEMV_ERR_CUDA;
    }
  }
  for (int j = 0; j < nr; ++j) {
    const Problem& q = ps[rw[j]];
    Plan pl;
    rowwarp_plan(*h, q.N, pl);
    RowArgs ra{static_cast<const uint8_t*>(q.W), static_cast<const uint16_t*>(x), q.y, q.N, K, q.alpha, q.beta,
               q.ydt, q.pair, static_cast<const uint8_t*>(q.WB)};
    launch_rowwarp_any(q.f, pl, ra, stream);
    if (cudaGetLastError() != cudaSuccess) return QGEMV_ERR_CUDA;
  }
  return QGEMV_OK;
}

qgemv_status_t qgemv_run_ex(qgemv_handle_t h, qgemv_format_t fmt, const void* x, const void* packed_W, int64_t N,
                            int64_t K, float alpha, float beta, void* y, qgemv_out_t out, cudaStream_t stream) {
  qgemv_problem_t p = {};
  p.fmt = fmt;
  p.packed_W = packed_W;
  p.packed_W_up = nullptr;
  p.N = N;
  p.y = y;
  p.alpha = alpha;
  p.beta = beta;
  p.out = out;
  p.swiglu = 0;
  return qgemv_run_group(h, x, K, 1, &p, stream);
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
