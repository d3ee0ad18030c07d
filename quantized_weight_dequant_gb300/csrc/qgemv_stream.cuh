// Streaming GEMV kernel.
//
// The row range of a CTA is covered by P row groups x Wk K-columns of warps.  Warp (p, wk)
// owns K-column wk (2048 elements = 8 superblocks): each lane keeps the activations of its
// 64-element piece in registers for the whole kernel, and the warp walks down the rows of
// its row group, R rows per stage, streaming only its own slice of each row.
//  * Weights reach shared memory through a private ring of D stages per warp, filled with
//    16-byte cp.async copies (cache-global): lane l copies bytes [16l + 512j, +16) of each
//    row slice, with the base+offset address forms and the per-lane predicates computed
//    once.  A stage is consumed after cp.async.wait_group, which the hardware tracks per
//    thread: a warp waiting for data stalls on its scoreboard and takes no issue slots
//    from warps that are decoding.
//  * Each lane decodes its piece of each row of a stage (qgemv_decode.cuh).  The R row
//    sums are reduced across the warp together: the first butterfly steps exchange whole
//    rows, so 2 rows take 5 shuffles and 4 rows take 6 (instead of 5 per row).
//    Rows past the end of the row group in its last stage are decoded from stale ring
//    bytes and dropped; lanes past a short last K-column are zeroed.
//  * The Wk partial sums of a row are added in a fixed order in shared memory at the end,
//    so results are bitwise reproducible.
//  * x is staged once per CTA in shared memory, in the decoders' form (fp16 pairs for the
//    integer-code formats and TQ1_0, scaled f16 for NVFP4), then copied by each lane to
//    registers.  NVFP4 elements the scaled form does not hold exactly are corrected per
//    lane from their residuals.
//  * Under programmatic dependent launch the first weight stages are requested before the
//    wait for the previous kernel (weights are not written by it); x is read after it.
//  * The body is shared by the single-matrix kernel (fp32 row sums stored as they are) and
//    the grouped kernel (several matrices of possibly different formats sharing x, one per
//    CTA range, with the general epilogue out = alpha r + beta out in fp32/fp16/bf16, and
//    the SwiGLU pairing of a gate and an up matrix).
#pragma once
#include <cuda_fp16.h>

#include <cstdint>

#include "qgemv_decode.cuh"
#include "qgemv_epilogue.cuh"
#include "qgemv_ptx.cuh"

// Optional tracing hooks for timeline studies: empty unless defined before this header.
#ifndef QG_TRACE
#define QG_TRACE(k)
#endif
#ifndef QG_TRACE_END
#define QG_TRACE_END()
#endif

namespace qg {

constexpr int kDevErrTimeout = 1;

struct StreamArgs {
  const uint8_t* W;     // stream 1: rows of packed blocks / NVFP4 nibbles
  const uint8_t* W2;    // stream 2: NVFP4 scales (null otherwise)
  const uint16_t* x;    // activations (fp16, bf16 for NVFP4)
  void* y;              // fp32 row sums (single-matrix kernel); grouped kernel: see ydt
  int64_t N;            // rows (virtual rows, 2 per output, with pair = 1)
  int rows_q, rows_rem; // units (rows; pairs with pair = 1) = ranges * rows_q + rows_rem:
                        // range b has rows_q units (+1 if b < rows_rem)
  int64_t row_bytes, row_bytes2;  // bytes per row of stream 1 / 2 (multiples of 16)
  int nsb;              // superblocks per row
  int Wk;               // K-columns (warps per row group) = ceil(nsb / 8)
  int P;                // row groups per CTA
  int red_rows;         // rows of the reduction buffer (>= rows of any CTA)
  int* err;
  uint64_t spin_ns;
  int test_stall;       // 1: warp 0 of CTA 0 also waits, bounded, on a barrier nothing completes
  int pdl;              // programmatic dependent launch: 0 off; 1 on, weight stages requested
                        // before the wait for the previous kernel; 2 on, x first (as with 0)
  // Split mode (split = 1): CTA b takes K-column b % Wk of the rows of row range b / Wk, all
  // its warps on that column (P = warps).  With Wk > 1 the column sums go to ws[kc * N + row]
  // and the last CTA of a row range (counted in cnt[range], left at 0 again) adds them.
  int split;
  float* ws;
  int* cnt;
  // Epilogue of the grouped kernel: out = alpha * r + beta * out (out is not read when
  // beta == 0), stored as ydt (0 fp32, 1 fp16, 2 bf16, round to nearest even).  r is the row
  // sum; with pair = 1 (SwiGLU) virtual row 2n is row n of the gate matrix (W, W2) and
  // virtual row 2n + 1 row n of the up matrix (WB, WB2), and r = silu(gate sum) * up sum.
  float alpha, beta;
  int ydt;
  int pair;
  const uint8_t* WB;
  const uint8_t* WB2;
};

// Grouped launch: CTAs [cta_end[i-1], cta_end[i]) run matrix i, of format fmt[i].
constexpr int kMaxGroup = 8;
struct GroupArgs {
  int count;
  int cta_end[kMaxGroup];
  int fmt[kMaxGroup];
  StreamArgs p[kMaxGroup];
};

__device__ __forceinline__ void emit(const StreamArgs& a, int64_t n, float r) {
  emit_out(a.y, a.ydt, a.alpha, a.beta, n, r);
}

// The Wk column sums of virtual row `row` (split mode), added in column order.
__device__ __forceinline__ float column_sum(const StreamArgs& a, int64_t row) {
  float v[16];  // all column sums of the row in flight at once (Wk <= 16)
#pragma unroll
  for (int w = 0; w < 16; ++w) v[w] = w < a.Wk ? __ldcg(a.ws + w * a.N + row) : 0.f;
  float s = v[0];
#pragma unroll
  for (int w = 1; w < 16; ++w) s += v[w];  // the zero padding adds nothing
  return s;
}

template <class Dec>
__host__ __device__ constexpr int slice_bytes() {
  return 8 * Dec::kSB + 8 * Dec::kSB2;
}

// Shared memory: [rings: warps * D * R * slice][reduction buffer][x staging: q (2K bytes
// and 16 bytes of padding per 64 values), e (K/32 floats)][decoder area: coef_sb bytes per
// superblock of the staged x][never-completing barrier], each part 16-byte aligned.
struct StreamSmem {
  size_t red, xq, xe, xc, bar, total;
};
__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~static_cast<size_t>(15); }
__host__ __device__ inline StreamSmem stream_smem(int warps, int D, int R, int slice, int Wk, int red_rows, int K,
                                                  int coef_sb) {
  StreamSmem m;
  m.red = static_cast<size_t>(warps) * D * R * slice;
  m.xq = align16(m.red + (Wk > 1 ? static_cast<size_t>(red_rows) * Wk * 4 : 0));
  m.xe = align16(m.xq + static_cast<size_t>(K) * 2 + static_cast<size_t>(K / 64) * 16);
  m.xc = align16(m.xe + static_cast<size_t>(K / 32) * 4);
  m.bar = align16(m.xc + static_cast<size_t>(K / 256) * coef_sb);
  m.total = m.bar + 16;
  return m;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// cp_async16 at [dst + DOFF] <- [src + SOFF] when p != 0 (a predicated copy, no branch).
template <int DOFF, int SOFF>
__device__ __forceinline__ void cp_async16_if(uint32_t dst, const void* src, uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t"
      "@q cp.async.cg.shared.global [%0+%3], [%1+%4], 16;\n\t}" ::"r"(dst),
      "l"(src), "r"(p), "n"(DOFF), "n"(SOFF)
      : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Sum of v[0..R) over the warp; lane l ends up holding the total of row l / (32 / R).
template <int R>
__device__ __forceinline__ float reduce_rows(const float (&v)[R], int lane) {
  float t;
  if constexpr (R == 1) {
    t = v[0];
  } else if constexpr (R == 2) {
    const bool up = lane & 16;
    t = (up ? v[1] : v[0]) + __shfl_xor_sync(0xffffffffu, up ? v[0] : v[1], 16);
  } else {
    static_assert(R == 4, "rows per stage: 1, 2 or 4");
    const bool up = lane & 16;
    const float k0 = (up ? v[2] : v[0]) + __shfl_xor_sync(0xffffffffu, up ? v[0] : v[2], 16);
    const float k1 = (up ? v[3] : v[1]) + __shfl_xor_sync(0xffffffffu, up ? v[1] : v[3], 16);
    const bool up8 = lane & 8;
    t = (up8 ? k1 : k0) + __shfl_xor_sync(0xffffffffu, up8 ? k0 : k1, 8);
  }
#pragma unroll
  for (int o = 32 / R / 2; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;
}

// One CTA's work: CTA `cta` of the launch (or of its matrix in a grouped launch).  MODE 0:
// the fp32 row sums are stored; 1: the grouped kernel's epilogue, pairs decided at run time
// (a.pair); 2: the same for launches whose matrices are all SwiGLU pairs.
template <class Dec, int R, int D, int MODE>
__device__ __forceinline__ void stream_body(const StreamArgs& a, const int cta, uint8_t* smem) {
  QG_TRACE(0);
  constexpr int SB = Dec::kSB, SB2 = Dec::kSB2, SLICE = slice_bytes<Dec>();
  constexpr int STAGE = R * SLICE;
  constexpr int J1 = (8 * SB / 16 + 31) / 32, J2 = (8 * SB2 / 16 + 31) / 32;  // copies per lane per row
  constexpr int LPR = 32 / R;  // lanes per row after the reduction
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  // Fused mode: warp = (row group p, K-column wk) over all Wk columns of the CTA's rows.
  // Split mode: every warp of the CTA is on K-column blockIdx.x % Wk.
  const int p = a.split ? warp : warp / a.Wk;
  constexpr bool GEN = MODE > 0;
  const unsigned ucta = GEN ? static_cast<unsigned>(cta) : blockIdx.x, uWk = static_cast<unsigned>(a.Wk);
  const int wk = a.split ? static_cast<int>(ucta % uWk) : warp % a.Wk;
  const int kc0 = a.split ? wk : 0, kc1 = a.split ? wk + 1 : a.Wk;  // K-columns this CTA reads

  // Contiguous row ranges: range b, then row group p within it (no 64-bit division), in
  // units of u rows (a gate/up pair of virtual rows with pair = 1).
  const bool pair = MODE == 2 || (MODE == 1 && R >= 2 && a.pair);
  const int b = a.split ? static_cast<int>(ucta / uWk) : static_cast<int>(ucta);
  int64_t r_lo, p_lo;
  int ncta, nrows;
  if (pair) {
    r_lo = 2 * (static_cast<int64_t>(b) * a.rows_q + min(b, a.rows_rem));
    const int ncu = a.rows_q + (b < a.rows_rem ? 1 : 0);
    const int pq = ncu / a.P, prem = ncu % a.P;
    ncta = 2 * ncu;
    p_lo = r_lo + 2 * (p * pq + min(p, prem));
    nrows = 2 * (pq + (p < prem ? 1 : 0));
  } else {
    r_lo = static_cast<int64_t>(b) * a.rows_q + min(b, a.rows_rem);
    ncta = a.rows_q + (b < a.rows_rem ? 1 : 0);
    const int pq = ncta / a.P, prem = ncta % a.P;
    p_lo = r_lo + p * pq + min(p, prem);
    nrows = pq + (p < prem ? 1 : 0);
  }
  const int ncols = min(8, a.nsb - 8 * wk);
  const int col = lane >> 2;
  const bool active = col < ncols;

  // The staging buffer holds the K-columns this CTA reads: all of x (fused) or one column.
  const int Kx = a.split ? min(2048, 256 * a.nsb) : 256 * a.nsb;
  const StreamSmem L = stream_smem(nwarps, D, R, SLICE, a.Wk, a.red_rows, Kx, Dec::kCoefSB);
  uint8_t* ring = smem + static_cast<size_t>(warp) * D * STAGE;
  float* red = reinterpret_cast<float*>(smem + L.red);
  const XStage X{reinterpret_cast<uint16_t*>(smem + L.xq), reinterpret_cast<float*>(smem + L.xe),
                 reinterpret_cast<int*>(smem + L.xc)};
  uint64_t* never_bar = reinterpret_cast<uint64_t*>(smem + L.bar);

  pdl_launch_dependents();  // the next kernel may start copying its weights right away
  if (a.test_stall && cta == 0 && warp == 0) {
    if (lane == 0) {
      mbar_init(smem_u32(never_bar), 1);
      fence_mbar_init();
      if (!mbar_wait_bounded(smem_u32(never_bar), 0, a.spin_ns)) atomicOr(a.err, kDevErrTimeout);
    }
    __syncwarp();
  }

  // Copy set-up: lane chunk j of a row slice is bytes [16 * lane + 512 * j, +16).
  const int n1 = ncols * SB / 16, n2 = ncols * SB2 / 16;
  uint32_t ok1[J1], ok2[J2 > 0 ? J2 : 1];
#pragma unroll
  for (int j = 0; j < J1; ++j) ok1[j] = lane + 32 * j < n1;
#pragma unroll
  for (int j = 0; j < J2; ++j) ok2[j] = lane + 32 * j < n2;
  // Rows of a stage are requested in order through running pointers; row bytes fit in 32 bits.
  const int rb1 = static_cast<int>(a.row_bytes), rb2 = static_cast<int>(a.row_bytes2);
  // Pairs: a warp streams the gate rows of its outputs (from gi), then their up rows (from
  // gb), one matrix at a time; both sums go to the workspace / reduction buffer, where the
  // epilogue combines them.
  const uint8_t* gi1 = a.W + p_lo * a.row_bytes + static_cast<int64_t>(wk) * 8 * SB + 16 * lane;
  const uint8_t* gi2 = (SB2 > 0) ? a.W2 + p_lo * a.row_bytes2 + static_cast<int64_t>(wk) * 8 * SB2 + 16 * lane : a.W;
  const uint8_t* gb1 = a.W;
  const uint8_t* gb2 = a.W;
  if (pair) {
    const int64_t wrow = p_lo / 2;
    gi1 = a.W + wrow * a.row_bytes + static_cast<int64_t>(wk) * 8 * SB + 16 * lane;
    gb1 = a.WB + wrow * a.row_bytes + static_cast<int64_t>(wk) * 8 * SB + 16 * lane;
    if (SB2 > 0) {
      gi2 = a.W2 + wrow * a.row_bytes2 + static_cast<int64_t>(wk) * 8 * SB2 + 16 * lane;
      gb2 = a.WB2 + wrow * a.row_bytes2 + static_cast<int64_t>(wk) * 8 * SB2 + 16 * lane;
    }
  }
  const uint32_t ring_sa = smem_u32(ring), ring_end = ring_sa + D * STAGE;
  const int nst = (nrows + R - 1) / R, nfull = nrows / R, tail = nrows - nfull * R;
  const int np = nrows / 2;  // pairs: outputs of this warp

  // This lane's copies of one row slice: to shared address d, from row pointers s1 / s2.
  auto copy_row = [&](uint32_t d, const uint8_t* s1, const uint8_t* s2) {
#pragma unroll
    for (int j = 0; j < J1; ++j) {
      switch (j) {  // immediate offsets: 512 j
        case 0: cp_async16_if<0, 0>(d, s1, ok1[j]); break;
        case 1: cp_async16_if<512, 512>(d, s1, ok1[j]); break;
        case 2: cp_async16_if<1024, 1024>(d, s1, ok1[j]); break;
        case 3: cp_async16_if<1536, 1536>(d, s1, ok1[j]); break;
        case 4: cp_async16_if<2048, 2048>(d, s1, ok1[j]); break;
      }
    }
    if (SB2 > 0) {
#pragma unroll
      for (int j = 0; j < J2; ++j) cp_async16_if<8 * SB, 0>(d + 512 * j, s2 + 512 * j, ok2[j]);
    }
  };
  // Requests stage st (issued in order) into the ring slot at shared address slot_sa: R rows,
  // or the `tail` rows of the short last stage (its other slots keep stale bytes, which are
  // decoded and dropped).
  auto issue = [&](int st, uint32_t slot_sa) {
    const uint32_t d = slot_sa + 16 * lane;
    if constexpr (GEN && R >= 2) {
      if (pair) {  // position q: gate row q (q < np) or up row q - np
        const int q0 = st * R;
        if (q0 + R <= np || (q0 >= np && q0 + R <= nrows)) {  // a whole stage of one matrix
          const bool up = q0 >= np;
          const int64_t j = up ? q0 - np : q0;
          const uint8_t* s1 = (up ? gb1 : gi1) + j * rb1;
          const uint8_t* s2 = (up ? gb2 : gi2) + j * rb2;
#pragma unroll
          for (int r = 0; r < R; ++r) copy_row(d + r * SLICE, s1 + r * rb1, s2 + r * rb2);
        } else {  // the stage that crosses from gate to up rows, or the short last one
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const int q = q0 + r;
            if (q < nrows) {
              const bool up = q >= np;
              const int64_t j = up ? q - np : q;
              copy_row(d + r * SLICE, (up ? gb1 : gi1) + j * rb1, (up ? gb2 : gi2) + j * rb2);
            }
          }
        }
        cp_async_commit();
        return;
      }
    }
    if (st < nfull) {
#pragma unroll
      for (int r = 0; r < R; ++r) copy_row(d + r * SLICE, gi1 + r * rb1, gi2 + r * rb2);
      gi1 += R * rb1;
      gi2 += R * rb2;
    } else if (st < nst) {
      for (int r = 0; r < tail; ++r) copy_row(d + r * SLICE, gi1 + r * rb1, gi2 + r * rb2);
    }
    cp_async_commit();
  };
  static_assert(J1 <= 5, "row slice of at most 160 16-byte chunks");

  // Activations: thread t loads 16-byte pieces t, t + blockDim.x, ... of x (coalesced, four
  // at a time in flight) and converts them into the staging buffer.  Without programmatic
  // dependent launch the first loads are issued ahead of the weight stages, so they are not
  // queued behind them.  With it, the weight stages are requested before the wait for the
  // previous kernel (whose output x may be), and x after.  The piece count is a multiple of
  // 32, so every warp runs the same number of conversions (they shuffle within groups of
  // lanes) and the predicates below are warp-uniform.  These loops run once per launch and
  // are kept rolled: straight-line start-up code is fetched while the weight stream already
  // loads the memory system.
  // Pieces of the K-columns this CTA reads (32 per superblock, so whole warps drop out).
  const int pc0 = 256 * kc0, pc1 = 32 * min(a.nsb, 8 * kc1);
  const uint4* const xs = reinterpret_cast<const uint4*>(a.x) + pc0;
  const int npc = pc1 - pc0, nt = static_cast<int>(blockDim.x), tid = static_cast<int>(threadIdx.x);
  auto stage_x = [&](bool stages_after_first_loads) {
#pragma unroll 1
    for (int i0 = 0; i0 < npc; i0 += 4 * nt) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i0 + u * nt + tid < npc) v[u] = __ldcg(xs + i0 + u * nt + tid);
      if (stages_after_first_loads && i0 == 0) {
#pragma unroll 1
        for (int s = 0; s < D - 1; ++s) issue(s, ring_sa + s * STAGE);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i0 + u * nt + tid < npc) Dec::stage_piece(v[u], i0 + u * nt + tid, X);
    }
  };
  if (a.pdl == 1) {
#pragma unroll 1
    for (int s = 0; s < D - 1; ++s) issue(s, ring_sa + s * STAGE);
    pdl_wait();
    QG_TRACE(1);
    stage_x(false);
  } else {
    pdl_wait();  // at once without programmatic dependent launch
    QG_TRACE(1);
    stage_x(true);
  }
  __syncthreads();
  QG_TRACE(2);
  Dec dec;
  dec.init(lane & 3);
  dec.load_x(X, 8 * (wk - kc0) + col, lane & 3, active);  // superblock index within the buffer
  QG_TRACE(6);

  // Where row sums go: y (one K-column), the workspace (split mode) or the CTA's reduction
  // buffer (fused mode, stride Wk).
  float* const out = (a.Wk == 1 && !pair) ? static_cast<float*>(a.y) + p_lo
                     : a.split ? a.ws + wk * a.N + p_lo
                               : red + static_cast<int>(p_lo - r_lo) * a.Wk + wk;
  const int ostride = (a.Wk == 1 || a.split) ? 1 : a.Wk;

  uint32_t cs = ring_sa;                     // slot of stage st
  uint32_t is = ring_sa + (D - 1) * STAGE;   // slot for stage st + D - 1 (freed by st - 1)
  const uint32_t lo1 = col * SB, lo2 = 8 * SB + col * SB2;  // this lane's superblock in a row slice
  const bool writer = lane % LPR == 0;
  float* optr = out + (lane / LPR) * ostride;
  for (int st = 0; st < nst; ++st) {
    issue(st + D - 1, is);
    if (st == 0) QG_TRACE(7);
    cp_async_wait<D - 1>();
    __syncwarp();
    if (st == 0) QG_TRACE(3);
    typename Dec::Raw raw[R];
#pragma unroll
    for (int r = 0; r < R; ++r) raw[r] = dec.fetch(cs + lo1 + r * SLICE, cs + lo2 + r * SLICE);
    float v[R];
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] = dec.compute(raw[r]);
    if constexpr (Dec::kResidual) {
      // Elements of this lane's x that the staged form does not hold exactly (none for
      // typical inputs): their residuals times their weights, from the same ring slot.
      if (dec.has_residual()) {
#pragma unroll
        for (int r = 0; r < R; ++r) v[r] += dec.correction(cs + lo1 + r * SLICE, cs + lo2 + r * SLICE);
      }
    }
    __syncwarp();  // every lane is done with this slot before it is refilled
    is = cs;
    cs = (cs + STAGE == ring_end) ? ring_sa : cs + STAGE;
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] = active ? v[r] : 0.f;
    const float sum = reduce_rows<R>(v, lane) * Dec::kOut;  // the decoder's unit, once per row
    if (pair) {  // virtual row 2j (gate) or 2j + 1 (up) of the warp's output j
      const int q = st * R + lane / LPR;
      if (writer && q < nrows) out[(q < np ? 2 * q : 2 * (q - np) + 1) * ostride] = sum;
    } else if (GEN && a.Wk == 1) {  // final sums: the epilogue
      const int rr = st * R + lane / LPR;
      if (writer && rr < nrows) emit(a, p_lo + rr, sum);
    } else {
      if (writer && st * R + lane / LPR < nrows) *optr = sum;
      optr += R * ostride;
    }
  }
  cp_async_wait<0>();
  QG_TRACE(4);

  if (a.Wk > 1 && !a.split) {
    __syncthreads();
    if (pair) {
      for (int i = threadIdx.x; i < ncta / 2; i += blockDim.x) {
        float g = 0.f, up = 0.f;
        for (int w = 0; w < a.Wk; ++w) g += red[(2 * i) * a.Wk + w];
        for (int w = 0; w < a.Wk; ++w) up += red[(2 * i + 1) * a.Wk + w];
        emit(a, (r_lo >> 1) + i, silu_f(g) * up);
      }
    } else {
      for (int i = threadIdx.x; i < ncta; i += blockDim.x) {
        float s = 0.f;
        for (int w = 0; w < a.Wk; ++w) s += red[i * a.Wk + w];
        if (GEN)
          emit(a, r_lo + i, s);
        else
          static_cast<float*>(a.y)[r_lo + i] = s;
      }
    }
  } else if (a.Wk > 1 || pair) {
    // Publish this CTA's column sums, then count the CTA in; the last of the Wk CTAs of the
    // row range adds the Wk column sums of each row in column order and resets the count.
    __shared__ int last;
    __syncthreads();  // every column sum of this CTA is written
    if (threadIdx.x == 0) {
      // acq_rel: releases the CTA's column sums (cumulative over the barrier) with the count,
      // and acquires the other CTAs' sums for the CTA that turns out to be last.
      int old;
      asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(a.cnt + b) : "memory");
      last = old == a.Wk - 1;
    }
    __syncthreads();
    if (last) {
      if (pair) {
        for (int i = threadIdx.x; i < ncta / 2; i += blockDim.x)
          emit(a, (r_lo >> 1) + i, silu_f(column_sum(a, r_lo + 2 * i)) * column_sum(a, r_lo + 2 * i + 1));
      } else {
        for (int i = threadIdx.x; i < ncta; i += blockDim.x) {
          const float s = column_sum(a, r_lo + i);
          if (GEN)
            emit(a, r_lo + i, s);
          else
            static_cast<float*>(a.y)[r_lo + i] = s;
        }
      }
      if (threadIdx.x == 0) a.cnt[b] = 0;
    }
  }
  QG_TRACE(5);
  QG_TRACE_END();
}

// Single matrix: fp32 row sums.
template <class Dec, int R, int D>
__global__ void __launch_bounds__(512, 1) stream_kernel(const StreamArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  stream_body<Dec, R, D, 0>(a, static_cast<int>(blockIdx.x), smem);
}

// Grouped launch of matrices of one format (the common case: a smaller kernel than the
// mixed-format one below, whose six decoders crowd the instruction cache).
// PAIRS: every matrix of the launch is a SwiGLU pair (the pairing compiled in).
template <class Dec, int R, int D, bool PAIRS>
__global__ void __launch_bounds__(512, 1) group_kernel_1(const __grid_constant__ GroupArgs g) {
  extern __shared__ __align__(128) uint8_t smem[];
  int i = 0;
  while (i + 1 < g.count && static_cast<int>(blockIdx.x) >= g.cta_end[i]) ++i;
  stream_body<Dec, R, D, PAIRS ? 2 : 1>(g.p[i], static_cast<int>(blockIdx.x) - (i > 0 ? g.cta_end[i - 1] : 0), smem);
}

// Grouped launch: up to kMaxGroup matrices (any formats, one x) with the general epilogue.
template <int R, int D>
__global__ void __launch_bounds__(512, 1) group_kernel(const __grid_constant__ GroupArgs g) {
  extern __shared__ __align__(128) uint8_t smem[];
  int i = 0;
  while (i + 1 < g.count && static_cast<int>(blockIdx.x) >= g.cta_end[i]) ++i;
  const int cta = static_cast<int>(blockIdx.x) - (i > 0 ? g.cta_end[i - 1] : 0);
  const StreamArgs& a = g.p[i];
  switch (g.fmt[i]) {
    case F_Q4K: stream_body<DecQ4K, R, D, 1>(a, cta, smem); break;
    case F_Q5K: stream_body<DecQ5K, R, D, 1>(a, cta, smem); break;
    case F_Q6K: stream_body<DecQ6K, R, D, 1>(a, cta, smem); break;
    case F_Q80: stream_body<DecQ80, R, D, 1>(a, cta, smem); break;
    case F_TQ10: stream_body<DecTQ10, R, D, 1>(a, cta, smem); break;
    case F_NVFP4: stream_body<DecNVFP4, R, D, 1>(a, cta, smem); break;
  }
}

// One-format grouped kernels of one decoder: R in {2, 4}, D in {2, 3, 4}, pairs compiled in
// or not.
template <class Dec, bool PAIRS>
const void* group_kernel_1_table(int R, int D) {
  const int di = D >= 4 ? 2 : D >= 3 ? 1 : 0;
  static const void* const t[2][3] = {
      {reinterpret_cast<const void*>(&group_kernel_1<Dec, 2, 2, PAIRS>),
       reinterpret_cast<const void*>(&group_kernel_1<Dec, 2, 3, PAIRS>),
       reinterpret_cast<const void*>(&group_kernel_1<Dec, 2, 4, PAIRS>)},
      {reinterpret_cast<const void*>(&group_kernel_1<Dec, 4, 2, PAIRS>),
       reinterpret_cast<const void*>(&group_kernel_1<Dec, 4, 3, PAIRS>),
       reinterpret_cast<const void*>(&group_kernel_1<Dec, 4, 4, PAIRS>)}};
  return t[R >= 4 ? 1 : 0][di];
}

// Kernel table of one decoder: R in {1, 2, 4} rows per stage, D in {2, 3, 4} ring stages.
template <class Dec>
const void* stream_kernel_table(int R, int D) {
  const int ri = R >= 4 ? 2 : R >= 2 ? 1 : 0;
  const int di = D >= 4 ? 2 : D >= 3 ? 1 : 0;
  static const void* const t[3][3] = {
      {reinterpret_cast<const void*>(&stream_kernel<Dec, 1, 2>), reinterpret_cast<const void*>(&stream_kernel<Dec, 1, 3>),
       reinterpret_cast<const void*>(&stream_kernel<Dec, 1, 4>)},
      {reinterpret_cast<const void*>(&stream_kernel<Dec, 2, 2>), reinterpret_cast<const void*>(&stream_kernel<Dec, 2, 3>),
       reinterpret_cast<const void*>(&stream_kernel<Dec, 2, 4>)},
      {reinterpret_cast<const void*>(&stream_kernel<Dec, 4, 2>), reinterpret_cast<const void*>(&stream_kernel<Dec, 4, 3>),
       reinterpret_cast<const void*>(&stream_kernel<Dec, 4, 4>)}};
  return t[ri][di];
}

}  // namespace qg
