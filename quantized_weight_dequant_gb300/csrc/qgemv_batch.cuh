// Small-batch dequant GEMV: Y[m, n] = sum_k X[m, k] * dequant(W)[n, k] for M = 1..8
// activation vectors, every weight decoded once and used by all of them.
//
// At M = 1 the product is a matrix-vector product and the streaming kernel's integer dot
// products fit it best ("fp4_gemv" page: no MMA at M = 1); from a few vectors on, the same
// decoded weight meets several activations, which is what the tensor cores' mma.sync
// contraction does without any shared-memory round trip: the weights are decoded in
// registers straight into the B fragments of m16n8k16 (8 weight rows as its N) and the
// activation vectors are its M (16 slots, M of them used).
//
//  * Work split as in the streaming kernel's split mode: a CTA takes one 2048-wide
//    K-column of a row range; warp p takes row group p of the range, 8 rows per stage,
//    through a private ring of D stages filled with 16-byte cp.async copies.
//  * Activations: the CTA stages its K-column of all M vectors once, already in the
//    A-fragment order (lane (g, t4) reads the pair of fp16 values for vector g at its k
//    slots with one 8-byte shared load per k-step).  Unused vector slots hold zeros.
//  * Lane (g, t4) decodes row g of a stage, 64 elements of each superblock (chunk t4), and
//    gets back the sums of rows 2 t4 and 2 t4 + 1 for vector g from the accumulator.
//  * Q4_K: B = q * s_g, an exact integer <= 945 in fp16 (the 6-bit group scale folded in):
//    one LOP3 puts two nibbles into fp16 (1024 + q) / (1024 + 16 q), one fused multiply-add
//    scales and removes the offset.  The group minimum term sum_g m_g X_g goes through an
//    m16n8k8 product (A = the group sums of x split into two fp16 parts, B = m_g), and the
//    superblock scales d, dmin are applied to both sums in fp32 once per superblock.
//  * NVFP4: B = e2m1 * |e4m3 block scale|, exact in fp16; x (bf16) is staged as fp16 times
//    2^sigma per vector and K-column (sigma from the column's largest |x|), and the sums are
//    scaled back when written.
//  * Results: with one K-column they are written to Y; otherwise every CTA writes its
//    column sums to the workspace and the last CTA of the range adds them in column order.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "qgemv_decode.cuh"
#include "qgemv_ptx.cuh"
#include "qgemv_stream.cuh"

namespace qg {

constexpr int kBatchMax = 8;  // activation vectors (the MMA's M slots used)
constexpr int kBatchRows = 8;  // weight rows per stage (the MMA's N)

struct BatchArgs {
  const uint8_t* W;   // stream 1: packed blocks / NVFP4 nibbles
  const uint8_t* W2;  // stream 2: NVFP4 scales (null otherwise)
  const uint16_t* x;  // [M, K] fp16 (bf16 for NVFP4)
  float* y;           // [M, N] fp32
  int64_t N;
  int M;
  int K;
  int nsb;            // superblocks per row
  int Wk;             // K-columns = ceil(nsb / 8)
  int rows_q, rows_rem;  // range b has rows_q (+1 if b < rows_rem) rows
  int64_t row_bytes, row_bytes2;
  float* ws;          // Wk > 1: column sums [Wk][M][N]
  int* cnt;           // per-range arrival counts, zero between launches
};

// Shared memory: [rings: warps * D * 8 * slice][x fragments: 8 sb * 16 steps * 32 lanes * 8 B]
// [group sums (Q4_K): 8 sb * 32 lanes * 8 B][per-vector scales 2^-sigma: 8 floats][flag].
struct BatchSmem {
  size_t xa, xs, sc, total;
};
__host__ __device__ inline BatchSmem batch_smem(int warps, int D, int slice) {
  BatchSmem m;
  m.xa = static_cast<size_t>(warps) * D * kBatchRows * slice;
  m.xs = m.xa + 8 * 16 * 32 * 8;
  m.sc = m.xs + 8 * 32 * 8;
  m.total = m.sc + kBatchMax * 4 + 16;
  return m;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  const uint32_t z = 0u;  // vector slots 8..15 are unused
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(z), "r"(a2), "r"(z), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma1688(float (&d)[4], uint32_t a0, uint32_t b0) {
  const uint32_t z = 0u;
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(z), "r"(b0));
}
__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint2 lds_v2(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}

// Two small non-negative integers (< 1024) as the fp16 pair (lo, hi), exactly.
__device__ __forceinline__ uint32_t int2_to_h2(uint32_t lo, uint32_t hi) {
  return hsub2_u((lo | (hi << 16)) | 0x64006400u, 0x64006400u);
}

// ----------------------------------------------------------------------------- Q4_K
struct BatchQ4K {
  static constexpr int kSB = 144, kSB2 = 0;

  // x chunk of 4 fp16 values (elements e..e+3 of a superblock, e % 4 == 0) -> its slot in the
  // fragment buffer: k-step s and lane t4 part.  Byte j of chunk t4 holds element 64 t4 + j
  // (low nibble) and 64 t4 + 32 + j (high nibble); a 32-bit word of bytes b0..b3 gives the
  // pairs (b0, b2) and (b1, b3), so step 2i (low) / 2i + 1 (high) of word i reads elements
  // (base, base + 2) and (base + 1, base + 3), base = 64 t4 + 32 hi + 4 i.
  __device__ __forceinline__ static void chunk_slot(int e, int& step, int& t4, uint2& v, uint2 raw) {
    t4 = e >> 6;
    const int hi = (e >> 5) & 1, i = (e & 31) >> 2;
    step = 2 * i + hi;
    v.x = __byte_perm(raw.x, raw.y, 0x5410);  // (x0, x2)
    v.y = __byte_perm(raw.x, raw.y, 0x7632);  // (x1, x3)
  }

  // Lane (g, t4) of a warp: the superblock at shared address `blk` of row g; `hd0`, `hd1`
  // the first words (d, dmin) of rows 2 t4 and 2 t4 + 1; xa / xs its fragment addresses.
  __device__ __forceinline__ static void superblock(uint32_t blk, uint32_t hd0, uint32_t hd1, int t4,
                                                    uint32_t xa, uint32_t xs, float& acc0, float& acc1) {
    const uint4 hdr = lds_v4(blk);
    const uint4 q0 = lds_v4(blk + 16 + 32 * t4), q1 = lds_v4(blk + 32 + 32 * t4);
    // 6-bit scales and mins of groups 2 t4 and 2 t4 + 1 ("Kernel code" mask arithmetic)
    uint32_t sl, sh, ml, mh;
    {
      const int jl = 2 * t4, jh = 2 * t4 + 1;
      const int ql = jl & 3, qh = jh & 3;
      const uint32_t S0 = hdr.y, S1 = hdr.z, S2 = hdr.w;
      auto byte_of = [](uint32_t w, int q) { return (w >> (8 * q)) & 0xFFu; };
      if (t4 < 2) {
        sl = byte_of(S0, ql) & 63u;
        sh = byte_of(S0, qh) & 63u;
        ml = byte_of(S1, ql) & 63u;
        mh = byte_of(S1, qh) & 63u;
      } else {
        sl = (byte_of(S2, ql) & 15u) | ((byte_of(S0, ql) >> 6) << 4);
        sh = (byte_of(S2, qh) & 15u) | ((byte_of(S0, qh) >> 6) << 4);
        ml = (byte_of(S2, ql) >> 4) | ((byte_of(S1, ql) >> 6) << 4);
        mh = (byte_of(S2, qh) >> 4) | ((byte_of(S1, qh) >> 6) << 4);
      }
    }
    const uint32_t S = int2_to_h2(sl, sh);                       // (s_lo, s_hi)
    const uint32_t SL = __byte_perm(S, S, 0x1010);               // (s_lo, s_lo)
    const uint32_t SH = hmul2_u(__byte_perm(S, S, 0x3232), 0x2C002C00u);  // s_hi / 16
    const uint32_t CL = hmul2_u(SL, 0xE400E400u);                // -1024 s_lo
    const uint32_t CH = hmul2_u(SH, 0xE400E400u);                // -64 s_hi
    const uint32_t Bm = int2_to_h2(ml, mh);                      // (m_lo, m_hi)
    float dq[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t w0 = w[i], w8 = w[i] >> 8;
      const uint32_t l0 = hfma2_u((w0 & 0x000F000Fu) | 0x64006400u, SL, CL);
      const uint32_t l1 = hfma2_u((w8 & 0x000F000Fu) | 0x64006400u, SL, CL);
      const uint32_t h0 = hfma2_u((w0 & 0x00F000F0u) | 0x64006400u, SH, CH);
      const uint32_t h1 = hfma2_u((w8 & 0x00F000F0u) | 0x64006400u, SH, CH);
      const uint2 xl = lds_v2(xa + (2 * i) * 256), xh = lds_v2(xa + (2 * i + 1) * 256);
      mma16816(dq, xl.x, xl.y, l0, l1);
      mma16816(dq, xh.x, xh.y, h0, h1);
    }
    float dm[4] = {0.f, 0.f, 0.f, 0.f};
    const uint2 X = lds_v2(xs);  // group sums / 64: (hi parts), (lo parts)
    mma1688(dm, X.x, Bm);
    mma1688(dm, X.y, Bm);
    const float d0 = h2f(hd0), m0 = h2f(hd0 >> 16) * 64.f, d1 = h2f(hd1), m1 = h2f(hd1 >> 16) * 64.f;
    acc0 += fmaf(d0, dq[0], -m0 * dm[0]);
    acc1 += fmaf(d1, dq[1], -m1 * dm[1]);
  }
};

// ----------------------------------------------------------------------------- NVFP4
struct BatchNVFP4 {
  static constexpr int kSB = 128, kSB2 = 16;

  // Chunk t4 of a superblock is nibble bytes [32 t4, 32 t4 + 32) = elements 64 t4 + [0, 64);
  // word i (elements 64 t4 + 8 i + [0, 8)) feeds steps 2 i (elements +0..3) and 2 i + 1
  // (+4..7), each as the pairs (e, e + 1) and (e + 2, e + 3) of its cvt.e2m1x2 results.
  __device__ __forceinline__ static void chunk_slot(int e, int& step, int& t4, uint2& v, uint2 raw) {
    t4 = e >> 6;
    step = (e & 63) >> 2;
    v = raw;
  }

  __device__ __forceinline__ static void superblock(uint32_t nib, uint32_t sc, int t4, uint32_t xa, float (&dq)[4]) {
    const uint4 q0 = lds_v4(nib + 32 * t4), q1 = lds_v4(nib + 32 * t4 + 16);
    const uint32_t s4 = lds_u32(sc + 4 * t4) & 0x7F7F7F7Fu;  // |scale| of blocks 4 t4 .. 4 t4 + 3
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t sh = DecNVFP4::e4m3x2((s4 >> (8 * b)) & 0xFFu);
      const uint32_t sv = __byte_perm(sh, sh, 0x1010);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int i = 2 * b + u;
        uint32_t h[4];
        DecNVFP4::e2m1x8(w[i], h);
        const uint2 xl = lds_v2(xa + (2 * i) * 256), xh = lds_v2(xa + (2 * i + 1) * 256);
        mma16816(dq, xl.x, xl.y, hmul2_u(h[0], sv), hmul2_u(h[1], sv));
        mma16816(dq, xh.x, xh.y, hmul2_u(h[2], sv), hmul2_u(h[3], sv));
      }
    }
  }
};

template <class Fmt>
__host__ __device__ constexpr int batch_slice() {
  return 8 * Fmt::kSB + 8 * Fmt::kSB2;
}

template <class Fmt, int D>
__global__ void __launch_bounds__(256, 1) batch_kernel(const __grid_constant__ BatchArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int SB = Fmt::kSB, SB2 = Fmt::kSB2, SLICE = batch_slice<Fmt>();
  constexpr int STAGE = kBatchRows * SLICE;
  constexpr int J1 = (8 * SB / 16 + 31) / 32, J2 = (8 * SB2 / 16 + 31) / 32;
  constexpr bool kIsNVFP4 = SB2 > 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  const unsigned uWk = static_cast<unsigned>(a.Wk);
  const int wk = static_cast<int>(blockIdx.x % uWk), b = static_cast<int>(blockIdx.x / uWk);
  const int64_t r_lo = static_cast<int64_t>(b) * a.rows_q + min(b, a.rows_rem);
  const int ncta = a.rows_q + (b < a.rows_rem ? 1 : 0);
  const int pq = ncta / nwarps, prem = ncta % nwarps;
  const int64_t p_lo = r_lo + warp * pq + min(warp, prem);
  const int nrows = pq + (warp < prem ? 1 : 0);
  const int ncols = min(8, a.nsb - 8 * wk);  // superblocks in this K-column
  const BatchSmem L = batch_smem(nwarps, D, SLICE);
  const uint32_t ring_sa = smem_u32(smem) + static_cast<uint32_t>(warp) * D * STAGE, ring_end = ring_sa + D * STAGE;
  const uint32_t xa_sa = smem_u32(smem + L.xa), xs_sa = smem_u32(smem + L.xs);
  float* const vscale = reinterpret_cast<float*>(smem + L.sc);

  pdl_launch_dependents();

  // Copies: lane chunk j of a row slice is bytes [16 lane + 512 j, +16).
  const int n1 = ncols * SB / 16, n2 = ncols * SB2 / 16;
  uint32_t ok1[J1], ok2[J2 > 0 ? J2 : 1];
#pragma unroll
  for (int j = 0; j < J1; ++j) ok1[j] = lane + 32 * j < n1;
#pragma unroll
  for (int j = 0; j < J2; ++j) ok2[j] = lane + 32 * j < n2;
  const int rb1 = static_cast<int>(a.row_bytes), rb2 = static_cast<int>(a.row_bytes2);
  const uint8_t* gi1 = a.W + p_lo * a.row_bytes + static_cast<int64_t>(wk) * 8 * SB + 16 * lane;
  const uint8_t* gi2 = kIsNVFP4 ? a.W2 + p_lo * a.row_bytes2 + static_cast<int64_t>(wk) * 8 * SB2 + 16 * lane : a.W;
  const int nst = (nrows + kBatchRows - 1) / kBatchRows, nfull = nrows / kBatchRows;
  const int tail = nrows - nfull * kBatchRows;
  auto copy_row = [&](uint32_t d, const uint8_t* s1, const uint8_t* s2) {
#pragma unroll
    for (int j = 0; j < J1; ++j) {
      switch (j) {
        case 0: cp_async16_if<0, 0>(d, s1, ok1[j]); break;
        case 1: cp_async16_if<512, 512>(d, s1, ok1[j]); break;
        case 2: cp_async16_if<1024, 1024>(d, s1, ok1[j]); break;
        case 3: cp_async16_if<1536, 1536>(d, s1, ok1[j]); break;
        case 4: cp_async16_if<2048, 2048>(d, s1, ok1[j]); break;
      }
    }
    if constexpr (kIsNVFP4) {
#pragma unroll
      for (int j = 0; j < J2; ++j) cp_async16_if<8 * SB, 0>(d + 512 * j, s2 + 512 * j, ok2[j]);
    }
  };
  auto issue = [&](int st, uint32_t slot_sa) {
    const uint32_t d = slot_sa + 16 * lane;
    if (st < nfull) {
#pragma unroll
      for (int r = 0; r < kBatchRows; ++r) copy_row(d + r * SLICE, gi1 + r * rb1, gi2 + r * rb2);
      gi1 += kBatchRows * rb1;
      gi2 += kBatchRows * rb2;
    } else if (st < nst) {
      for (int r = 0; r < tail; ++r) copy_row(d + r * SLICE, gi1 + r * rb1, gi2 + r * rb2);
    }
    cp_async_commit();
  };
  static_assert(J1 <= 5, "row slice of at most 160 16-byte chunks");

  // Weight stages first (they do not depend on the previous kernel), then x.
#pragma unroll 1
  for (int s = 0; s < D - 1; ++s) issue(s, ring_sa + s * STAGE);
  pdl_wait();

  // ---- x staging: the CTA's K-column of every vector, in fragment order.
  const int kc0 = 2048 * wk;
  if constexpr (kIsNVFP4) {
    // per vector: sigma with max |x| * 2^sigma in [2^14, 2^15) over this K-column
    int* const vmax = reinterpret_cast<int*>(vscale);
    if (threadIdx.x < kBatchMax) vmax[threadIdx.x] = 0;
    __syncthreads();
    for (int idx = threadIdx.x; idx < a.M * 512; idx += blockDim.x) {
      const int v = idx >> 9, c = idx & 511;
      if (4 * c < 256 * ncols) {
        const uint2 r = __ldcg(reinterpret_cast<const uint2*>(a.x + static_cast<int64_t>(v) * a.K + kc0) + c);
        const uint32_t m = max(max(r.x & 0x7FFFu, (r.x >> 16) & 0x7FFFu), max(r.y & 0x7FFFu, (r.y >> 16) & 0x7FFFu));
        if (m) atomicMax(vmax + v, static_cast<int>(m));
      }
    }
    __syncthreads();
    if (threadIdx.x < kBatchMax) {
      const int m = vmax[threadIdx.x];
      const int e8 = (m >> 7) & 0xFF;  // bf16 biased exponent of the largest |x|
      reinterpret_cast<int*>(vscale)[threadIdx.x] = m ? max(-100, min(100, 141 - e8)) : 0;  // sigma
    }
    __syncthreads();
  }
  for (int idx = threadIdx.x; idx < kBatchMax * 512; idx += blockDim.x) {
    const int v = idx >> 9, c = idx & 511;
    const int sb = c >> 6, e = 4 * (c & 63);
    uint2 raw = make_uint2(0u, 0u);
    if (v < a.M && sb < ncols) {
      raw = __ldcg(reinterpret_cast<const uint2*>(a.x + static_cast<int64_t>(v) * a.K + kc0) + c);
      if constexpr (kIsNVFP4) {
        const float f = p2(reinterpret_cast<const int*>(vscale)[v]);
        const __half2 h0 = __floats2half2_rn(bf2f(raw.x) * f, bf2f(raw.x >> 16) * f);
        const __half2 h1 = __floats2half2_rn(bf2f(raw.y) * f, bf2f(raw.y >> 16) * f);
        raw = make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
      }
    }
    int step, tq;
    uint2 val;
    Fmt::chunk_slot(e, step, tq, val, raw);
    const int ln = 4 * v + tq;
    *reinterpret_cast<uint2*>(smem + L.xa + ((sb * 16 + step) * 32 + ln) * 8) = val;
    if constexpr (!kIsNVFP4) {
      // group sums of x (for the minimum term): 8 chunks of 4 make a group of 32
      float s = __half2float(__ushort_as_half(static_cast<unsigned short>(raw.x & 0xFFFFu))) +
                __half2float(__ushort_as_half(static_cast<unsigned short>(raw.x >> 16))) +
                __half2float(__ushort_as_half(static_cast<unsigned short>(raw.y & 0xFFFFu))) +
                __half2float(__ushort_as_half(static_cast<unsigned short>(raw.y >> 16)));
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      s += __shfl_xor_sync(0xffffffffu, s, 4);
      if ((c & 7) == 0) {
        const int grp = e >> 5;  // group of the superblock: the m16n8k8 k index
        const float sc = s * (1.0f / 64.0f);  // keeps the fp16 parts finite for any fp16 x
        const __half hi = __float2half_rn(sc);
        const __half lo = __float2half_rn(sc - __half2float(hi));
        uint16_t* dst = reinterpret_cast<uint16_t*>(smem + L.xs + (sb * 32 + 4 * v + (grp >> 1)) * 8);
        dst[grp & 1] = __half_as_ushort(hi);
        dst[2 + (grp & 1)] = __half_as_ushort(lo);
      }
    }
  }
  __syncthreads();
  float oscale = 1.f;  // output scale of this lane's vector g
  if constexpr (kIsNVFP4) oscale = p2(-reinterpret_cast<const int*>(vscale)[g]);

  // ---- main loop: 8 rows per stage, every superblock of the K-column.
  float* const out = a.Wk == 1 ? a.y + p_lo : a.ws + (static_cast<int64_t>(wk) * a.M) * a.N + p_lo;
  const bool writer = g < a.M;
  uint32_t cs = ring_sa, is = ring_sa + (D - 1) * STAGE;
  const uint32_t xa_lane = xa_sa + lane * 8, xs_lane = xs_sa + lane * 8;
  for (int st = 0; st < nst; ++st) {
    issue(st + D - 1, is);
    cp_async_wait<D - 1>();
    __syncwarp();
    float acc0 = 0.f, acc1 = 0.f;
    if constexpr (!kIsNVFP4) {
      for (int c = 0; c < ncols; ++c) {
        const uint32_t hd0 = lds_u32(cs + (2 * t4) * SLICE + SB * c);
        const uint32_t hd1 = lds_u32(cs + (2 * t4 + 1) * SLICE + SB * c);
        Fmt::superblock(cs + g * SLICE + SB * c, hd0, hd1, t4, xa_lane + c * 16 * 256, xs_lane + c * 256, acc0, acc1);
      }
    } else {
      float dq[4] = {0.f, 0.f, 0.f, 0.f};
      for (int c = 0; c < ncols; ++c)
        BatchNVFP4::superblock(cs + g * SLICE + SB * c, cs + g * SLICE + 8 * SB + SB2 * c, t4, xa_lane + c * 16 * 256, dq);
      acc0 = dq[0] * oscale;
      acc1 = dq[1] * oscale;
    }
    __syncwarp();  // every lane is done with this slot before it is refilled
    is = cs;
    cs = (cs + STAGE == ring_end) ? ring_sa : cs + STAGE;
    const int r0 = st * kBatchRows + 2 * t4;
    if (writer && r0 < nrows) out[static_cast<int64_t>(g) * a.N + r0] = acc0;
    if (writer && r0 + 1 < nrows) out[static_cast<int64_t>(g) * a.N + r0 + 1] = acc1;
  }
  cp_async_wait<0>();

  if (a.Wk > 1) {
    __shared__ int last;
    __syncthreads();
    if (threadIdx.x == 0) {
      int old;
      asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(a.cnt + b) : "memory");
      last = old == a.Wk - 1;
    }
    __syncthreads();
    if (last) {
      for (int i = threadIdx.x; i < ncta * a.M; i += blockDim.x) {
        const int v = i / ncta, r = i - v * ncta;
        float s = 0.f;
        for (int w = 0; w < a.Wk; ++w) s += __ldcg(a.ws + (static_cast<int64_t>(w) * a.M + v) * a.N + r_lo + r);
        a.y[static_cast<int64_t>(v) * a.N + r_lo + r] = s;
      }
      if (threadIdx.x == 0) a.cnt[b] = 0;
    }
  }
}

template <class Fmt>
const void* batch_kernel_table(int D) {
  switch (D) {
    case 2: return reinterpret_cast<const void*>(&batch_kernel<Fmt, 2>);
    default: return reinterpret_cast<const void*>(&batch_kernel<Fmt, 3>);
  }
}

}  // namespace qg
