// Small-batch dequant GEMV: Y[m, n] = sum_k X[m, k] * dequant(W)[n, k] for M = 1..8
// activation vectors, every weight decoded once and used by all of them.
//
// At M = 1 the product is a matrix-vector product and the streaming kernel's exact
// mixed-precision FMAs fit it best ("fp4_gemv" page: no MMA at M = 1); from a few vectors on, the same
// decoded weight meets several activations, which is what the tensor cores' mma.sync
// contraction does without any shared-memory round trip for the weights: they are decoded
// in registers straight into the A fragments of m16n8k16 (16 weight rows as its M), and the
// activation vectors are its N (8 slots, M of them used).
//
//  * Work split: a CTA (16 warps) takes one 1024-wide K-column (4 superblocks) of a row
//    range; warp p takes row group p of the range in tiles of 16 rows, each tile in stages
//    of 2 superblocks, through a private ring of D stages filled with 16-byte cp.async
//    copies (row slots padded so the 16 rows of a stage start in different banks).
//  * Activations: the CTA stages its K-column of all M vectors once, already in B-fragment
//    order (lane (g, t4) reads the pair of fp16 values for vector g at its k slots with one
//    8-byte shared load per k-step).  Unused vector slots hold zeros.
//  * Lane (g, t4) decodes rows g and g + 8 of a stage, 64 elements of each superblock
//    (chunk t4), and receives the sums of those rows for vectors 2 t4 and 2 t4 + 1.
//  * Q4_K: A = q * s_g, an exact integer <= 945 in fp16 (the 6-bit group scale folded in):
//    one LOP3 puts two nibbles into fp16 (1024 + q) / (1024 + 16 q), one fused multiply-add
//    scales and removes the offset.  The group minimum term sum_g m_g X_g goes through an
//    m16n8k8 product (A = m_g, B = the group sums of x split into two fp16 parts), and the
//    superblock scales d, dmin are applied to both sums in fp32 once per superblock.
//  * NVFP4: A = e2m1 * |e4m3 block scale|, exact in fp16; x (bf16) is staged as fp16 times
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

constexpr int kBatchMax = 8;        // activation vectors (the MMA's N)
constexpr int kBatchRows = 16;      // weight rows per stage (the MMA's M)
constexpr int kBatchColSB = 4;      // superblocks per K-column
constexpr int kBatchStageSB = 2;    // superblocks per stage by default (a 16-row tile takes 1 or 2)
constexpr int kBatchThreads = 512;  // 16 warps per CTA

struct BatchArgs {
  const uint8_t* W;   // stream 1: packed blocks / NVFP4 nibbles
  const uint8_t* W2;  // stream 2: NVFP4 scales (null otherwise)
  const uint16_t* x;  // [M, K] fp16 (bf16 for NVFP4)
  float* y;           // [M, N] fp32
  int64_t N;
  int M;
  int K;
  int nsb;            // superblocks per row
  int Wk;             // K-columns = ceil(nsb / 4)
  int rows_q, rows_rem;  // range b has rows_q (+1 if b < rows_rem) rows
  int64_t row_bytes, row_bytes2;
  float* ws;          // Wk > 1: column sums [Wk][M][N]
  int* cnt;           // per-range arrival counts, zero between launches
};

// Shared memory: [rings: warps * D * 16 * slot][x fragments: 4 sb * 16 steps * 32 lanes * 8 B]
// [group sums (Q4_K): 4 sb * 32 lanes * 8 B][per-vector sigma: 8 ints].
struct BatchSmem {
  size_t xa, xs, sc, total;
};
__host__ __device__ inline BatchSmem batch_smem(int warps, int D, int slice) {
  BatchSmem m;
  m.xa = static_cast<size_t>(warps) * D * kBatchRows * slice;
  m.xs = m.xa + kBatchColSB * 16 * 32 * 8;
  m.sc = m.xs + kBatchColSB * 32 * 8;
  m.total = m.sc + kBatchMax * 4 + 16;
  return m;
}

// D += A B: A fragment {a0: row g, k 2t4..2t4+1; a1: row g+8; a2: row g, k 2t4+8..; a3: row
// g+8, k 2t4+8..}, B fragment {b0: k 2t4..2t4+1, column g; b1: k 2t4+8..}, D {row g, columns
// 2t4, 2t4+1; row g+8, columns 2t4, 2t4+1} (fp16 pairs, fp32 accumulators).
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// The k = 8 form: A {a0: row g, k 2t4..2t4+1; a1: row g+8}, B {b0: k 2t4..2t4+1, column g}.
__device__ __forceinline__ void mma1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
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

// (a & mask) | c in one LOP3 (c a register: the compiler would otherwise spend a second
// logic op on a second immediate).
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
  return d;
}

// Two small non-negative integers (< 1024) as the fp16 pair (lo, hi), exactly.
__device__ __forceinline__ uint32_t int2_to_h2(uint32_t lo, uint32_t hi) {
  return hsub2_u((lo | (hi << 16)) | 0x64006400u, 0x64006400u);
}

// ----------------------------------------------------------------------------- Q4_K
// Decoders.  Each has kSB / kSB2 (bytes of a superblock in stream 1 / 2); kMinTerm (a group
// minimum term, taken through the staged group sums of x); kFolded (every scale folded into A,
// so the accumulators run over a whole tile; otherwise the superblock scales d, dmin are
// applied to each superblock's sums); kBF16 (x is bf16, staged as scaled fp16); chunk_slot
// (where an aligned chunk of 4 x values goes in the fragment buffer); and superblock (one
// superblock c of a stage, rows g and g + 8 from the row slots at rg / r8).
struct BatchQ4K {
  static constexpr int kSB = 144, kSB2 = 0;
  static constexpr int kStageSB = kBatchStageSB, kPad = 16;  // superblocks per stage, slot padding
  static constexpr bool kMinTerm = true, kFolded = false, kBF16 = false, kWindow = false;

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

  // Scales and mins of groups 2 t4 and 2 t4 + 1 from a block header (12 packed bytes in
  // hdr.y..w; "Kernel code" mask arithmetic) as fp16 pairs (lo group, hi group).  Groups 0..3
  // take the low 6 bits of bytes 0..3 / 4..7; groups 4..7 a nibble of bytes 8..11 below the
  // top two bits of bytes 0..3 / 4..7.  Selects, so the warp does not diverge.
  __device__ __forceinline__ static void group_scales(const uint4& hdr, int t4, uint32_t& S, uint32_t& Mn) {
    const uint32_t sh16 = 16u * (t4 & 1);  // byte q = 2 (t4 & 1) in bits 0..7, byte q + 1 in 8..15
    const uint32_t B0 = hdr.y >> sh16, B1 = hdr.z >> sh16, B2 = hdr.w >> sh16;
    const uint32_t c0 = B0 & 0xFFu, c1 = (B0 >> 8) & 0xFFu;  // S0[q], S0[q + 1]
    const uint32_t e0 = B1 & 0xFFu, e1 = (B1 >> 8) & 0xFFu;  // S1[q], S1[q + 1]
    const uint32_t f0 = B2 & 0xFFu, f1 = (B2 >> 8) & 0xFFu;  // S2[q], S2[q + 1]
    const bool split = t4 >= 2;
    const uint32_t sl = split ? ((f0 & 15u) | ((c0 >> 6) << 4)) : (c0 & 63u);
    const uint32_t sh = split ? ((f1 & 15u) | ((c1 >> 6) << 4)) : (c1 & 63u);
    const uint32_t ml = split ? ((f0 >> 4) | ((e0 >> 6) << 4)) : (e0 & 63u);
    const uint32_t mh = split ? ((f1 >> 4) | ((e1 >> 6) << 4)) : (e1 & 63u);
    S = int2_to_h2(sl, sh);
    Mn = int2_to_h2(ml, mh);
  }

  // Lane (g, t4): adds the superblock's contribution to the lane's four sums y.
  __device__ __forceinline__ static void superblock(uint32_t rg, uint32_t r8, int c, int t4, uint32_t xa, uint32_t xs,
                                                    uint32_t magic, float (&y)[4]) {
    const uint32_t bg = rg + kSB * c, b8 = r8 + kSB * c;
    const uint4 hg = lds_v4(bg), h8 = lds_v4(b8);
    const uint4 g0 = lds_v4(bg + 16 + 32 * t4), g1 = lds_v4(bg + 32 + 32 * t4);
    const uint4 e0 = lds_v4(b8 + 16 + 32 * t4), e1 = lds_v4(b8 + 32 + 32 * t4);
    uint32_t Sg, Mg, S8, M8;
    group_scales(hg, t4, Sg, Mg);
    group_scales(h8, t4, S8, M8);
    // low-nibble pairs: (1024 + q) s - 1024 s; high-nibble pairs: (1024 + 16 q) s/16 - 64 s
    const uint32_t SLg = __byte_perm(Sg, Sg, 0x1010), SL8 = __byte_perm(S8, S8, 0x1010);
    const uint32_t SHg = hmul2_u(__byte_perm(Sg, Sg, 0x3232), 0x2C002C00u);
    const uint32_t SH8 = hmul2_u(__byte_perm(S8, S8, 0x3232), 0x2C002C00u);
    const uint32_t CLg = hmul2_u(SLg, 0xE400E400u), CL8 = hmul2_u(SL8, 0xE400E400u);
    const uint32_t CHg = hmul2_u(SHg, 0xE400E400u), CH8 = hmul2_u(SH8, 0xE400E400u);
    const uint32_t wg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const uint32_t w8[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
    float dq[2][4] = {};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t a = wg[i], a8 = wg[i] >> 8, b = w8[i], b8s = w8[i] >> 8;
      const uint2 xl = lds_v2(xa + (2 * i) * 256), xh = lds_v2(xa + (2 * i + 1) * 256);
      mma16816(dq[0], hfma2_u(and_or<0x000F000Fu>(a, magic), SLg, CLg),
               hfma2_u(and_or<0x000F000Fu>(b, magic), SL8, CL8),
               hfma2_u(and_or<0x000F000Fu>(a8, magic), SLg, CLg),
               hfma2_u(and_or<0x000F000Fu>(b8s, magic), SL8, CL8), xl.x, xl.y);
      mma16816(dq[1], hfma2_u(and_or<0x00F000F0u>(a, magic), SHg, CHg),
               hfma2_u(and_or<0x00F000F0u>(b, magic), SH8, CH8),
               hfma2_u(and_or<0x00F000F0u>(a8, magic), SHg, CHg),
               hfma2_u(and_or<0x00F000F0u>(b8s, magic), SH8, CH8), xh.x, xh.y);
    }
    float dm[4] = {};
    const uint2 X = lds_v2(xs);  // group sums / 64: (hi parts), (lo parts)
    mma1688(dm, Mg, M8, X.x);
    mma1688(dm, Mg, M8, X.y);
    const float dg = h2f(hg.x), mg = h2f(hg.x >> 16) * 64.f, d8 = h2f(h8.x), m8 = h2f(h8.x >> 16) * 64.f;
    y[0] += fmaf(dg, dq[0][0] + dq[1][0], -mg * dm[0]);
    y[1] += fmaf(dg, dq[0][1] + dq[1][1], -mg * dm[1]);
    y[2] += fmaf(d8, dq[0][2] + dq[1][2], -m8 * dm[2]);
    y[3] += fmaf(d8, dq[0][3] + dq[1][3], -m8 * dm[3]);
  }
};

// ----------------------------------------------------------------------------- NVFP4
struct BatchNVFP4 {
  static constexpr int kSB = 128, kSB2 = 16;
  static constexpr int kStageSB = kBatchStageSB, kPad = 16;
  static constexpr bool kMinTerm = false, kFolded = true, kBF16 = true, kWindow = false;

  // Chunk t4 of a superblock is nibble bytes [32 t4, 32 t4 + 32) = elements 64 t4 + [0, 64);
  // word i (elements 64 t4 + 8 i + [0, 8)) feeds steps 2 i (elements +0..3) and 2 i + 1
  // (+4..7), each as the pairs (e, e + 1) and (e + 2, e + 3) of its cvt.e2m1x2 results.
  __device__ __forceinline__ static void chunk_slot(int e, int& step, int& t4, uint2& v, uint2 raw) {
    t4 = e >> 6;
    step = (e & 63) >> 2;
    v = raw;
  }

  // Nibbles of superblock c at 128 c of a row slot, its scales at 2 * 128 + 16 c.
  __device__ __forceinline__ static void superblock(uint32_t rg, uint32_t r8, int c, int t4, uint32_t xa, uint32_t,
                                                    uint32_t, float (&dq)[2][4]) {
    const uint32_t ng = rg + kSB * c, n8 = r8 + kSB * c;
    const uint32_t sg = rg + kStageSB * kSB + kSB2 * c, s8 = r8 + kStageSB * kSB + kSB2 * c;
    const uint4 g0 = lds_v4(ng + 32 * t4), g1 = lds_v4(ng + 32 * t4 + 16);
    const uint4 e0 = lds_v4(n8 + 32 * t4), e1 = lds_v4(n8 + 32 * t4 + 16);
    const uint32_t sG = lds_u32(sg + 4 * t4) & 0x7F7F7F7Fu;  // |scale| of blocks 4 t4 .. 4 t4 + 3
    const uint32_t s8v = lds_u32(s8 + 4 * t4) & 0x7F7F7F7Fu;
    const uint32_t wg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const uint32_t w8[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t tg = DecNVFP4::e4m3x2((sG >> (8 * b)) & 0xFFu), t8 = DecNVFP4::e4m3x2((s8v >> (8 * b)) & 0xFFu);
      const uint32_t vg = __byte_perm(tg, tg, 0x1010), v8 = __byte_perm(t8, t8, 0x1010);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int i = 2 * b + u;
        uint32_t hg[4], h8[4];
        DecNVFP4::e2m1x8(wg[i], hg);
        DecNVFP4::e2m1x8(w8[i], h8);
        const uint2 xl = lds_v2(xa + (2 * i) * 256), xh = lds_v2(xa + (2 * i + 1) * 256);
        mma16816(dq[0], hmul2_u(hg[0], vg), hmul2_u(h8[0], v8), hmul2_u(hg[1], vg), hmul2_u(h8[1], v8), xl.x, xl.y);
        mma16816(dq[1], hmul2_u(hg[2], vg), hmul2_u(h8[2], v8), hmul2_u(hg[3], vg), hmul2_u(h8[3], v8), xh.x, xh.y);
      }
    }
  }
};

// ----------------------------------------------------------------------------- Q5_K
// The Q4_K layout with a fifth bit per code: qh[32] at 16, quants at 48.  Codes (q5 <= 31)
// times the 6-bit group scale stay exact fp16 integers (<= 1953).
struct BatchQ5K {
  static constexpr int kSB = 176, kSB2 = 0;
  static constexpr int kStageSB = kBatchStageSB, kPad = 16;
  static constexpr bool kMinTerm = true, kFolded = false, kBF16 = false, kWindow = false;

  __device__ __forceinline__ static void chunk_slot(int e, int& step, int& t4, uint2& v, uint2 raw) {
    BatchQ4K::chunk_slot(e, step, t4, v, raw);
  }

  __device__ __forceinline__ static void superblock(uint32_t rg, uint32_t r8, int c, int t4, uint32_t xa, uint32_t xs,
                                                    uint32_t magic, float (&y)[4]) {
    const uint32_t bg = rg + kSB * c, b8 = r8 + kSB * c;
    const uint4 hg = lds_v4(bg), h8 = lds_v4(b8);
    const uint4 g0 = lds_v4(bg + 48 + 32 * t4), g1 = lds_v4(bg + 64 + 32 * t4);
    const uint4 e0 = lds_v4(b8 + 48 + 32 * t4), e1 = lds_v4(b8 + 64 + 32 * t4);
    const uint4 qg0 = lds_v4(bg + 16), qg1 = lds_v4(bg + 32);  // qh[0..32) of row g
    const uint4 q80 = lds_v4(b8 + 16), q81 = lds_v4(b8 + 32);
    uint32_t Sg, Mg, S8, M8;
    BatchQ4K::group_scales(hg, t4, Sg, Mg);
    BatchQ4K::group_scales(h8, t4, S8, M8);
    // both planes: (1024 + q5) s - 1024 s
    const uint32_t SLg = __byte_perm(Sg, Sg, 0x1010), SL8 = __byte_perm(S8, S8, 0x1010);
    const uint32_t SHg = __byte_perm(Sg, Sg, 0x3232), SH8 = __byte_perm(S8, S8, 0x3232);
    const uint32_t CLg = hmul2_u(SLg, 0xE400E400u), CL8 = hmul2_u(SL8, 0xE400E400u);
    const uint32_t CHg = hmul2_u(SHg, 0xE400E400u), CH8 = hmul2_u(SH8, 0xE400E400u);
    const uint32_t wg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const uint32_t w8[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
    const uint32_t hqg[8] = {qg0.x, qg0.y, qg0.z, qg0.w, qg1.x, qg1.y, qg1.z, qg1.w};
    const uint32_t hq8[8] = {q80.x, q80.y, q80.z, q80.w, q81.x, q81.y, q81.z, q81.w};
    const uint32_t sh = 2u * t4;  // qh bit 2 t4 (low nibbles) and 2 t4 + 1 (high nibbles)
    float dq[2][4] = {};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // 5-bit codes of the word's four bytes, low- and high-nibble planes
      const uint32_t hg_ = hqg[i] >> sh, h8_ = hq8[i] >> sh;
      const uint32_t lg = and_or<0x0F0F0F0Fu>(wg[i], (hg_ << 4) & 0x10101010u);
      const uint32_t ug = and_or<0x0F0F0F0Fu>(wg[i] >> 4, (hg_ << 3) & 0x10101010u);
      const uint32_t l8 = and_or<0x0F0F0F0Fu>(w8[i], (h8_ << 4) & 0x10101010u);
      const uint32_t u8 = and_or<0x0F0F0F0Fu>(w8[i] >> 4, (h8_ << 3) & 0x10101010u);
      const uint2 xl = lds_v2(xa + (2 * i) * 256), xh = lds_v2(xa + (2 * i + 1) * 256);
      mma16816(dq[0], hfma2_u(and_or<0x001F001Fu>(lg, magic), SLg, CLg),
               hfma2_u(and_or<0x001F001Fu>(l8, magic), SL8, CL8),
               hfma2_u(and_or<0x001F001Fu>(lg >> 8, magic), SLg, CLg),
               hfma2_u(and_or<0x001F001Fu>(l8 >> 8, magic), SL8, CL8), xl.x, xl.y);
      mma16816(dq[1], hfma2_u(and_or<0x001F001Fu>(ug, magic), SHg, CHg),
               hfma2_u(and_or<0x001F001Fu>(u8, magic), SH8, CH8),
               hfma2_u(and_or<0x001F001Fu>(ug >> 8, magic), SHg, CHg),
               hfma2_u(and_or<0x001F001Fu>(u8 >> 8, magic), SH8, CH8), xh.x, xh.y);
    }
    float dm[4] = {};
    const uint2 X = lds_v2(xs);
    mma1688(dm, Mg, M8, X.x);
    mma1688(dm, Mg, M8, X.y);
    const float dg = h2f(hg.x), mg = h2f(hg.x >> 16) * 64.f, d8 = h2f(h8.x), m8 = h2f(h8.x >> 16) * 64.f;
    y[0] += fmaf(dg, dq[0][0] + dq[1][0], -mg * dm[0]);
    y[1] += fmaf(dg, dq[0][1] + dq[1][1], -mg * dm[1]);
    y[2] += fmaf(d8, dq[0][2] + dq[1][2], -m8 * dm[2]);
    y[3] += fmaf(d8, dq[0][3] + dq[1][3], -m8 * dm[3]);
  }
};

// ----------------------------------------------------------------------------- Q8_0
// A superblock is 8 blocks of 34 bytes (d, then 32 int8 codes).  Lane t4 takes blocks 2 t4 and
// 2 t4 + 1 (bytes [68 t4, 68 t4 + 68), read as 17 aligned words), one word of 4 codes per
// k-step.  The block scale changes between the lanes of a k-step, so it cannot wait for the
// accumulator: A = fp16(d' q), rounded once per weight (relative error at most 2^-11, a
// quarter of the GEMV bound), with d' = d 2^sigma, sigma per row and superblock chosen from
// the row's largest block scale so that every |d' q| < 2^15.  That keeps the operands out of
// the fp16 subnormals (where rounding would be an absolute 2^-25, not a relative error) for
// every block within 2^21 of the row's largest one; the superblock's sums are multiplied by
// 2^-sigma in fp32.
struct BatchQ80 {
  static constexpr int kSB = 272, kSB2 = 0;
  // one superblock per stage (two would not fit 16 warps x 2 stages), slots padded by 32 so
  // the word loads of the 8 rows g fall in different banks
  static constexpr int kStageSB = 1, kPad = 32;
  static constexpr bool kMinTerm = false, kFolded = false, kBF16 = false, kWindow = false;

  // elements 64 t4 + 4 s + (0..3): pairs (x0, x2) and (x1, x3), as bytes (b0, b2), (b1, b3)
  __device__ __forceinline__ static void chunk_slot(int e, int& step, int& t4, uint2& v, uint2 raw) {
    t4 = e >> 6;
    step = (e & 63) >> 2;
    v.x = __byte_perm(raw.x, raw.y, 0x5410);
    v.y = __byte_perm(raw.x, raw.y, 0x7632);
  }

  // The lane's two blocks of one row: 17 aligned words from `base` (68 t4 into the superblock).
  // Block 2 t4: d in bytes 0..1, codes in bytes 2..33 (unaligned: one PRMT per word); block
  // 2 t4 + 1: d in bytes 34..35, codes in bytes 36..67 (aligned).
  __device__ __forceinline__ static void lane_blocks(uint32_t base, uint32_t (&q)[16], uint32_t& dA, uint32_t& dB) {
    uint32_t w[17];
#pragma unroll
    for (int k = 0; k < 17; ++k) w[k] = lds_u32(base + 4 * k);
    dA = w[0] & 0xFFFFu;
    dB = w[8] >> 16;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      q[k] = __byte_perm(w[k], w[k + 1], 0x5432);
      q[8 + k] = w[9 + k];
    }
  }

  // The row's scale 2^sigma from the largest |d| of its 8 blocks (the lane's two, then the
  // four lanes t4 of the row), and the lane's two scaled block scales as fp16 pairs.
  __device__ __forceinline__ static float row_scale(uint32_t dA, uint32_t dB, uint32_t& pA, uint32_t& pB) {
    uint32_t m = max(dA & 0x7FFFu, dB & 0x7FFFu);
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
    // |d| < 2^(E + 1) for the largest: 2^sigma = 2^(7 - E) puts it in [2^7, 2^8), |d' q| < 2^15
    const int E = m ? static_cast<int>((__float_as_uint(h2f(m)) >> 23) & 0xFFu) - 127 : 0;
    const float sc = p2(7 - E);
    const uint32_t a = __half_as_ushort(__float2half_rn(h2f(dA) * sc));
    const uint32_t b = __half_as_ushort(__float2half_rn(h2f(dB) * sc));
    pA = a | (a << 16);
    pB = b | (b << 16);
    return p2(E - 7);
  }

  __device__ __forceinline__ static void superblock(uint32_t rg, uint32_t r8, int c, int t4, uint32_t xa, uint32_t,
                                                    uint32_t magic, float (&y)[4]) {
    uint32_t qg[16], q8[16], dAg, dBg, dA8, dB8;
    lane_blocks(rg + kSB * c + 68 * t4, qg, dAg, dBg);
    lane_blocks(r8 + kSB * c + 68 * t4, q8, dA8, dB8);
    uint32_t pAg, pBg, pA8, pB8;
    const float ig = row_scale(dAg, dBg, pAg, pBg), i8 = row_scale(dA8, dB8, pA8, pB8);
    const uint32_t off = 0x64806480u;  // fp16 (1152, 1152) = 1024 + 128
    float dq[2][4] = {};
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      const uint32_t dg = s < 8 ? pAg : pBg, d8 = s < 8 ? pA8 : pB8;
      const uint32_t ug = qg[s] ^ 0x80808080u, u8 = q8[s] ^ 0x80808080u;  // q + 128 per byte
      const uint2 xs_ = lds_v2(xa + s * 256);
      mma16816(dq[s & 1], hmul2_u(hsub2_u(and_or<0x00FF00FFu>(ug, magic), off), dg),
               hmul2_u(hsub2_u(and_or<0x00FF00FFu>(u8, magic), off), d8),
               hmul2_u(hsub2_u(and_or<0x00FF00FFu>(ug >> 8, magic), off), dg),
               hmul2_u(hsub2_u(and_or<0x00FF00FFu>(u8 >> 8, magic), off), d8), xs_.x, xs_.y);
    }
    y[0] = fmaf(dq[0][0] + dq[1][0], ig, y[0]);
    y[1] = fmaf(dq[0][1] + dq[1][1], ig, y[1]);
    y[2] = fmaf(dq[0][2] + dq[1][2], i8, y[2]);
    y[3] = fmaf(dq[0][3] + dq[1][3], i8, y[3]);
  }
};

// N words at a 2-byte aligned shared address: N + 1 aligned loads, each word pieced together
// from two of them (a no-op permutation when the address is 4-byte aligned).
template <int N>
__device__ __forceinline__ void lds_run(uint32_t addr, uint32_t (&w)[N]) {
  const uint32_t b = addr & ~3u, sel = 0x3210u + (addr & 2u) * 0x1111u;
  uint32_t t[N + 1];
#pragma unroll
  for (int k = 0; k <= N; ++k) t[k] = lds_u32(b + 4 * k);
#pragma unroll
  for (int k = 0; k < N; ++k) w[k] = __byte_perm(t[k], t[k + 1], sel);
}

// ----------------------------------------------------------------------------- TQ1_0
// Windowed formats (kWindow): their blocks (54 / 210 bytes) do not start on 16-byte
// boundaries, so a stage copies the aligned 16-byte chunks that cover its superblocks (the
// stage's data starts kMaxOff or fewer bytes into the slot) and reads words with lds_run.
//
// TQ1_0 ("metal: TQ1_0 kernel performance", section 2, the il walk): byte m of qs[0..32)
// holds digit n of elements 32 n + m, byte 32 + m of qs holds digit n of elements 160 + 16 n +
// m, byte m of qh holds digit n < 4 of elements 240 + 4 n + m.  Lane t4 takes qs bytes [8 t4, 8 t4 + 8) (steps 2 n + w for
// its words w = 0, 1), qs bytes [32 + 4 t4, 36 + 4 t4) (steps 10 + n) and digit n = t4 of the
// qh word (step 15).  The digits come out of the floor pair as in the stream decoder: with the
// even and the odd bytes in 16-bit lanes, q <- 3 q splits into the digit (bits 8..9) and the
// rest (bits 0..7); the digit, put into the fp16 mantissa of 1024, is scaled to t - 1 with one
// exact half FMA: (1024 + 256 t) / 256 - 5.  A superblock's sums get its d in fp32.
struct BatchTQ10 {
  static constexpr int kSB = 54, kSB2 = 0;
  static constexpr int kStageSB = 4, kPad = 16, kMaxOff = 8;  // stage starts at 216 wk: offset 0 or 8
  static constexpr bool kMinTerm = false, kFolded = false, kBF16 = false, kWindow = true;

  __device__ __forceinline__ static void chunk_slot(int e, int& step, int& t4, uint2& v, uint2 raw) {
    if (e < 160) {
      const int m = e & 31;
      t4 = m >> 3;
      step = 2 * (e >> 5) + ((m >> 2) & 1);
    } else if (e < 240) {
      t4 = ((e - 160) & 15) >> 2;
      step = 10 + ((e - 160) >> 4);
    } else {
      t4 = (e - 240) >> 2;
      step = 15;
    }
    v.x = __byte_perm(raw.x, raw.y, 0x5410);  // (x0, x2)
    v.y = __byte_perm(raw.x, raw.y, 0x7632);  // (x1, x3)
  }

  // The lane's words of one row: qs region 1 (2 words), region 2 (1 word), qh and d.
  __device__ __forceinline__ static void row_words(uint32_t blk, int t4, uint32_t (&w1)[2], uint32_t& w2, uint32_t& wh,
                                                   float& d) {
    lds_run<2>(blk + 8 * t4, w1);
    uint32_t r2[1], th[2];
    lds_run<1>(blk + 32 + 4 * t4, r2);
    lds_run<2>(blk + 48, th);
    w2 = r2[0];
    wh = th[0];
    d = h2f(th[1]);
  }

  // Next digit of the (even or odd byte) lanes q: returns t - 1 as an fp16 pair.
  __device__ __forceinline__ static uint32_t digit(uint32_t& q, uint32_t magic) {
    const uint32_t r = q * 3u;
    q = r & 0x00FF00FFu;
    return hfma2_u(and_or<0x03000300u>(r, magic), 0x1C001C00u, 0xC500C500u);  // x 2^-8, - 5
  }

  __device__ __forceinline__ static void superblock(uint32_t rg, uint32_t r8, int c, int t4, uint32_t xa, uint32_t,
                                                    uint32_t magic, float (&y)[4]) {
    uint32_t ag[2], a8[2], bg, b8, hg, h8;
    float dg, d8;
    row_words(rg + kSB * c, t4, ag, bg, hg, dg);
    row_words(r8 + kSB * c, t4, a8, b8, h8, d8);
    float dq[2][4] = {};
    auto steps = [&](uint32_t wg, uint32_t w8, int s0, int ds) {
      uint32_t eg = wg & 0x00FF00FFu, og = (wg >> 8) & 0x00FF00FFu;
      uint32_t e8 = w8 & 0x00FF00FFu, o8 = (w8 >> 8) & 0x00FF00FFu;
#pragma unroll
      for (int n = 0; n < 5; ++n) {
        const int s = s0 + ds * n;
        const uint2 xv = lds_v2(xa + s * 256);
        const uint32_t A0 = digit(eg, magic), A1 = digit(e8, magic), A2 = digit(og, magic), A3 = digit(o8, magic);
        mma16816(dq[n & 1], A0, A1, A2, A3, xv.x, xv.y);
      }
    };
    steps(ag[0], a8[0], 0, 2);
    steps(ag[1], a8[1], 1, 2);
    steps(bg, b8, 10, 1);
    {  // qh: digit t4 of each byte, q = b 3^t4 mod 256 first
      const uint32_t p3 = (t4 & 2 ? 9u : 1u) * (t4 & 1 ? 3u : 1u);
      uint32_t eg = ((hg & 0x00FF00FFu) * p3) & 0x00FF00FFu, og = (((hg >> 8) & 0x00FF00FFu) * p3) & 0x00FF00FFu;
      uint32_t e8 = ((h8 & 0x00FF00FFu) * p3) & 0x00FF00FFu, o8 = (((h8 >> 8) & 0x00FF00FFu) * p3) & 0x00FF00FFu;
      const uint2 xv = lds_v2(xa + 15 * 256);
      const uint32_t A0 = digit(eg, magic), A1 = digit(e8, magic), A2 = digit(og, magic), A3 = digit(o8, magic);
      mma16816(dq[1], A0, A1, A2, A3, xv.x, xv.y);
    }
    y[0] += dg * (dq[0][0] + dq[1][0]);
    y[1] += dg * (dq[0][1] + dq[1][1]);
    y[2] += d8 * (dq[0][2] + dq[1][2]);
    y[3] += d8 * (dq[0][3] + dq[1][3]);
  }
};

// ----------------------------------------------------------------------------- Q6_K
// Element i = 128 H + 32 r + l (half H, quarter r, l < 32): low four bits in ql[64 H + 32 (r & 1)
// + l] (low nibble for r < 2), top two bits (qh[32 H + l] >> 2 r) & 3, scale sc[8 H + 2 r +
// l / 16].  Lane t4 takes l in [8 t4, 8 t4 + 8): step 8 H + 2 r + u reads word u of that range,
// whose four elements share the scale sc[8 H + 2 r + t4 / 2].  A = (q6 - 32) sc in fp16: exact
// while |(q6 - 32) sc| <= 2048 (scales up to 64 in magnitude), else rounded once, a relative
// error of at most 2^-11 per weight.  One superblock per stage (two would not fit).
struct BatchQ6K {
  static constexpr int kSB = 210, kSB2 = 0;
  static constexpr int kStageSB = 1, kPad = 16, kMaxOff = 14;  // superblock j starts at 2 j mod 16
  static constexpr bool kMinTerm = false, kFolded = false, kBF16 = false, kWindow = true;

  __device__ __forceinline__ static void chunk_slot(int e, int& step, int& t4, uint2& v, uint2 raw) {
    const int l = e & 31;
    t4 = l >> 3;
    step = 8 * (e >> 7) + 2 * ((e >> 5) & 3) + ((l >> 2) & 1);
    v.x = __byte_perm(raw.x, raw.y, 0x5410);
    v.y = __byte_perm(raw.x, raw.y, 0x7632);
  }

  struct Row {
    uint32_t ql[2][2][2];  // [H][r & 1][u]
    uint32_t qh[2][2];     // [H][u]
    uint32_t sc[4];        // sc[0..16)
    float d;
  };
  __device__ __forceinline__ static void row_words(uint32_t blk, int t4, Row& R) {
#pragma unroll
    for (int H = 0; H < 2; ++H) {
#pragma unroll
      for (int j = 0; j < 2; ++j) lds_run<2>(blk + 64 * H + 32 * j + 8 * t4, R.ql[H][j]);
      lds_run<2>(blk + 128 + 32 * H + 8 * t4, R.qh[H]);
    }
    uint32_t t[5];
    lds_run<5>(blk + 192, t);
#pragma unroll
    for (int k = 0; k < 4; ++k) R.sc[k] = t[k];
    R.d = h2f(t[4]);
  }

  // fp16 pair (s, s) of int8 byte k of word w (k a run-time index 0..3)
  __device__ __forceinline__ static uint32_t scale2(uint32_t w, uint32_t sel) {
    return hsub2_u((__byte_perm(w, 0u, sel) ^ 0x00800080u) | 0x64006400u, 0x64806480u);  // (1152 + s) - 1152
  }

  // fp16 (1024 + q6) pairs of the even (e) and odd (o) bytes of word u, quarter r
  template <int R>
  __device__ __forceinline__ static void codes(uint32_t ql, uint32_t qh, uint32_t magic, uint32_t& e, uint32_t& o) {
    constexpr int sl = 4 * (R >> 1);
    const uint32_t he = R < 3 ? (qh << (4 - 2 * R)) : (qh >> 2);  // bits 2R..2R+1 of bytes 0, 2 to 4..5
    const uint32_t ho = qh >> (4 + 2 * R);                          // of bytes 1, 3
    e = and_or<0x000F000Fu>(ql >> sl, and_or<0x00300030u>(he, magic));
    o = and_or<0x000F000Fu>(ql >> (8 + sl), and_or<0x00300030u>(ho, magic));
  }

  __device__ __forceinline__ static void superblock(uint32_t rg, uint32_t r8, int c, int t4, uint32_t xa, uint32_t,
                                                    uint32_t magic, float (&y)[4]) {
    Row G, E;
    row_words(rg + kSB * c, t4, G);
    row_words(r8 + kSB * c, t4, E);
    const uint32_t hb = static_cast<uint32_t>(t4 >> 1);
    const uint32_t sel0 = 0x4040u | hb | (hb << 8), sel1 = sel0 + 0x0202u;  // bytes hb / hb + 2, in both lanes
    const uint32_t off = 0x64206420u;  // fp16 (1056, 1056) = 1024 + 32
    float dq[2][4] = {};
#pragma unroll
    for (int H = 0; H < 2; ++H) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t sw = (r & 1) ? sel1 : sel0;
        const uint32_t sg = scale2(G.sc[2 * H + (r >> 1)], sw), s8 = scale2(E.sc[2 * H + (r >> 1)], sw);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          uint32_t eg, og, e8, o8;
          switch (r) {
            case 0: codes<0>(G.ql[H][0][u], G.qh[H][u], magic, eg, og), codes<0>(E.ql[H][0][u], E.qh[H][u], magic, e8, o8); break;
            case 1: codes<1>(G.ql[H][1][u], G.qh[H][u], magic, eg, og), codes<1>(E.ql[H][1][u], E.qh[H][u], magic, e8, o8); break;
            case 2: codes<2>(G.ql[H][0][u], G.qh[H][u], magic, eg, og), codes<2>(E.ql[H][0][u], E.qh[H][u], magic, e8, o8); break;
            default: codes<3>(G.ql[H][1][u], G.qh[H][u], magic, eg, og), codes<3>(E.ql[H][1][u], E.qh[H][u], magic, e8, o8); break;
          }
          const int s = 8 * H + 2 * r + u;
          const uint2 xv = lds_v2(xa + s * 256);
          mma16816(dq[u], hmul2_u(hsub2_u(eg, off), sg), hmul2_u(hsub2_u(e8, off), s8), hmul2_u(hsub2_u(og, off), sg),
                   hmul2_u(hsub2_u(o8, off), s8), xv.x, xv.y);
        }
      }
    }
    y[0] += G.d * (dq[0][0] + dq[1][0]);
    y[1] += G.d * (dq[0][1] + dq[1][1]);
    y[2] += E.d * (dq[0][2] + dq[1][2]);
    y[3] += E.d * (dq[0][3] + dq[1][3]);
  }
};

// Bytes of one row slot in a ring stage: the row's superblocks of the stage (stream 1, then
// stream 2; for windowed formats the covering aligned chunks) plus padding, so that the 16
// rows of a stage start in different shared-memory banks.
template <class Fmt>
__host__ __device__ constexpr int batch_chunks() {
  if constexpr (Fmt::kWindow)
    return (Fmt::kMaxOff + Fmt::kStageSB * Fmt::kSB + 15) / 16;
  else
    return Fmt::kStageSB * (Fmt::kSB + Fmt::kSB2) / 16;
}
template <class Fmt>
__host__ __device__ constexpr int batch_slice() {
  return 16 * batch_chunks<Fmt>() + Fmt::kPad;
}

template <class Fmt, int D>
__global__ void __launch_bounds__(kBatchThreads, 1) batch_kernel(const __grid_constant__ BatchArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int SB = Fmt::kSB, SB2 = Fmt::kSB2, SLICE = batch_slice<Fmt>();
  constexpr int STAGE = kBatchRows * SLICE;
  constexpr bool kTwo = SB2 > 0;  // a second stream (NVFP4 scales)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  const unsigned uWk = static_cast<unsigned>(a.Wk);
  const int wk = static_cast<int>(blockIdx.x % uWk), b = static_cast<int>(blockIdx.x / uWk);
  const int64_t r_lo = static_cast<int64_t>(b) * a.rows_q + min(b, a.rows_rem);
  const int ncta = a.rows_q + (b < a.rows_rem ? 1 : 0);
  const int pq = ncta / nwarps, prem = ncta % nwarps;
  const int64_t p_lo = r_lo + warp * pq + min(warp, prem);
  const int nrows = pq + (warp < prem ? 1 : 0);
  const int ncols = min(kBatchColSB, a.nsb - kBatchColSB * wk);  // superblocks in this K-column
  const BatchSmem L = batch_smem(nwarps, D, SLICE);
  const uint32_t ring_sa = smem_u32(smem) + static_cast<uint32_t>(warp) * D * STAGE, ring_end = ring_sa + D * STAGE;
  const uint32_t xa_sa = smem_u32(smem + L.xa), xs_sa = smem_u32(smem + L.xs);
  float* const vscale = reinterpret_cast<float*>(smem + L.sc);

  pdl_launch_dependents();

  // Copies.  A stage is 16 rows x CPR 16-byte chunks (2 superblocks of stream 1, then of
  // stream 2); lane l copies chunks l + 32 j, whose row, source offset (from the stage's row
  // block) and slot offset are fixed per lane.
  constexpr int SSB = Fmt::kStageSB;
  constexpr int CPR = batch_chunks<Fmt>();
  constexpr int NCH = kBatchRows * CPR;  // chunks per stage
  constexpr int JN = (NCH + 31) / 32;
  const int rb1 = static_cast<int>(a.row_bytes), rb2 = static_cast<int>(a.row_bytes2);
  // csb: windowed formats: the chunk's first byte in the window; otherwise its superblock
  uint32_t coff[JN], doff[JN], crow[JN], csb[JN], c2[JN];
#pragma unroll
  for (int j = 0; j < JN; ++j) {
    const int q = lane + 32 * j, row = q / CPR, off = q % CPR;
    const bool two = kTwo && off >= SSB * SB / 16;
    const int o2 = off - SSB * SB / 16;
    coff[j] = two ? row * rb2 + o2 * 16 : row * rb1 + off * 16;
    if constexpr (Fmt::kWindow)
      csb[j] = q < NCH ? off * 16 : 0x7fffffff;  // chunks past the stage: never copied
    else
      csb[j] = q < NCH ? (two ? o2 : (off * 16) / SB) : SSB;
    crow[j] = row;
    c2[j] = two;
    doff[j] = row * SLICE + off * 16;
  }
  const int ntiles = (nrows + kBatchRows - 1) / kBatchRows;
  const int spt = (ncols + SSB - 1) / SSB;  // stages per tile
  const int nst = ntiles * spt;
  auto issue = [&](int st, uint32_t slot_sa) {
    if (st < nst) {
      const int tile = st / spt, h = st - tile * spt;
      const int trows = min(kBatchRows, nrows - tile * kBatchRows);
      const int64_t r0 = p_lo + tile * kBatchRows;
      const int sb0 = kBatchColSB * wk + SSB * h;  // first superblock of the stage in the row
      const int nsb_left = ncols - SSB * h;
      if constexpr (Fmt::kWindow) {
        // the stage's bytes start o bytes into their 16-byte chunk (rows are 16-byte multiples)
        const int o = (sb0 * SB) & 15;
        const uint8_t* base1 = a.W + r0 * a.row_bytes + static_cast<int64_t>(sb0) * SB - o;
        const int need = o + min(SSB, nsb_left) * SB;
#pragma unroll
        for (int j = 0; j < JN; ++j) {
          const uint32_t ok = (static_cast<int>(crow[j]) < trows) & (static_cast<int>(csb[j]) < need);
          cp_async16_if<0, 0>(slot_sa + doff[j], base1 + coff[j], ok);
        }
      } else {
        const uint8_t* base1 = a.W + r0 * a.row_bytes + static_cast<int64_t>(sb0) * SB;
        const uint8_t* base2 = kTwo ? a.W2 + r0 * a.row_bytes2 + static_cast<int64_t>(sb0) * SB2 : base1;
#pragma unroll
        for (int j = 0; j < JN; ++j) {
          const uint32_t ok = (static_cast<int>(crow[j]) < trows) & (static_cast<int>(csb[j]) < nsb_left);
          cp_async16_if<0, 0>(slot_sa + doff[j], (c2[j] ? base2 : base1) + coff[j], ok);
        }
      }
    }
    cp_async_commit();
  };

  // Weight stages first (they do not depend on the previous kernel), then x.
#pragma unroll 1
  for (int s = 0; s < D - 1; ++s) issue(s, ring_sa + s * STAGE);
  pdl_wait();

  // ---- x staging: the CTA's K-column of every vector, in fragment order.  Thread t handles
  // the 4-value chunks t + 256 k of the 8 x 256 chunks: all its loads are issued first, so
  // their latencies overlap.
  const int kc0 = 256 * kBatchColSB * wk;
  constexpr int kChunks = 64 * kBatchColSB;  // 4-value chunks per vector in the K-column
  constexpr int kItems = kBatchMax * kChunks / kBatchThreads;
  uint2 raw[kItems];
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const int idx = threadIdx.x + kBatchThreads * k, v = idx / kChunks, c = idx % kChunks;
    raw[k] = make_uint2(0u, 0u);
    if (v < a.M && (c >> 6) < ncols)
      raw[k] = __ldcg(reinterpret_cast<const uint2*>(a.x + static_cast<int64_t>(v) * a.K + kc0) + c);
  }
  if constexpr (Fmt::kBF16) {
    // per vector: sigma with max |x| * 2^sigma in [2^14, 2^15) over this K-column
    int* const vmax = reinterpret_cast<int*>(vscale);
    if (threadIdx.x < kBatchMax) vmax[threadIdx.x] = 0;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const int v = (threadIdx.x + kBatchThreads * k) / kChunks;  // uniform over the warp
      uint32_t m = max(max(raw[k].x & 0x7FFFu, (raw[k].x >> 16) & 0x7FFFu),
                       max(raw[k].y & 0x7FFFu, (raw[k].y >> 16) & 0x7FFFu));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0 && m) atomicMax(vmax + v, static_cast<int>(m));
    }
    __syncthreads();
    if (threadIdx.x < kBatchMax) {
      const int m = vmax[threadIdx.x];
      const int e8 = (m >> 7) & 0xFF;  // bf16 biased exponent of the largest |x|
      vmax[threadIdx.x] = m ? max(-100, min(100, 141 - e8)) : 0;  // sigma
    }
    __syncthreads();
  }
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const int idx = threadIdx.x + kBatchThreads * k, v = idx / kChunks, c = idx % kChunks;
    const int sb = c >> 6, e = 4 * (c & 63);
    uint2 r = raw[k];
    if constexpr (Fmt::kBF16) {
      const float f = p2(reinterpret_cast<const int*>(vscale)[v]);
      const __half2 h0 = __floats2half2_rn(bf2f(r.x) * f, bf2f(r.x >> 16) * f);
      const __half2 h1 = __floats2half2_rn(bf2f(r.y) * f, bf2f(r.y >> 16) * f);
      r = make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
    }
    int step, tq;
    uint2 val;
    Fmt::chunk_slot(e, step, tq, val, r);
    const int ln = 4 * v + tq;
    *reinterpret_cast<uint2*>(smem + L.xa + ((sb * 16 + step) * 32 + ln) * 8) = val;
    if constexpr (Fmt::kMinTerm) {
      // group sums of x (for the minimum term): 8 chunks of 4 make a group of 32
      float gs = __half2float(__ushort_as_half(static_cast<unsigned short>(r.x & 0xFFFFu))) +
                 __half2float(__ushort_as_half(static_cast<unsigned short>(r.x >> 16))) +
                 __half2float(__ushort_as_half(static_cast<unsigned short>(r.y & 0xFFFFu))) +
                 __half2float(__ushort_as_half(static_cast<unsigned short>(r.y >> 16)));
      gs += __shfl_xor_sync(0xffffffffu, gs, 1);
      gs += __shfl_xor_sync(0xffffffffu, gs, 2);
      gs += __shfl_xor_sync(0xffffffffu, gs, 4);
      if ((c & 7) == 0) {
        const int grp = e >> 5;  // group of the superblock: the m16n8k8 k index
        const float sc = gs * (1.0f / 64.0f);  // keeps the fp16 parts finite for any fp16 x
        const __half hi = __float2half_rn(sc);
        const __half lo = __float2half_rn(sc - __half2float(hi));
        uint16_t* dst = reinterpret_cast<uint16_t*>(smem + L.xs + (sb * 32 + 4 * v + (grp >> 1)) * 8);
        dst[grp & 1] = __half_as_ushort(hi);
        dst[2 + (grp & 1)] = __half_as_ushort(lo);
      }
    }
  }
  __syncthreads();
  // output scales of this lane's vectors 2 t4 and 2 t4 + 1 (bf16 x: 2^-sigma)
  float osc0 = 1.f, osc1 = 1.f;
  if constexpr (Fmt::kBF16) {
    osc0 = p2(-reinterpret_cast<const int*>(vscale)[2 * t4]);
    osc1 = p2(-reinterpret_cast<const int*>(vscale)[2 * t4 + 1]);
  }

  // ---- main loop: tiles of 16 rows, in stages of 2 superblocks.
  float* const out = a.Wk == 1 ? a.y + p_lo : a.ws + (static_cast<int64_t>(wk) * a.M) * a.N + p_lo;
  const int v0 = 2 * t4, v1 = 2 * t4 + 1;  // this lane's vectors
  uint32_t magic;  // fp16 (1024, 1024): the exponent under which two nibbles become fp16
  asm("mov.b32 %0, 0x64006400;" : "=r"(magic));
  uint32_t cs = ring_sa, is = ring_sa + (D - 1) * STAGE;
  const uint32_t xa_lane = xa_sa + lane * 8, xs_lane = xs_sa + lane * 8;
  float y[4] = {0.f, 0.f, 0.f, 0.f};  // (row g, v0), (row g, v1), (row g + 8, v0), (row g + 8, v1)
  float dq[2][4] = {};                 // folded scales: the tile's accumulator chains
  for (int st = 0; st < nst; ++st) {
    issue(st + D - 1, is);
    cp_async_wait<D - 1>();
    __syncwarp();
    const int tile = st / spt, h = st - tile * spt;
    uint32_t rg = cs + g * SLICE, r8 = cs + (g + 8) * SLICE;
    if constexpr (Fmt::kWindow) {
      const uint32_t o = static_cast<uint32_t>((kBatchColSB * wk + SSB * h) * SB) & 15u;
      rg += o;
      r8 += o;
    }
#pragma unroll
    for (int c = 0; c < SSB; ++c) {
      const int sbk = SSB * h + c;  // superblock within the K-column
      if (sbk < ncols) {
        if constexpr (Fmt::kFolded)
          Fmt::superblock(rg, r8, c, t4, xa_lane + sbk * 16 * 256, xs_lane + sbk * 256, magic, dq);
        else
          Fmt::superblock(rg, r8, c, t4, xa_lane + sbk * 16 * 256, xs_lane + sbk * 256, magic, y);
      }
    }
    __syncwarp();  // every lane is done with this slot before it is refilled
    is = cs;
    cs = (cs + STAGE == ring_end) ? ring_sa : cs + STAGE;
    if (h == spt - 1) {  // the tile's last stage: its sums are complete
      if constexpr (Fmt::kFolded) {
        y[0] = (dq[0][0] + dq[1][0]) * osc0;
        y[1] = (dq[0][1] + dq[1][1]) * osc1;
        y[2] = (dq[0][2] + dq[1][2]) * osc0;
        y[3] = (dq[0][3] + dq[1][3]) * osc1;
#pragma unroll
        for (int u = 0; u < 4; ++u) dq[0][u] = dq[1][u] = 0.f;
      }
      const int r0 = tile * kBatchRows + g, r1 = r0 + 8;
      if (v0 < a.M && r0 < nrows) out[static_cast<int64_t>(v0) * a.N + r0] = y[0];
      if (v1 < a.M && r0 < nrows) out[static_cast<int64_t>(v1) * a.N + r0] = y[1];
      if (v0 < a.M && r1 < nrows) out[static_cast<int64_t>(v0) * a.N + r1] = y[2];
      if (v1 < a.M && r1 < nrows) out[static_cast<int64_t>(v1) * a.N + r1] = y[3];
#pragma unroll
      for (int u = 0; u < 4; ++u) y[u] = 0.f;
    }
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
      // Every (vector, row) of the range: the Wk column sums added in column order.  Four
      // outputs per thread and pass, so their loads are in flight together.
      const int total = ncta * a.M;
      for (int i0 = threadIdx.x; i0 < total; i0 += 4 * kBatchThreads) {
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        int64_t o[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = min(i0 + u * kBatchThreads, total - 1);
          const int v = i / ncta;
          o[u] = static_cast<int64_t>(v) * a.N + r_lo + (i - v * ncta);
        }
        for (int w = 0; w < a.Wk; ++w) {
          const float* col = a.ws + static_cast<int64_t>(w) * a.M * a.N;
#pragma unroll
          for (int u = 0; u < 4; ++u) s[u] += __ldcg(col + o[u]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (i0 + u * kBatchThreads < total) a.y[o[u]] = s[u];
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
