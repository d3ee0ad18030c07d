// Per-format register decoders of the streaming GEMV kernel.
//
// Work split: a row is cut into 256-element superblocks (one Q4_K / Q5_K / Q6_K / TQ1_0
// block, eight Q8_0 blocks, or 256 NVFP4 elements with their 16 scales) and into K-columns
// of 8 superblocks (2048 elements).  A warp owns one K-column; lane L = 4*col + c owns
// piece c (64 elements) of superblock col.
//
// Activations: the CTA first stages x in shared memory once, converted piece by piece (8
// elements) into the form the decoders consume (stage_piece); each lane then copies its
// 64 values into 32 registers (two values each) and keeps them for the whole kernel,
// together with the per-group sums its offsets need.  Every product of an activation and
// a weight is exact, and every result meets |y - y_ref| <= 2e-3 sum|x w| + 1e-5 for any
// finite x: the only rounding is fp32 accumulation.
//
// Integer-code formats (Q4_K, Q5_K, Q6_K, Q8_0) multiply the fp16 activations as they are
// ("Writing a high performant GEMV + dequant for Metal", section "Compute": the activations
// are read as floats and multiplied by the masked nibbles).  A code v < 1024 placed in the
// low bits of a 16-bit half is the f16 subnormal v * 2^-24, so the masked (or assembled)
// code bytes, moved into 16-bit lanes by a byte permute, are exact f16 operands; the mixed
// precision FMA (sm_100+ `fma.rn.f32.f16`) forms x * v * 2^-24 exactly and adds it in fp32.
// Signed codes (Q6_K's q - 32, Q8_0's int8) are made by one exact f16x2 subtraction of the
// offset in the same subnormal units.  Group scales, minima and the 2^-24 units are applied
// once per group in fp32.
//
// TQ1_0 also keeps x as fp16: its base-3 digits, stepped out of the packed bytes two at a
// time, become the exact f16 operands (t - 1) 2^-16 of the same FMAs.
//
// NVFP4 decodes E2M1/E4M3 with the hardware f16 conversions and accumulates f16 x f16
// products exactly in fp32; its bf16 activations are staged as f16 times a power of two per
// 32-element chunk.  An element that this form does not hold exactly leaves a residual (its
// low bits, an exact bf16 value) that a per-lane correction adds in fp32; typical inputs
// have none, so the correction costs one predicate test per row.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "qgemv_ptx.cuh"

namespace qg {

enum : int { F_Q4K = 0, F_NVFP4 = 1, F_TQ10 = 2, F_Q5K = 3, F_Q6K = 4, F_Q80 = 5 };

__device__ __forceinline__ float h2f(uint32_t bits16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}
__device__ __forceinline__ float bf2f(uint32_t bits16) { return __uint_as_float((bits16 & 0xFFFFu) << 16); }
__device__ __forceinline__ float p2(int e) { return __uint_as_float(static_cast<uint32_t>(e + 127) << 23); }

constexpr float kTwo24 = 16777216.0f;
constexpr float kTwo44 = 17592186044416.0f;
constexpr float kTwo48 = 281474976710656.0f;

// c0 += lo(x2) * lo(q2); c1 += hi(x2) * hi(q2)   (f16 x f16 -> exact product, f32 accumulate)
__device__ __forceinline__ void fma2h(float& c0, float& c1, uint32_t x2, uint32_t q2) {
  asm("{\n\t.reg .b16 xl, xh, ql, qh;\n\t"
      "mov.b32 {xl, xh}, %2;\n\tmov.b32 {ql, qh}, %3;\n\t"
      "fma.rn.f32.f16 %0, xl, ql, %0;\n\tfma.rn.f32.f16 %1, xh, qh, %1;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "r"(x2), "r"(q2));
}
// lo(a) * (lo(b), hi(b))
__device__ __forceinline__ void mul1x2h(float& r0, float& r1, uint32_t a2, uint32_t b2) {
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.f16 %0, al, bl, 0f00000000;\n\tfma.rn.f32.f16 %1, al, bh, 0f00000000;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "r"(a2), "r"(b2));
}
// a - b on f16 pairs (subnormals kept: exact whenever the difference is representable)
__device__ __forceinline__ uint32_t hsub2_raw(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Bytes 0 and 2 / 1 and 3 of a word, each zero-extended into a 16-bit lane.
__device__ __forceinline__ uint32_t bytes02(uint32_t w) { return __byte_perm(w, 0u, 0x4240); }
__device__ __forceinline__ uint32_t bytes13(uint32_t w) { return __byte_perm(w, 0u, 0x4341); }

// ------------------------------------------------------------------- activation staging
// The CTA's copy of x in shared memory: q: 16-bit values, 16 bytes of padding after every 64
// (so the 64-element pieces that the lanes of a quarter-warp copy to registers start on
// different banks), e[K/32] one float per 32-element chunk, g: the decoder's per-superblock
// area (kCoefSB bytes each), for decoders that have one.
struct XStage {
  uint16_t* q;
  float* e;
  int* g;
};
// 16-byte slot of staged piece i (elements 8i .. 8i+7) in q, and the first value of the
// 32-element chunk that starts at element k (a multiple of 32).
__device__ __forceinline__ int xq_slot(int i) { return i + (i >> 3); }
__device__ __forceinline__ const uint16_t* xq_at(const uint16_t* q, int k) { return q + k + 8 * (k >> 6); }

// max of the two unsigned 16-bit halves, lane-wise (sm_90+)
__device__ __forceinline__ uint32_t vmax_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Eight words starting at a 2-byte aligned shared address: nine aligned 32-bit loads and
// a byte permute per word (selector 0x3210 when already 4-byte aligned, 0x5432 otherwise).
__device__ __forceinline__ void lds_words8_a2(uint32_t addr, uint32_t (&w)[8]) {
  const uint32_t a4 = addr & ~3u;
  const uint32_t sel = (addr & 2u) ? 0x5432u : 0x3210u;
  uint32_t W[9];
#pragma unroll
  for (int i = 0; i < 9; ++i) W[i] = lds_u32(a4 + 4 * i);
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = __byte_perm(W[j], W[j + 1], sel);
}

// 32 staged values (one chunk).  Loaded with volatile shared loads: the registers they fill
// must stay live for the whole kernel, and a plain load could be re-executed on every stage
// instead (rematerialised from the staging buffer).
__device__ __forceinline__ void ld_chunk(const uint16_t* q, uint32_t (&v)[16]) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(q));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 a = lds_v4(sa + 16 * i);
    v[4 * i] = a.x, v[4 * i + 1] = a.y, v[4 * i + 2] = a.z, v[4 * i + 3] = a.w;
  }
}
// Activations are staged in 16-byte pieces of 8 values: piece i of x is loaded by one
// thread, and the four pieces of a 32-element chunk sit in four adjacent lanes of a warp
// (i & 3 == lane & 3), which share the chunk's largest magnitude by two shuffles.
__device__ __forceinline__ uint32_t chunk_max_mag(const uint4& v) {
  uint32_t m2 = vmax_u16x2(vmax_u16x2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu), vmax_u16x2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
  uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
  return max(m, __shfl_xor_sync(0xffffffffu, m, 2));
}

// Integer-code formats: x stays fp16, exactly.  Within every four consecutive elements
// (a, b, c, d) the pairs are stored as (a, c), (b, d): the order in which bytes02 / bytes13
// deliver the codes of a code word.  With SUMS, e[chunk] = (sum of the chunk's 32 values,
// in fp32, in a fixed order) * 2^-24, for the group-minimum term.
template <bool SUMS>
__device__ __forceinline__ void flt_stage_piece(uint4 v, int i, const XStage& X) {
  reinterpret_cast<uint4*>(X.q)[xq_slot(i)] =
      make_uint4(__byte_perm(v.x, v.y, 0x5410), __byte_perm(v.x, v.y, 0x7632), __byte_perm(v.z, v.w, 0x5410),
                 __byte_perm(v.z, v.w, 0x7632));
  if constexpr (SUMS) {
    float s0 = 0.f, s1 = 0.f;
    fma2h(s0, s1, v.x, 0x3C003C00u);  // times f16 1.0
    fma2h(s0, s1, v.y, 0x3C003C00u);
    fma2h(s0, s1, v.z, 0x3C003C00u);
    fma2h(s0, s1, v.w, 0x3C003C00u);
    float s = s0 + s1;
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    if ((i & 3) == 0) X.e[i >> 2] = s * (1.0f / kTwo24);
  }
}

// Lane registers of an integer-code decoder: runs run0 (registers 0..15) and run1 (16..31)
// of its piece as staged fp16 pairs.
struct FltX {
  uint32_t xr[32];

  __device__ __forceinline__ void load(const XStage& X, int k0, int k1, bool active) {
    if (active) {
      uint32_t a[16], b[16];
      ld_chunk(xq_at(X.q, k0), a);
      ld_chunk(xq_at(X.q, k1), b);
#pragma unroll
      for (int i = 0; i < 16; ++i) xr[i] = a[i], xr[16 + i] = b[i];
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) xr[i] = 0u;
    }
  }
};

// ------------------------------------------------------------------------------- Q4_K
// Lane piece c = quant bytes [32c, 32c+32): low nibbles are elements 64c + t (group 2c),
// high nibbles 64c + 32 + t (group 2c+1).  For quant word u (bytes t..t+3, t = 4u) the
// low nibbles of bytes 0, 2 and of bytes 1, 3 become f16 pairs by one mask each (w and
// w >> 8), and the high nibbles, left in place (16 q), by one mask each: eight exact
// products per word, against the activation pairs (t, t+2), (t+1, t+3) and (32+t, 34+t),
// (33+t, 35+t).  Per group: d*s*sum(x q) - dmin*m*sum(x), the scale/min pairs unpacked
// from the block header (the page's mask arithmetic) and multiplied by d / dmin with
// mixed-precision FMAs (a 6-bit value placed as an f16 subnormal gives d*s*2^-24 exactly).
struct DecQ4K : FltX {
  static constexpr int kSB = 144, kSB2 = 0;
  static constexpr float kOut = kTwo48;  // unit of compute()'s results
  static constexpr int kCoefSB = 0;
  static constexpr bool kResidual = false;
  int c;
  uint32_t sel_s, sel_h, m1, m2, shm;
  uint32_t qoff;   // byte offset of this lane's quants in a block
  float xs0, xs1;  // sums of x over the two groups, times 2^-24 (xs1 also times 16)

  __device__ __forceinline__ static void stage_piece(uint4 v, int i, const XStage& X) { flt_stage_piece<true>(v, i, X); }

  __device__ __forceinline__ void init(int c_) {
    c = c_;
    qoff = 16 + 32 * c;
    const int j = 2 * (c & 1);  // byte index of group 2c within its scale word
    // c < 2: s = S[2c], S[2c+1] & 63 (word h.y); c >= 2: low nibbles of S[2c+4], S[2c+5]
    // (word h.w) with bits 6..7 of S[2c-4], S[2c-3] (word h.y) above them.
    sel_s = (c < 2) ? (0x4040u | ((j + 1) << 8) | j) : (0x4040u | ((j + 5) << 8) | (j + 4));
    sel_h = 0x4040u | ((j + 1) << 8) | j;
    m1 = (c < 2) ? 0x003F003Fu : 0x000F000Fu;
    m2 = (c < 2) ? 0u : 0x00300030u;
    shm = (c < 2) ? 0u : 4u;
  }
  __device__ __forceinline__ void load_x(const XStage& X, int sbcol, int c_, bool active) {
    const int k0 = 256 * sbcol + 64 * c_;
    load(X, k0, k0 + 32, active);
    xs0 = active ? X.e[k0 >> 5] : 0.f;
    xs1 = active ? X.e[(k0 >> 5) + 1] : 0.f;
  }
  // d*s_lo, d*s_hi, dmin*m_lo, dmin*m_hi (times 2^-24) from the block header.
  __device__ __forceinline__ void scales(const uint4 h, float& ds_lo, float& ds_hi, float& dm_lo, float& dm_hi) const {
    const uint32_t s2 = (__byte_perm(h.y, h.w, sel_s) & m1) | ((__byte_perm(h.y, 0u, sel_h) >> 2) & m2);
    const uint32_t m2v = ((__byte_perm(h.z, h.w, sel_s) >> shm) & m1) | ((__byte_perm(h.z, 0u, sel_h) >> 2) & m2);
    mul1x2h(ds_lo, ds_hi, h.x, s2);
    mul1x2h(dm_lo, dm_hi, h.x >> 16, m2v);
  }
  // a_lo = sum(x q) 2^-24 (group 2c), a_hi the same for group 2c+1 (16 times too large with
  // HI16: high nibbles left in place).  Returns the piece's sum in units of 2^-48 (kOut):
  // ds_lo a_lo + ds_hi a_hi - (dm_lo xs0 + dm_hi xs1).
  template <bool HI16>
  __device__ __forceinline__ float combine(float a_lo, float a_hi, float ds_lo, float ds_hi, float dm_lo,
                                           float dm_hi) const {
    const float m = fmaf(dm_lo, xs0, dm_hi * xs1);
    return fmaf(ds_lo, a_lo, fmaf(HI16 ? ds_hi * 0.0625f : ds_hi, a_hi, -m));
  }

  // blk: shared-window address of the row's superblock slice (16-byte aligned).
  // Two phases, so that a stage's rows are all loaded before any is computed: fetch() reads
  // the lane's 48 bytes of the row from the ring, compute() needs no shared memory.
  struct Raw {
    uint4 h, q0, q1;
  };
  __device__ __forceinline__ Raw fetch(uint32_t blk, uint32_t) const {
    const uint32_t q = blk + qoff;
    return Raw{lds_v4_at<0>(blk), lds_v4_at<0>(q), lds_v4_at<16>(q)};
  }
  __device__ __forceinline__ float compute(const Raw& R_) const {
    const uint4 h = R_.h, q0 = R_.q0, q1 = R_.q1;
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    float a[2] = {0.f, 0.f}, b[2] = {0.f, 0.f};  // the rows of a stage give the other chains
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t w8 = w[u] >> 8;
      fma2h(a[0], a[1], xr[2 * u], w[u] & 0x000F000Fu);      // elements t, t+2
      fma2h(a[0], a[1], xr[2 * u + 1], w8 & 0x000F000Fu);    // t+1, t+3
      fma2h(b[0], b[1], xr[16 + 2 * u], w[u] & 0x00F000F0u);  // 32+t, 34+t (16 q)
      fma2h(b[0], b[1], xr[16 + 2 * u + 1], w8 & 0x00F000F0u);
    }
    float ds_lo, ds_hi, dm_lo, dm_hi;
    scales(h, ds_lo, ds_hi, dm_lo, dm_hi);
    return combine<true>(a[0] + a[1], b[0] + b[1], ds_lo, ds_hi, dm_lo, dm_hi);
  }
};

// ------------------------------------------------------------------------------- Q5_K
// Q4_K's piece split, activations and scales (quants at byte 48); the fifth bit of element
// 64c + t (low) / 64c + 32 + t (high) is bit 2c / 2c+1 of qh[t] (qh at byte 16).  A funnel
// shift brings it to bit 4 of each byte, next to its nibble; the 5-bit code bytes then
// become f16 pairs by byte permutes.
struct DecQ5K : DecQ4K {
  static constexpr int kSB = 176, kSB2 = 0;
  static constexpr int kCoefSB = 0;
  uint32_t rl, rh;  // rotate amounts bringing bit 2c / 2c+1 of each byte to bit 4

  __device__ __forceinline__ void init(int c_) {
    DecQ4K::init(c_);
    rl = (4u - 2u * c_) & 31u;
    rh = (3u - 2u * c_) & 31u;
  }

  struct Raw {
    uint32_t b;
  };
  __device__ __forceinline__ Raw fetch(uint32_t blk, uint32_t) const { return Raw{blk}; }
  __device__ __forceinline__ float compute(const Raw& R_) const { return row(R_.b, 0); }
  __device__ __forceinline__ float row(uint32_t blk, uint32_t) const {
    const uint4 h = lds_v4(blk);
    const uint4 e0 = lds_v4(blk + 16);
    const uint4 e1 = lds_v4(blk + 32);
    const uint4 qa = lds_v4(blk + 48 + 32 * c);
    const uint4 qb = lds_v4(blk + 64 + 32 * c);
    const uint32_t w[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    const uint32_t e[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
    float a[2] = {0.f, 0.f}, b[2] = {0.f, 0.f};
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t L = (w[u] & 0x0F0F0F0Fu) | (__funnelshift_l(e[u], e[u], rl) & 0x10101010u);
      const uint32_t H = ((w[u] >> 4) & 0x0F0F0F0Fu) | (__funnelshift_l(e[u], e[u], rh) & 0x10101010u);
      fma2h(a[0], a[1], xr[2 * u], bytes02(L));
      fma2h(a[0], a[1], xr[2 * u + 1], bytes13(L));
      fma2h(b[0], b[1], xr[16 + 2 * u], bytes02(H));
      fma2h(b[0], b[1], xr[16 + 2 * u + 1], bytes13(H));
    }
    float ds_lo, ds_hi, dm_lo, dm_hi;
    scales(h, ds_lo, ds_hi, dm_lo, dm_hi);
    return combine<false>(a[0] + a[1], b[0] + b[1], ds_lo, ds_hi, dm_lo, dm_hi);
  }
};

// ------------------------------------------------------------------------------- Q6_K
// Lane piece c: half H = c>>1, rr = c&1.  Byte ql[64H + 32rr + t] holds, in its low
// nibble, element 128H + 32rr + t and, in its high nibble, element 128H + 32(rr+2) + t;
// their top two bits are bits 2rr..2rr+1 / 2rr+4..2rr+5 of qh[32H + t].  The 6-bit codes
// are assembled bytewise, moved into f16 lanes and made signed (q - 32) by one exact f16
// subtraction per pair; each 16-element scale group keeps its own sums.  Blocks are 210
// bytes (2-byte aligned), so quant words are read with a byte permute.
struct DecQ6K : FltX {
  static constexpr int kSB = 210, kSB2 = 0;
  static constexpr float kOut = kTwo24;
  static constexpr int kCoefSB = 0;
  static constexpr bool kResidual = false;
  int c;
  uint32_t rlo, rhi;  // rotate amounts bringing qh bits 2rr / 2rr+4 of each byte to bit 4

  __device__ __forceinline__ static void stage_piece(uint4 v, int i, const XStage& X) { flt_stage_piece<false>(v, i, X); }
  __device__ __forceinline__ void init(int c_) {
    c = c_;
    const int rr = c & 1;
    rlo = (4u - 2u * rr) & 31u;
    rhi = (32u - 2u * rr) & 31u;
  }
  __device__ __forceinline__ void load_x(const XStage& X, int sbcol, int c_, bool active) {
    const int k0 = 256 * sbcol + 128 * (c_ >> 1) + 32 * (c_ & 1);
    load(X, k0, k0 + 64, active);
  }

  // blk: shared-window address of the row's superblock (2-byte aligned: 210-byte blocks).
  struct Raw {
    uint32_t b;
  };
  __device__ __forceinline__ Raw fetch(uint32_t blk, uint32_t) const { return Raw{blk}; }
  __device__ __forceinline__ float compute(const Raw& R_) const { return row(R_.b, 0); }
  __device__ __forceinline__ float row(uint32_t blk, uint32_t) const {
    const int H = c >> 1, rr = c & 1;
    const uint32_t ql = blk + 64 * H + 32 * rr;
    const uint32_t qh = blk + 128 + 32 * H;
    float acc[4][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
    uint32_t lw[8], hw[8];
    lds_words8_a2(ql, lw);
    lds_words8_a2(qh, hw);
    constexpr uint32_t k32 = 0x00200020u;  // 32 * 2^-24 in both halves
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t l = lw[u], e = hw[u];
      const uint32_t lo6 = (l & 0x0F0F0F0Fu) | (__funnelshift_l(e, e, rlo) & 0x30303030u);
      const uint32_t hi6 = ((l >> 4) & 0x0F0F0F0Fu) | (__funnelshift_l(e, e, rhi) & 0x30303030u);
      const int g = u >> 2;
      fma2h(acc[g][0], acc[g][1], xr[2 * u], hsub2_raw(bytes02(lo6), k32));
      fma2h(acc[g][0], acc[g][1], xr[2 * u + 1], hsub2_raw(bytes13(lo6), k32));
      fma2h(acc[2 + g][0], acc[2 + g][1], xr[16 + 2 * u], hsub2_raw(bytes02(hi6), k32));
      fma2h(acc[2 + g][0], acc[2 + g][1], xr[16 + 2 * u + 1], hsub2_raw(bytes13(hi6), k32));
    }
    const uint32_t sc = blk + 192 + 8 * H + 2 * rr;
    const float d = h2f(lds_u16(blk + 208));
    const float r0 = fmaf(static_cast<float>(lds_s8(sc)), acc[0][0] + acc[0][1],
                          static_cast<float>(lds_s8(sc + 1)) * (acc[1][0] + acc[1][1]));
    const float r1 = fmaf(static_cast<float>(lds_s8(sc + 4)), acc[2][0] + acc[2][1],
                          static_cast<float>(lds_s8(sc + 5)) * (acc[3][0] + acc[3][1]));
    return d * (r0 + r1);
  }
};

// ------------------------------------------------------------------------------- Q8_0
// A superblock is eight 34-byte blocks; lane piece c = blocks 2c and 2c+1 (elements
// 64c + 32e + j).  Each int8 code byte is offset to b + 128 (one xor per word), moved into
// an f16 lane as the subnormal (b + 128) 2^-24 and made b 2^-24 by one exact subtraction.
struct DecQ80 : FltX {
  static constexpr int kSB = 272, kSB2 = 0;
  static constexpr float kOut = kTwo24;
  static constexpr int kCoefSB = 0;
  static constexpr bool kResidual = false;
  int c;

  __device__ __forceinline__ static void stage_piece(uint4 v, int i, const XStage& X) { flt_stage_piece<false>(v, i, X); }
  __device__ __forceinline__ void init(int c_) { c = c_; }
  __device__ __forceinline__ void load_x(const XStage& X, int sbcol, int c_, bool active) {
    load(X, 256 * sbcol + 64 * c_, 256 * sbcol + 64 * c_ + 32, active);
  }

  struct Raw {
    uint32_t b;
  };
  __device__ __forceinline__ Raw fetch(uint32_t blk, uint32_t) const { return Raw{blk}; }
  __device__ __forceinline__ float compute(const Raw& R_) const { return row(R_.b, 0); }
  __device__ __forceinline__ float row(uint32_t sblk, uint32_t) const {
    constexpr uint32_t k128 = 0x00800080u;  // 128 * 2^-24 in both halves
    float r[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint32_t blk = sblk + 34 * (2 * c + e);
      float a[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t qw[8];
      lds_words8_a2(blk + 2, qw);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t v = qw[u] ^ 0x80808080u;
        const int o = 2 * (u & 1);
        fma2h(a[o], a[o + 1], xr[16 * e + 2 * u], hsub2_raw(bytes02(v), k128));
        fma2h(a[o], a[o + 1], xr[16 * e + 2 * u + 1], hsub2_raw(bytes13(v), k128));
      }
      r[e] = h2f(lds_u16(blk)) * ((a[0] + a[1]) + (a[2] + a[3]));
    }
    return r[0] + r[1];
  }
};

// The lane's residual correction: residual values (16-bit, in the lane's own element order
// j = 0..63) at shared address `ra` and the 64-bit mask of the elements that have one.
struct Residual {
  uint32_t rm0, rm1, ra;
  __device__ __forceinline__ bool any() const { return (rm0 | rm1) != 0u; }
  __device__ __forceinline__ void clear() { rm0 = rm1 = 0u, ra = 0u; }
  // Calls f(j, residual bits) for every set element, in increasing j.
  template <class F>
  __device__ __forceinline__ void each(F&& f) const {
    uint32_t m0 = rm0, m1 = rm1;
    while (m0 | m1) {
      int j;
      if (m0) {
        j = __ffs(m0) - 1;
        m0 &= m0 - 1u;
      } else {
        j = 31 + __ffs(m1);
        m1 &= m1 - 1u;
      }
      f(j, lds_u16(ra + 2u * j));
    }
  }
};

// ------------------------------------------------------------------------------- NVFP4
// Superblock = 256 elements: 128 nibble bytes (stream 1) and 16 E4M3 scales (stream 2).
// Lane piece c = nibble bytes [32c, 32c+32) and scales [4c, 4c+4); register k holds the
// activations of nibble byte k (elements 2k, 2k+1: low nibble = even element).  E2M1 and
// E4M3 are decoded by the hardware conversions to f16 (exact for every code) and f16 x f16
// products accumulate exactly in fp32.  The bf16 activations are staged per 32-element
// chunk as f16 times a power of two chosen from the chunk's largest |x| so that every
// value is below 2^14: f16 then holds each bf16 value exactly unless it is more than about
// 2^30 below the chunk maximum.  Such an element's lost low bits (a bf16 value) are its
// residual, added by the lane's correction; the power of two is removed per chunk.
// Decoder area per superblock: residuals [256] (bf16 bits, element order), then one mask
// byte per 8 elements.
struct DecNVFP4 {
  static constexpr int kSB = 128, kSB2 = 16;
  static constexpr float kOut = 1.f;
  static constexpr int kCoefSB = 256 * 2 + 32;
  static constexpr bool kResidual = true;
  uint32_t xr[32];
  float xf0, xf1;
  int c;
  Residual res;

  __device__ __forceinline__ static void stage_piece(uint4 v, int i, const XStage& X) {
    const int e8 = static_cast<int>(chunk_max_mag(v) >> 7);  // bf16 biased exponent
    // 2^(e8-127) <= max < 2^(e8-126): scale by 2^(140 - e8) to bring it below 2^14.
    const int sg = max(-126, min(126, 140 - e8));
    const float scale = p2(sg), inv = p2(-sg);
    uint32_t w[4] = {v.x, v.y, v.z, v.w}, r[4];
    uint32_t mask = 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float x0 = bf2f(w[k]), x1 = bf2f(w[k] >> 16);
      const __half2 h2 = __floats2half2_rn(x0 * scale, x1 * scale);
      // what f16 lost: x minus its staged value (an exact bf16 value: low bits of x)
      const float d0 = x0 - __low2float(h2) * inv, d1 = x1 - __high2float(h2) * inv;
      r[k] = (__float_as_uint(d0) >> 16) | (__float_as_uint(d1) & 0xFFFF0000u);
      mask |= (d0 != 0.f ? 1u : 0u) << (2 * k);
      mask |= (d1 != 0.f ? 1u : 0u) << (2 * k + 1);
      w[k] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    reinterpret_cast<uint4*>(X.q)[xq_slot(i)] = make_uint4(w[0], w[1], w[2], w[3]);
    if ((i & 3) == 0) X.e[i >> 2] = inv;
    uint8_t* area = reinterpret_cast<uint8_t*>(X.g) + (i >> 5) * kCoefSB;
    reinterpret_cast<uint4*>(area)[i & 31] = make_uint4(r[0], r[1], r[2], r[3]);
    area[512 + (i & 31)] = static_cast<uint8_t>(mask);
  }
  __device__ __forceinline__ void init(int c_) { c = c_; }
  __device__ __forceinline__ void load_x(const XStage& X, int sbcol, int c_, bool active) {
    const int k0 = 256 * sbcol + 64 * c_;
    if (active) {
      uint32_t a[16], b[16];
      ld_chunk(xq_at(X.q, k0), a);
      ld_chunk(xq_at(X.q, k0 + 32), b);
#pragma unroll
      for (int i = 0; i < 16; ++i) xr[i] = a[i], xr[16 + i] = b[i];
      const uint32_t ea = static_cast<uint32_t>(__cvta_generic_to_shared(X.e));
      xf0 = __uint_as_float(lds_u32(ea + 4 * (k0 >> 5)));
      xf1 = __uint_as_float(lds_u32(ea + 4 * (k0 >> 5) + 4));
      const uint32_t area = static_cast<uint32_t>(__cvta_generic_to_shared(X.g)) + sbcol * kCoefSB;
      res.rm0 = lds_u32(area + 512 + 8 * c_);
      res.rm1 = lds_u32(area + 512 + 8 * c_ + 4);
      res.ra = area + 128 * c_;
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) xr[i] = 0u;
      xf0 = xf1 = 0.f;
      res.clear();
    }
  }

  __device__ __forceinline__ static uint32_t e2m1x2(uint32_t byte) {
    uint32_t h;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h) : "r"(byte));
    return h;
  }
  // The four bytes of w (eight E2M1 codes) as four f16 pairs, byte i in h[i].
  __device__ __forceinline__ static void e2m1x8(uint32_t w, uint32_t (&h)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
  }
  __device__ __forceinline__ static uint32_t e4m3x2(uint32_t two) {
    uint32_t h;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h) : "r"(two));
    return h;
  }

  struct Raw {
    uint4 q0, q1;
    uint32_t s4;
  };
  __device__ __forceinline__ Raw fetch(uint32_t nib, uint32_t sc) const {
    return Raw{lds_v4(nib + 32 * c), lds_v4(nib + 32 * c + 16), lds_u32(sc + 4 * c)};
  }
  __device__ __forceinline__ float compute(const Raw& R_) const {
    const uint4 q0 = R_.q0, q1 = R_.q1;
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const uint32_t s4 = R_.s4 & 0x7F7F7F7Fu;  // |scale|
    float r[2] = {0.f, 0.f};
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t wd = w[2 * b + u];
        uint32_t hw[4];
        e2m1x8(wd, hw);
        fma2h(a0, a1, xr[8 * b + 4 * u + 0], hw[0]);
        fma2h(a2, a3, xr[8 * b + 4 * u + 1], hw[1]);
        fma2h(a0, a1, xr[8 * b + 4 * u + 2], hw[2]);
        fma2h(a2, a3, xr[8 * b + 4 * u + 3], hw[3]);
      }
      const float sv = h2f(e4m3x2((s4 >> (8 * b)) & 0xFFu));
      r[b >> 1] = fmaf(sv, (a0 + a1) + (a2 + a3), r[b >> 1]);
    }
    return fmaf(r[0], xf0, r[1] * xf1);
  }
  __device__ __forceinline__ bool has_residual() const { return res.any(); }
  // Sum of residual x element j times its weight e2m1 * |e4m3|, exact products in fp32.
  __device__ __forceinline__ float correction(uint32_t nib, uint32_t sc) const {
    float acc = 0.f;
    res.each([&](int j, uint32_t rbits) {
      const uint32_t byte = lds_u8(nib + 32 * c + (j >> 1));
      const uint32_t e = e2m1x2(byte);
      const float wv = h2f((j & 1) ? (e >> 16) : e);
      const float sv = h2f(e4m3x2(lds_u8(sc + 4 * c + (j >> 4)) & 0x7Fu));
      acc = fmaf(bf2f(rbits), wv * sv, acc);
    });
    return acc;
  }
};

// ------------------------------------------------------------------------------- TQ1_0
// Lane piece c = qs bytes [12c, 12c+12) (three words) and qh byte c: 60 + 4 elements.  The
// digit of weight n of byte b is floor(3^(n+1) b / 256) mod 3 ("metal: TQ1_0 kernel
// performance", section 1), taken one step at a time: with r = b, r3 = 3 r gives the digit
// t = r3 >> 8 (0, 1 or 2) and r = r3 & 255 for the next one.  Bytes 0, 2 and bytes 1, 3 of
// a word share the 16-bit lanes of one register, so one multiply steps two bytes (3 r < 2^16
// never carries into the next lane).  t stays in bits 8..9 of its lane: as an f16 subnormal
// that is t 2^-16, made (t - 1) 2^-16 by one exact f16 subtraction, and its product with
// the fp16 activation is exact (mixed-precision FMA, fp32 accumulation); d and 2^16 are
// applied once per row.  The qh byte carries four digits: its two lanes start at digits 0
// and 2 (b and 9b mod 256) and take two steps.
// Staging: x is kept as fp16, each superblock in its own 528-byte slot of the decoder area
// (256 values and 16 bytes of padding, so the slots of the eight superblocks a warp reads
// start on different banks); each lane gathers its 64 values once, in the order compute()
// takes them: register 10 w + 2 n + h holds the digit-n elements of bytes h and h + 2 of
// word w, registers 30 / 31 the qh digits (0, 2) / (1, 3).
struct DecTQ10 : FltX {
  static constexpr int kSB = 54, kSB2 = 0;
  static constexpr float kOut = 65536.f;
  static constexpr int kCoefSB = 528;
  static constexpr bool kResidual = false;
  int c;

  __device__ __forceinline__ static void stage_piece(uint4 v, int i, const XStage& X) {
    *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(X.g) + kCoefSB * (i >> 5) + 16 * (i & 31)) = v;
  }
  __device__ __forceinline__ void init(int c_) { c = c_; }
  __device__ __forceinline__ void load_x(const XStage& X, int sbcol, int c_, bool active) {
    if (!active) {
#pragma unroll
      for (int i = 0; i < 32; ++i) xr[i] = 0u;
      return;
    }
    const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(X.g)) + static_cast<uint32_t>(kCoefSB * sbcol);
    // Word w of the piece is bytes p..p+3, p = 12 c + 4 w (a multiple of 4, all in one of the
    // two qs runs), whose digit-n elements are four consecutive staged values: one 8-byte load
    // and two byte permutes give the pairs (bytes 0, 2) and (1, 3).
#pragma unroll
    for (int w = 0; w < 3; ++w) {
      const int p = 12 * c_ + 4 * w;
      const bool first = p < 32;
#pragma unroll
      for (int n = 0; n < 5; ++n) {
        const int e = first ? 32 * n + p : 160 + 16 * n + (p - 32);
        uint32_t lo, hi;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(lo), "=r"(hi) : "r"(base + 2u * static_cast<uint32_t>(e)));
        xr[10 * w + 2 * n] = __byte_perm(lo, hi, 0x5410);      // elements p, p + 2
        xr[10 * w + 2 * n + 1] = __byte_perm(lo, hi, 0x7632);  // p + 1, p + 3
      }
    }
    auto xv = [&](int n) { return lds_u16(base + 2u * static_cast<uint32_t>(240 + 4 * n + c_)); };
    xr[30] = xv(0) | (xv(2) << 16);
    xr[31] = xv(1) | (xv(3) << 16);
  }

  struct Raw {
    uint32_t b;
  };
  __device__ __forceinline__ Raw fetch(uint32_t blk, uint32_t) const { return Raw{blk}; }
  __device__ __forceinline__ float compute(const Raw& R_) const { return row(R_.b, 0); }
  // blk: shared-window address of the row's block (2-byte aligned: 54-byte blocks).
  __device__ __forceinline__ float row(uint32_t blk, uint32_t) const {
    constexpr uint32_t kOne = 0x01000100u;  // 2^-16 in both f16 halves
    const uint32_t q = blk + 12 * c;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < 3; ++w) {
      const uint32_t W = lds_u16(q + 4 * w) | (lds_u16(q + 4 * w + 2) << 16);
      uint32_t re = bytes02(W), ro = bytes13(W);
#pragma unroll
      for (int n = 0; n < 5; ++n) {
        re *= 3u;
        ro *= 3u;
        const uint32_t te = hsub2_raw(re & 0x03000300u, kOne), to = hsub2_raw(ro & 0x03000300u, kOne);
        if (n < 4) re &= 0x00FF00FFu, ro &= 0x00FF00FFu;
        fma2h(acc[0], acc[1], xr[10 * w + 2 * n], te);
        fma2h(acc[2], acc[3], xr[10 * w + 2 * n + 1], to);
      }
    }
    const uint32_t b = lds_u8(blk + 48 + c);
    uint32_t rq = b | (((9u * b) & 0xFFu) << 16);
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      rq *= 3u;
      const uint32_t tq = hsub2_raw(rq & 0x03000300u, kOne);
      rq &= 0x00FF00FFu;
      fma2h(acc[2 * n], acc[2 * n + 1], xr[30 + n], tq);
    }
    return h2f(lds_u16(blk + 52)) * ((acc[0] + acc[1]) + (acc[2] + acc[3]));
  }
};

}  // namespace qg
