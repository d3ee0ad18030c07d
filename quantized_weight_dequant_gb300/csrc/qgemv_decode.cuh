// Per-format register decoders of the streaming GEMV kernel.
//
// Work split: a row is cut into 256-element superblocks (one Q4_K / Q5_K / Q6_K / TQ1_0
// block, eight Q8_0 blocks, or 256 NVFP4 elements with their 16 scales) and into K-columns
// of 8 superblocks (2048 elements).  A warp owns one K-column; lane L = 4*col + c owns
// piece c (64 elements) of superblock col.
//
// Activations: the CTA first stages x in shared memory once, converted piece by piece (8
// elements) into the form the decoders consume (stage_piece); each lane then copies the
// two 32-element runs of its piece into 32 registers (two values each) and keeps them for
// the whole kernel, together with the per-chunk factors and sums its offsets need.
//
// Integer-code formats (Q4_K, Q5_K, Q6_K, Q8_0): the codes of a row piece are byte
// vectors (masked or assembled in place, never shifted down to one code per register)
// and their dot product with the activations, held as 16-bit fixed point, is taken four
// bytes at a time by dp2a into int32; the group scale, the group minimum times the
// activation sum, and the fixed-point exponent are applied once per group.  This is the
// GPU form of the Q4_K page's "multiply by the masked nibbles and correct once per
// block" ("Writing a high performant GEMV + dequant for Metal", section "Compute").
// Block scales use mixed-precision FMAs (sm_100+ `fma.rn.f32.f16`): a small integer v in
// the low 10 bits of a 16-bit half is the f16 subnormal v * 2^-24, so d (f16) times a
// 6-bit scale placed there is d*s*2^-24, exact, in one instruction.
// NVFP4 decodes E2M1/E4M3 with the hardware f16 conversions and accumulates f16 x f16
// products exactly in fp32; TQ1_0 extracts base-3 digits with one rounding FMA each.
#pragma once
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

// ------------------------------------------------------------------- activation staging
// The CTA's copy of x in shared memory: q[K] 16-bit values, e[K/32] one float per 32-element
// chunk, s[K/16] one int per 16-element half chunk (what they hold depends on the format).
struct XStage {
  uint16_t* q;
  float* e;
  int* s;
  int* g;  // decoder coefficients (kCoefSB bytes per superblock), for decoders that have them
};

// d = c + a.h0 * b.b0 + a.h1 * b.b1 (lo) / a.h0 * b.b2 + a.h1 * b.b3 (hi); a two int16,
// b four bytes (unsigned or signed).
__device__ __forceinline__ int dp2a_lo_u(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2a_hi_u(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2a_lo_s(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.lo.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2a_hi_s(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.hi.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

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

// Integer-code formats: a chunk of 32 fp16 activations becomes 16-bit fixed point
// x_i = round(x * 2^e), e chosen per chunk so that its largest |x| lands in [2^14, 2^15).
// Values within a factor 16 of that largest one convert exactly (fp16 has 11 significant
// bits); smaller ones are rounded with error at most 2^-15 of it.  Dot products with the
// integer codes are then exact int32 sums (dp2a), and the code term and the group-minimum
// term of a block use the same x_i.
//  * Conversion is one mixed-precision FMA per value: x (f16) * 2^e1 (f16) + M (f32) with
//    M = 1.5 * 2^(23 - (e - e1)), whose ulp is 2^(e1 - e), so the sum is rounded to
//    nearest-even at exactly x * 2^e; its low 16 mantissa bits are then x_i in two's
//    complement (|x_i| < 2^15 keeps the sum inside M's binade).  e1 = min(e, 15) keeps
//    the f16 multiplier representable.
//  * e[chunk] = 2^-e * 2^24 (the 2^24 undoes the subnormal scale factors of the decoders);
//    s[2 chunk + h] = sum of x_i over half h, by dp2a against byte weights (1, 1).
__device__ __forceinline__ void int_stage_piece(uint4 v, int i, const XStage& X) {
  const int e5 = static_cast<int>(chunk_max_mag(v) >> 10);  // f16 biased exponent
  const int e = 29 - min(e5, 30);                             // in [-1, 29]
  const int e1 = min(e, 15);
  const uint32_t s1 = static_cast<uint32_t>(e1 + 15) << 10;  // f16 2^e1
  const uint32_t s2 = s1 | (s1 << 16);
  const float M = 1.5f * p2(23 - (e - e1));
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
  int hs = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float f0 = M, f1 = M;
    fma2h(f0, f1, w[k], s2);
    w[k] = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x5410);
    hs = dp2a_lo_u(w[k], 0x0101u, hs);
  }
  hs += __shfl_xor_sync(0xffffffffu, hs, 1);
  reinterpret_cast<uint4*>(X.q)[i] = make_uint4(w[0], w[1], w[2], w[3]);
  if ((i & 1) == 0) X.s[i >> 1] = hs;
  if ((i & 3) == 0) X.e[i >> 2] = p2(24 - e);
}

// Lane registers of an integer-code decoder: runs run0 (registers 0..15) and run1 (16..31)
// of its piece, the factors of their chunks and the four half-chunk sums (run0 halves,
// then run1 halves).
struct IntX {
  uint32_t xr[32];
  float xf0, xf1;
  int xsi[4];

  __device__ __forceinline__ void load(const XStage& X, int k0, int k1, bool active) {
    if (active) {
      uint32_t a[16], b[16];
      ld_chunk(X.q + k0, a);
      ld_chunk(X.q + k1, b);
#pragma unroll
      for (int i = 0; i < 16; ++i) xr[i] = a[i], xr[16 + i] = b[i];
      const uint32_t ea = static_cast<uint32_t>(__cvta_generic_to_shared(X.e));
      const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(X.s));
      xf0 = __uint_as_float(lds_u32(ea + 4 * (k0 >> 5)));
      xf1 = __uint_as_float(lds_u32(ea + 4 * (k1 >> 5)));
      xsi[0] = static_cast<int>(lds_u32(sa + 4 * (k0 >> 4)));
      xsi[1] = static_cast<int>(lds_u32(sa + 4 * (k0 >> 4) + 4));
      xsi[2] = static_cast<int>(lds_u32(sa + 4 * (k1 >> 4)));
      xsi[3] = static_cast<int>(lds_u32(sa + 4 * (k1 >> 4) + 4));
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) xr[i] = 0u;
      xf0 = xf1 = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) xsi[m] = 0;
    }
  }
};

// ------------------------------------------------------------------------------- Q4_K
// Lane piece c = quant bytes [32c, 32c+32): low nibbles are elements 64c + t (group 2c),
// high nibbles 64c + 32 + t (group 2c+1).  For quant word u (bytes t..t+3, t = 4u) the
// four low nibbles (word & 0x0F0F0F0F) and the four high nibbles ((word >> 4) & same)
// are byte vectors that dp2a multiplies with activation pairs (t, t+1), (t+2, t+3) and
// (32+t, 33+t), (34+t, 35+t): the GPU form of "multiply by the masked nibbles and correct
// once per block" of the Q4_K page (section "Compute").  Group scales: d (f16) times a
// 6-bit scale placed as an f16 subnormal gives d*s*2^-24 in one instruction.
struct DecQ4K : IntX {
  static constexpr int kSB = 144, kSB2 = 0;
  static constexpr int kCoefSB = 0;
  int c;
  uint32_t sel_s, sel_h, m1, m2, shm;
  uint32_t qoff;   // byte offset of this lane's quants in a block
  float xs0, xs1;  // activation sums of the two groups

  __device__ __forceinline__ static void stage_piece(uint4 v, int i, const XStage& X) { int_stage_piece(v, i, X); }

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
  __device__ __forceinline__ void load_x_plain(const XStage& X, int sbcol, int c_, bool active) {
    load(X, 256 * sbcol + 64 * c_, 256 * sbcol + 64 * c_ + 32, active);
    xs0 = static_cast<float>(xsi[0] + xsi[1]);
    xs1 = static_cast<float>(xsi[2] + xsi[3]);
  }
  __device__ __forceinline__ void load_x(const XStage& X, int sbcol, int c_, bool active) {
    load_x_plain(X, sbcol, c_, active);
    xs1 *= 16.f;  // the high-nibble dot products come out 16 times too large: see row()
    xf1 *= 0.0625f;
  }
  // d*s_lo, d*s_hi, dmin*m_lo, dmin*m_hi (times 2^-24) from the block header.
  __device__ __forceinline__ void scales(const uint4 h, float& ds_lo, float& ds_hi, float& dm_lo, float& dm_hi) const {
    const uint32_t s2 = (__byte_perm(h.y, h.w, sel_s) & m1) | ((__byte_perm(h.y, 0u, sel_h) >> 2) & m2);
    const uint32_t m2v = ((__byte_perm(h.z, h.w, sel_s) >> shm) & m1) | ((__byte_perm(h.z, 0u, sel_h) >> 2) & m2);
    mul1x2h(ds_lo, ds_hi, h.x, s2);
    mul1x2h(dm_lo, dm_hi, h.x >> 16, m2v);
  }
  __device__ __forceinline__ float combine(int lo, int hi, float ds_lo, float ds_hi, float dm_lo, float dm_hi) const {
    const float t0 = fmaf(ds_lo, static_cast<float>(lo), -dm_lo * xs0);
    const float t1 = fmaf(ds_hi, static_cast<float>(hi), -dm_hi * xs1);
    return fmaf(t0, xf0, t1 * xf1);
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
    int a0 = 0, a1 = 0, b0 = 0, b1 = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      // High nibbles stay in place: dp2a sees 16 q, and 16 * sum(x_i q) still fits int32
      // (32 values * 240 * 2^15 < 2^28); the factor 16 is folded into xs1 and xf1.
      const uint32_t L = w[u] & 0x0F0F0F0Fu, H = w[u] & 0xF0F0F0F0u;
      int& al = (u & 1) ? a1 : a0;
      int& ah = (u & 1) ? b1 : b0;
      al = dp2a_lo_u(xr[2 * u], L, al);
      al = dp2a_hi_u(xr[2 * u + 1], L, al);
      ah = dp2a_lo_u(xr[16 + 2 * u], H, ah);
      ah = dp2a_hi_u(xr[16 + 2 * u + 1], H, ah);
    }
    float ds_lo, ds_hi, dm_lo, dm_hi;
    scales(h, ds_lo, ds_hi, dm_lo, dm_hi);
    return combine(a0 + a1, b0 + b1, ds_lo, ds_hi, dm_lo, dm_hi);
  }
};

// ------------------------------------------------------------------------------- Q5_K
// Q4_K's piece split and activations (quants at byte 48); the fifth bit of element 64c + t
// (low) / 64c + 32 + t (high) is bit 2c / 2c+1 of qh[t] (qh at byte 16).  A funnel shift
// brings it to bit 4 of each byte, next to its nibble, before the dot product.
struct DecQ5K : DecQ4K {
  static constexpr int kSB = 176, kSB2 = 0;
  static constexpr int kCoefSB = 0;
  uint32_t rl, rh;  // rotate amounts bringing bit 2c / 2c+1 of each byte to bit 4

  __device__ __forceinline__ void load_x(const XStage& X, int sbcol, int c_, bool active) {
    load_x_plain(X, sbcol, c_, active);
  }

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
    int a0 = 0, a1 = 0, b0 = 0, b1 = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t L = (w[u] & 0x0F0F0F0Fu) | (__funnelshift_l(e[u], e[u], rl) & 0x10101010u);
      const uint32_t H = ((w[u] >> 4) & 0x0F0F0F0Fu) | (__funnelshift_l(e[u], e[u], rh) & 0x10101010u);
      int& al = (u & 1) ? a1 : a0;
      int& ah = (u & 1) ? b1 : b0;
      al = dp2a_lo_u(xr[2 * u], L, al);
      al = dp2a_hi_u(xr[2 * u + 1], L, al);
      ah = dp2a_lo_u(xr[16 + 2 * u], H, ah);
      ah = dp2a_hi_u(xr[16 + 2 * u + 1], H, ah);
    }
    float ds_lo, ds_hi, dm_lo, dm_hi;
    scales(h, ds_lo, ds_hi, dm_lo, dm_hi);
    return combine(a0 + a1, b0 + b1, ds_lo, ds_hi, dm_lo, dm_hi);
  }
};

// ------------------------------------------------------------------------------- Q6_K
// Lane piece c: half H = c>>1, rr = c&1.  Byte ql[64H + 32rr + t] holds, in its low
// nibble, element 128H + 32rr + t and, in its high nibble, element 128H + 32(rr+2) + t;
// their top two bits are bits 2rr..2rr+1 / 2rr+4..2rr+5 of qh[32H + t].  The 6-bit codes
// are assembled bytewise and dotted with dp2a; the -32 offset is removed with the integer
// sums of the activations of each 16-element scale group.  Blocks are 210 bytes (2-byte
// aligned), so quant words are read as 16-bit pairs.
struct DecQ6K : IntX {
  static constexpr int kSB = 210, kSB2 = 0;
  static constexpr int kCoefSB = 0;
  int c;
  uint32_t rlo, rhi;  // rotate amounts bringing qh bits 2rr / 2rr+4 of each byte to bit 4

  __device__ __forceinline__ static void stage_piece(uint4 v, int i, const XStage& X) { int_stage_piece(v, i, X); }
  __device__ __forceinline__ void init(int c_) {
    c = c_;
    const int rr = c & 1;
    rlo = (4u - 2u * rr) & 31u;
    rhi = (32u - 2u * rr) & 31u;
  }
  __device__ __forceinline__ void load_x(const XStage& X, int sbcol, int c_, bool active) {
    const int k0 = 256 * sbcol + 128 * (c_ >> 1) + 32 * (c_ & 1);
    load(X, k0, k0 + 64, active);
    xsi[0] *= 32, xsi[1] *= 32, xsi[2] *= 32, xsi[3] *= 32;
    xf0 *= 1.0f / kTwo24;
    xf1 *= 1.0f / kTwo24;
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
    int acc[4] = {0, 0, 0, 0};
    uint32_t lw[8], hw[8];
    lds_words8_a2(ql, lw);
    lds_words8_a2(qh, hw);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t l = lw[u], e = hw[u];
      const uint32_t lo6 = (l & 0x0F0F0F0Fu) | (__funnelshift_l(e, e, rlo) & 0x30303030u);
      const uint32_t hi6 = ((l >> 4) & 0x0F0F0F0Fu) | (__funnelshift_l(e, e, rhi) & 0x30303030u);
      const int g = u >> 2;
      acc[g] = dp2a_lo_u(xr[2 * u], lo6, acc[g]);
      acc[g] = dp2a_hi_u(xr[2 * u + 1], lo6, acc[g]);
      acc[2 + g] = dp2a_lo_u(xr[16 + 2 * u], hi6, acc[2 + g]);
      acc[2 + g] = dp2a_hi_u(xr[16 + 2 * u + 1], hi6, acc[2 + g]);
    }
    const uint32_t sc = blk + 192 + 8 * H + 2 * rr;
    const float d = h2f(lds_u16(blk + 208));
    const float r0 = fmaf(static_cast<float>(lds_s8(sc)), static_cast<float>(acc[0] - xsi[0]),
                          static_cast<float>(lds_s8(sc + 1)) * static_cast<float>(acc[1] - xsi[1]));
    const float r1 = fmaf(static_cast<float>(lds_s8(sc + 4)), static_cast<float>(acc[2] - xsi[2]),
                          static_cast<float>(lds_s8(sc + 5)) * static_cast<float>(acc[3] - xsi[3]));
    return d * fmaf(r0, xf0, r1 * xf1);
  }
};

// ------------------------------------------------------------------------------- Q8_0
// A superblock is eight 34-byte blocks; lane piece c = blocks 2c and 2c+1 (elements
// 64c + 32e + j).  The int8 codes are dotted directly with signed dp2a.
struct DecQ80 : IntX {
  static constexpr int kSB = 272, kSB2 = 0;
  static constexpr int kCoefSB = 0;
  int c;

  __device__ __forceinline__ static void stage_piece(uint4 v, int i, const XStage& X) { int_stage_piece(v, i, X); }
  __device__ __forceinline__ void init(int c_) { c = c_; }
  __device__ __forceinline__ void load_x(const XStage& X, int sbcol, int c_, bool active) {
    load(X, 256 * sbcol + 64 * c_, 256 * sbcol + 64 * c_ + 32, active);
    xf0 *= 1.0f / kTwo24;
    xf1 *= 1.0f / kTwo24;
  }

  struct Raw {
    uint32_t b;
  };
  __device__ __forceinline__ Raw fetch(uint32_t blk, uint32_t) const { return Raw{blk}; }
  __device__ __forceinline__ float compute(const Raw& R_) const { return row(R_.b, 0); }
  __device__ __forceinline__ float row(uint32_t sblk, uint32_t) const {
    float r[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint32_t blk = sblk + 34 * (2 * c + e);
      int a0 = 0, a1 = 0;
      uint32_t qw[8];
      lds_words8_a2(blk + 2, qw);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t wd = qw[u];
        int& a = (u & 1) ? a1 : a0;
        a = dp2a_lo_s(xr[16 * e + 2 * u], wd, a);
        a = dp2a_hi_s(xr[16 * e + 2 * u + 1], wd, a);
      }
      r[e] = h2f(lds_u16(blk)) * static_cast<float>(a0 + a1);
    }
    return fmaf(r[0], xf0, r[1] * xf1);
  }
};

// ------------------------------------------------------------------------------- NVFP4
// Superblock = 256 elements: 128 nibble bytes (stream 1) and 16 E4M3 scales (stream 2).
// Lane piece c = nibble bytes [32c, 32c+32) and scales [4c, 4c+4); register k holds the
// activations of nibble byte k (elements 2k, 2k+1: low nibble = even element).  E2M1 and
// E4M3 are decoded by the hardware conversions to f16 (exact for every code) and f16 x f16
// products accumulate exactly in fp32.  The bf16 activations are staged per 32-element
// chunk as f16 times a power of two chosen from the chunk's largest |x| so that every
// value is below 2^14: f16 then holds each bf16 value exactly (values 2^27 times smaller
// than the largest lose low bits); the power of two is removed per chunk from the result.
struct DecNVFP4 {
  static constexpr int kSB = 128, kSB2 = 16;
  static constexpr int kCoefSB = 0;
  uint32_t xr[32];
  float xf0, xf1;
  int c;

  __device__ __forceinline__ static void stage_piece(uint4 v, int i, const XStage& X) {
    const int e8 = static_cast<int>(chunk_max_mag(v) >> 7);  // bf16 biased exponent
    // 2^(e8-127) <= max < 2^(e8-126): scale by 2^(140 - e8) to bring it below 2^14.
    const float scale = p2(max(-126, min(126, 140 - e8)));
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 h2 = __floats2half2_rn(bf2f(w[k]) * scale, bf2f(w[k] >> 16) * scale);
      w[k] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    reinterpret_cast<uint4*>(X.q)[i] = make_uint4(w[0], w[1], w[2], w[3]);
    if ((i & 3) == 0) X.e[i >> 2] = 1.0f / scale;
  }
  __device__ __forceinline__ void init(int c_) { c = c_; }
  __device__ __forceinline__ void load_x(const XStage& X, int sbcol, int c_, bool active) {
    const int k0 = 256 * sbcol + 64 * c_;
    if (active) {
      uint32_t a[16], b[16];
      ld_chunk(X.q + k0, a);
      ld_chunk(X.q + k0 + 32, b);
#pragma unroll
      for (int i = 0; i < 16; ++i) xr[i] = a[i], xr[16 + i] = b[i];
      const uint32_t ea = static_cast<uint32_t>(__cvta_generic_to_shared(X.e));
      xf0 = __uint_as_float(lds_u32(ea + 4 * (k0 >> 5)));
      xf1 = __uint_as_float(lds_u32(ea + 4 * (k0 >> 5) + 4));
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) xr[i] = 0u;
      xf0 = xf1 = 0.f;
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
};

// ------------------------------------------------------------------------------- TQ1_0
// Lane piece c = qs bytes [12c, 12c+12) (three words) and qh byte c.  For a byte b whose
// digits n = 0..4 weigh activations y_0..y_4: sum_n y_n t_n(b) = sum_{k=1..5} g_k F_k(b)
// with F_k(b) = floor(3^k b / 256), g_k = y_{k-1} - 3 y_k, y_5 = 0; qh bytes carry four
// digits, so their y_4 is 0 ("metal: TQ1_0 kernel performance", section 1, the zero-padded
// collapse).  Here everything is integer: the activations are 13-bit fixed point with one
// exponent per superblock, so every g_k fits int16; F_k of four bytes at once comes from
// multiplying the even and the odd bytes, spread into 16-bit lanes, by 3 (k times; b 3^k <
// 2^16 never carries into the next lane) and picking byte 1 of each lane; dp2a then takes
// the dot products with the int16 g pairs.
struct DecTQ10 {
  static constexpr int kSB = 54, kSB2 = 0;
  uint32_t gw[3][5][2];  // [word][k-1]: g of bytes 0,1 and of bytes 2,3 as int16 pairs
  int gq[4];             // qh byte: g_k, k = 1..4
  int xsum;              // sum of the lane's 64 fixed-point activations
  float xf;              // 2^-e of the superblock
  int c;

  __device__ __forceinline__ static int elem_of(int p, int n) {
    if (p < 32) return 32 * n + p;
    if (p < 48) return 160 + 16 * n + (p - 32);
    return 240 + 4 * n + (p - 48);
  }
  // 13-bit fixed point per superblock: the 32 pieces of a superblock are the 32 lanes of one
  // warp, which share the largest magnitude by shuffles.  Same conversion as the integer
  // formats (one mixed-precision FMA per value), with the maximum landing in [2^12, 2^13).
  __device__ __forceinline__ static void stage_piece(uint4 v, int i, const XStage& X) {
    uint32_t m2 = vmax_u16x2(vmax_u16x2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu), vmax_u16x2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int e5 = static_cast<int>(m >> 10);
    const int e = 27 - min(e5, 30);  // in [-3, 27]
    const int e1 = min(e, 15);
    const uint32_t s1 = static_cast<uint32_t>(e1 + 15) << 10;
    const uint32_t s2 = s1 | (s1 << 16);
    const float M = 1.5f * p2(23 - (e - e1));
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float f0 = M, f1 = M;
      fma2h(f0, f1, w[k], s2);
      w[k] = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x5410);
    }
    reinterpret_cast<uint4*>(X.q)[i] = make_uint4(w[0], w[1], w[2], w[3]);
    if ((i & 31) == 0) X.e[i >> 5] = p2(-e);
  }
  __device__ __forceinline__ void init(int c_) { c = c_; }
  // Collapse coefficients of every lane piece of the staged x, computed once per CTA by all
  // its threads (every warp of the CTA reads the same pieces).  Item (superblock, piece c,
  // part): parts 0..2 are the piece's qs words, part 3 its qh byte; each writes its g_k and
  // its partial sum of x into the piece's 40 words: g of word w at 10 w + 2 (k - 1) + h (h: bytes
  // 0,1 / 2,3 as int16 pairs), the qh g_k at 30 + k - 1, the four partial sums at 34..37.
  static constexpr int kCoefSB = 4 * 160;
  __device__ static void prep(const XStage& X, int nsb, int tid, int nthreads) {
    const uint32_t q0 = static_cast<uint32_t>(__cvta_generic_to_shared(X.q));
    for (int it = tid; it < 16 * nsb; it += nthreads) {
      const int sb = it >> 4, c = (it >> 2) & 3, part = it & 3;
      const uint32_t qa = q0 + 512u * sb;
      auto xi = [&](int p, int n) -> int { return static_cast<int>(static_cast<int16_t>(lds_u16(qa + 2 * elem_of(p, n)))); };
      int* g = X.g + (4 * sb + c) * 40;
      int xs = 0;
      if (part < 3) {
        int gg[4][5];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int p = 12 * c + 4 * part + j;
          int y[6];
#pragma unroll
          for (int n = 0; n < 5; ++n) y[n] = xi(p, n), xs += y[n];
          y[5] = 0;
#pragma unroll
          for (int k = 1; k <= 5; ++k) gg[j][k - 1] = y[k - 1] - 3 * y[k];
        }
#pragma unroll
        for (int k = 0; k < 5; ++k) {
          g[10 * part + 2 * k] = static_cast<int>((static_cast<uint32_t>(gg[0][k]) & 0xFFFFu) |
                                                  (static_cast<uint32_t>(gg[1][k]) << 16));
          g[10 * part + 2 * k + 1] = static_cast<int>((static_cast<uint32_t>(gg[2][k]) & 0xFFFFu) |
                                                      (static_cast<uint32_t>(gg[3][k]) << 16));
        }
      } else {
        int y[5];
#pragma unroll
        for (int n = 0; n < 4; ++n) y[n] = xi(48 + c, n), xs += y[n];
        y[4] = 0;
#pragma unroll
        for (int k = 1; k <= 4; ++k) g[30 + k - 1] = y[k - 1] - 3 * y[k];
      }
      g[34 + part] = xs;
    }
  }
  __device__ __forceinline__ void load_x(const XStage& X, int sbcol, int c_, bool active) {
    if (active) {
      const uint32_t ga = static_cast<uint32_t>(__cvta_generic_to_shared(X.g)) + 160u * (4 * sbcol + c_);
      uint32_t v[40];
#pragma unroll
      for (int i = 0; i < 10; ++i) {
        const uint4 t = lds_v4(ga + 16 * i);
        v[4 * i] = t.x, v[4 * i + 1] = t.y, v[4 * i + 2] = t.z, v[4 * i + 3] = t.w;
      }
#pragma unroll
      for (int w = 0; w < 3; ++w)
#pragma unroll
        for (int k = 0; k < 5; ++k) gw[w][k][0] = v[10 * w + 2 * k], gw[w][k][1] = v[10 * w + 2 * k + 1];
#pragma unroll
      for (int k = 0; k < 4; ++k) gq[k] = static_cast<int>(v[30 + k]);
      xsum = static_cast<int>(v[34]) + static_cast<int>(v[35]) + static_cast<int>(v[36]) + static_cast<int>(v[37]);
      xf = X.e[sbcol];
    } else {
#pragma unroll
      for (int w = 0; w < 3; ++w)
#pragma unroll
        for (int k = 0; k < 5; ++k) gw[w][k][0] = gw[w][k][1] = 0u;
#pragma unroll
      for (int k = 0; k < 4; ++k) gq[k] = 0;
      xsum = 0;
      xf = 0.f;
    }
  }

  struct Raw {
    uint32_t b;
  };
  __device__ __forceinline__ Raw fetch(uint32_t blk, uint32_t) const { return Raw{blk}; }
  __device__ __forceinline__ float compute(const Raw& R_) const { return row(R_.b, 0); }
  // blk: shared-window address of the row's block (2-byte aligned: 54-byte blocks).
  __device__ __forceinline__ float row(uint32_t blk, uint32_t) const {
    const uint32_t q = blk + 12 * c;
    int acc = 0;
#pragma unroll
    for (int w = 0; w < 3; ++w) {
      const uint32_t W = lds_u16(q + 4 * w) | (lds_u16(q + 4 * w + 2) << 16);
      uint32_t pe = __byte_perm(W, 0u, 0x4240);  // bytes 0, 2 in 16-bit lanes
      uint32_t po = __byte_perm(W, 0u, 0x4341);  // bytes 1, 3
#pragma unroll
      for (int k = 0; k < 5; ++k) {
        pe *= 3u;
        po *= 3u;
        const uint32_t F = __byte_perm(pe, po, 0x7351);  // F_k of bytes 0..3
        acc = dp2a_lo_u(gw[w][k][0], F, acc);
        acc = dp2a_hi_u(gw[w][k][1], F, acc);
      }
    }
    uint32_t pq = lds_u8(blk + 48 + c);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      pq *= 3u;
      acc += gq[k] * static_cast<int>(pq >> 8);
    }
    const float d = h2f(lds_u16(blk + 52));
    return d * static_cast<float>(acc - xsum) * xf;
  }
};

}  // namespace qg
