// Per-format register decoders of the streaming GEMV kernel.
//
// Work split: a row is cut into 256-element superblocks (one Q4_K / Q5_K / Q6_K / TQ1_0
// block, eight Q8_0 blocks, or 256 NVFP4 elements with their 16 scales) and into K-columns
// of 8 superblocks (2048 elements).  A warp owns one K-column; lane L = 4*col + c owns
// piece c (64 elements) of superblock col.  The lane loads the activations of its piece
// once (two runs of 32 contiguous values) and keeps them in 32 registers of f16 pairs, in
// the order its decode consumes them, plus the activation sums its offsets need.
//
// Exact decode with mixed-precision FMAs (sm_100+ `fma.rn.f32.f16`): a small integer v
// stored in the low 10 bits of a 16-bit half is the f16 subnormal v * 2^-24, so masking
// two fields into the two halves of a 32-bit register (one LOP3 per pair) gives two
// operands whose product with an f16 activation is exact in fp32.  The 2^-24 (and the
// 2^4 of a field sitting four bits up) is removed once per block.  This is the GPU form
// of the Q4_K page's "multiply by the masked but unshifted nibble and correct once at
// the end" ("Writing a high performant GEMV + dequant for Metal", section "Compute").
// Block scales are combined the same way: d (f16) times a 6-bit scale placed as a
// subnormal gives d*s*2^-24 in one instruction, without integer-to-float conversion.
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
__device__ __forceinline__ uint32_t ld_u16(const uint8_t* p) { return *reinterpret_cast<const uint16_t*>(p); }
__device__ __forceinline__ uint32_t ld_u32_a2(const uint8_t* p) { return ld_u16(p) | (ld_u16(p + 2) << 16); }

constexpr float kTwo24 = 16777216.0f;
constexpr float kTwo48 = 281474976710656.0f;

// c0 += lo(x2) * lo(q2); c1 += hi(x2) * hi(q2)   (f16 x f16 -> exact product, f32 accumulate)
__device__ __forceinline__ void fma2h(float& c0, float& c1, uint32_t x2, uint32_t q2) {
  asm("{\n\t.reg .b16 xl, xh, ql, qh;\n\t"
      "mov.b32 {xl, xh}, %2;\n\tmov.b32 {ql, qh}, %3;\n\t"
      "fma.rn.f32.f16 %0, xl, ql, %0;\n\tfma.rn.f32.f16 %1, xh, qh, %1;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "r"(x2), "r"(q2));
}
// (lo(a) * lo(b), hi(a) * hi(b)) in fp32, exact for f16 inputs.
__device__ __forceinline__ void mul2h(float& r0, float& r1, uint32_t a2, uint32_t b2) {
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.f16 %0, al, bl, 0f00000000;\n\tfma.rn.f32.f16 %1, ah, bh, 0f00000000;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "r"(a2), "r"(b2));
}
// lo(a) * (lo(b), hi(b))
__device__ __forceinline__ void mul1x2h(float& r0, float& r1, uint32_t a2, uint32_t b2) {
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.f16 %0, al, bl, 0f00000000;\n\tfma.rn.f32.f16 %1, al, bh, 0f00000000;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "r"(a2), "r"(b2));
}

// Bytes 0 and 1 of v into the low bytes of the two halves: [v.b0, 0, v.b1, 0].
__device__ __forceinline__ uint32_t spread01(uint32_t v) { return __byte_perm(v, 0u, 0x4140u); }

// ------------------------------------------------------------------- activation loader
// Decoders describe their x registers by: run0(c), run1(c) = superblock offsets of the two
// 32-element runs of lane piece c; xloc(k, h) in [0, 64) = which of those 64 values is
// half h of register k (run0 values first); xsum(k, h) = which sum the value enters
// (-1: none), and xsum_scale() the factor the sums are stored with.
__device__ __forceinline__ void load_runs(const uint16_t* __restrict__ x, int64_t base0, int64_t base1, bool active,
                                          uint32_t (&v)[32]) {
  if (active) {
    const uint4* p0 = reinterpret_cast<const uint4*>(x + base0);
    const uint4* p1 = reinterpret_cast<const uint4*>(x + base1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 a = __ldg(p0 + i), b = __ldg(p1 + i);
      v[4 * i] = a.x, v[4 * i + 1] = a.y, v[4 * i + 2] = a.z, v[4 * i + 3] = a.w;
      v[16 + 4 * i] = b.x, v[16 + 4 * i + 1] = b.y, v[16 + 4 * i + 2] = b.z, v[16 + 4 * i + 3] = b.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0u;
  }
}
__device__ __forceinline__ uint32_t half_of(const uint32_t (&v)[32], int i) { return (v[i >> 1] >> (16 * (i & 1))) & 0xFFFFu; }

template <class D>
__device__ __forceinline__ void load_x_f16(D& d, const uint16_t* __restrict__ x, int64_t sb, int c, bool active) {
  uint32_t v[32];
  load_runs(x, sb * 256 + D::run0(c), sb * 256 + D::run1(c), active, v);
  float sums[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    const uint32_t lo = half_of(v, D::xloc(k, 0)), hi = half_of(v, D::xloc(k, 1));
    d.xr[k] = lo | (hi << 16);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int si = D::xsum(k, h);
      if (si >= 0) sums[si] += h2f(h ? hi : lo);
    }
  }
#pragma unroll
  for (int m = 0; m < 4; ++m) d.xs[m] = sums[m] * D::xsum_scale();
}

// ------------------------------------------------------------------------------- Q4_K
// Lane piece c = quant bytes [32c, 32c+32): low nibbles are elements 64c + t (group
// 2c), high nibbles 64c + 32 + t (group 2c+1).  For quant word u (bytes t..t+3, t = 4u)
// the four registers are x pairs (t, t+2), (t+1, t+3), (32+t, 34+t), (33+t, 35+t),
// matching the masks 0x000F000F and 0x00F000F0 on the word and on the word >> 8.
struct DecQ4K {
  static constexpr int kSB = 144, kSB2 = 0;
  static constexpr bool kBf16X = false;
  uint32_t xr[32];
  float xs[4];  // xs[0] = 2^24 * sum of low-nibble x, xs[1] = 2^24 * sum of high-nibble x
  int c;
  uint32_t sel_s, sel_h, m1, m2, shm;

  __device__ __forceinline__ static int run0(int c) { return 64 * c; }
  __device__ __forceinline__ static int run1(int c) { return 64 * c + 32; }
  __device__ __forceinline__ static constexpr int xloc(int k, int h) {
    return 4 * (k >> 2) + ((k & 3) == 1 || (k & 3) == 3 ? 1 : 0) + ((k & 3) >= 2 ? 32 : 0) + 2 * h;
  }
  __device__ __forceinline__ static constexpr int xsum(int k, int) { return (k & 3) < 2 ? 0 : 1; }
  __device__ __forceinline__ static float xsum_scale() { return kTwo24; }
  __device__ __forceinline__ void load_x(const uint16_t* __restrict__ x, int64_t sb, int c_, bool active) {
    load_x_f16(*this, x, sb, c_, active);
  }

  __device__ __forceinline__ void init(int c_) {
    c = c_;
    const int j = 2 * (c & 1);  // byte index of group 2c within its scale word
    // c < 2: s = S[2c], S[2c+1] & 63 (word h.y); c >= 2: low nibbles of S[2c+4], S[2c+5]
    // (word h.w) with bits 6..7 of S[2c-4], S[2c-3] (word h.y) above them.
    sel_s = (c < 2) ? (0x4040u | ((j + 1) << 8) | j) : (0x4040u | ((j + 5) << 8) | (j + 4));
    sel_h = 0x4040u | ((j + 1) << 8) | j;
    m1 = (c < 2) ? 0x003F003Fu : 0x000F000Fu;
    m2 = (c < 2) ? 0u : 0x00300030u;
    shm = (c < 2) ? 0u : 4u;
  }

  __device__ __forceinline__ float row(const uint8_t* blk, const uint8_t*) const {
    const uint4 h = *reinterpret_cast<const uint4*>(blk);
    const uint4 q0 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
    const uint4 q1 = *reinterpret_cast<const uint4*>(blk + 32 + 32 * c);
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f, b0 = 0.f, b1 = 0.f, b2 = 0.f, b3 = 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t wd = w[u], ws = wd >> 8;
      fma2h(a0, a1, xr[4 * u + 0], wd & 0x000F000Fu);
      fma2h(a2, a3, xr[4 * u + 1], ws & 0x000F000Fu);
      fma2h(b0, b1, xr[4 * u + 2], wd & 0x00F000F0u);
      fma2h(b2, b3, xr[4 * u + 3], ws & 0x00F000F0u);
    }
    const float acc_lo = (a0 + a1) + (a2 + a3);          // 2^-24 * sum x q (low nibbles)
    const float acc_hi = ((b0 + b1) + (b2 + b3)) * 0.0625f;  // high nibbles sat 4 bits up
    // scale and min pairs of groups 2c, 2c+1 spread into f16 halves
    const uint32_t s2 = (__byte_perm(h.y, h.w, sel_s) & m1) | ((__byte_perm(h.y, 0u, sel_h) >> 2) & m2);
    const uint32_t m2v = ((__byte_perm(h.z, h.w, sel_s) >> shm) & m1) | ((__byte_perm(h.z, 0u, sel_h) >> 2) & m2);
    float ds_lo, ds_hi, dm_lo, dm_hi;
    mul1x2h(ds_lo, ds_hi, h.x, s2);          // d * s * 2^-24
    mul1x2h(dm_lo, dm_hi, h.x >> 16, m2v);   // dmin * m * 2^-24
    const float sq = fmaf(ds_lo, acc_lo, ds_hi * acc_hi);
    const float mx = fmaf(dm_lo, xs[0], dm_hi * xs[1]);
    return fmaf(sq, kTwo48, -mx);
  }
};

// ------------------------------------------------------------------------------- Q5_K
// Q4_K's piece split and x order (quants at byte 48); the fifth bit of element 64c + t
// (low) / 64c + 32 + t (high) is bit 2c / 2c+1 of qh[t] (qh at byte 16).  It is rotated
// next to its nibble (bit 4 of a half for low nibbles, bit 8 for high nibbles, which
// already sit 4 bits up) before the multiply.
struct DecQ5K : DecQ4K {
  static constexpr int kSB = 176, kSB2 = 0;
  uint32_t rl, rh;  // rotate amounts bringing bit 2c to bit 4 and bit 2c+1 to bit 8

  __device__ __forceinline__ void init(int c_) {
    DecQ4K::init(c_);
    rl = (4u - 2u * c_) & 31u;
    rh = (8u - 2u * c_ - 1u) & 31u;
  }

  __device__ __forceinline__ float row(const uint8_t* blk, const uint8_t*) const {
    const uint4 h = *reinterpret_cast<const uint4*>(blk);
    const uint4 e0 = *reinterpret_cast<const uint4*>(blk + 16);
    const uint4 e1 = *reinterpret_cast<const uint4*>(blk + 32);
    const uint4 qa = *reinterpret_cast<const uint4*>(blk + 48 + 32 * c);
    const uint4 qb = *reinterpret_cast<const uint4*>(blk + 64 + 32 * c);
    const uint32_t w[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    const uint32_t e[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f, b0 = 0.f, b1 = 0.f, b2 = 0.f, b3 = 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t wd = w[u], ws = wd >> 8, ed = e[u], es = ed >> 8;
      const uint32_t l02 = (wd & 0x000F000Fu) | (__funnelshift_l(ed, ed, rl) & 0x00100010u);
      const uint32_t l13 = (ws & 0x000F000Fu) | (__funnelshift_l(es, es, rl) & 0x00100010u);
      const uint32_t h02 = (wd & 0x00F000F0u) | (__funnelshift_l(ed, ed, rh) & 0x01000100u);
      const uint32_t h13 = (ws & 0x00F000F0u) | (__funnelshift_l(es, es, rh) & 0x01000100u);
      fma2h(a0, a1, xr[4 * u + 0], l02);
      fma2h(a2, a3, xr[4 * u + 1], l13);
      fma2h(b0, b1, xr[4 * u + 2], h02);
      fma2h(b2, b3, xr[4 * u + 3], h13);
    }
    const float acc_lo = (a0 + a1) + (a2 + a3);
    const float acc_hi = ((b0 + b1) + (b2 + b3)) * 0.0625f;
    const uint32_t s2 = (__byte_perm(h.y, h.w, sel_s) & m1) | ((__byte_perm(h.y, 0u, sel_h) >> 2) & m2);
    const uint32_t m2v = ((__byte_perm(h.z, h.w, sel_s) >> shm) & m1) | ((__byte_perm(h.z, 0u, sel_h) >> 2) & m2);
    float ds_lo, ds_hi, dm_lo, dm_hi;
    mul1x2h(ds_lo, ds_hi, h.x, s2);
    mul1x2h(dm_lo, dm_hi, h.x >> 16, m2v);
    const float sq = fmaf(ds_lo, acc_lo, ds_hi * acc_hi);
    const float mx = fmaf(dm_lo, xs[0], dm_hi * xs[1]);
    return fmaf(sq, kTwo48, -mx);
  }
};

// ------------------------------------------------------------------------------- Q6_K
// Lane piece c: half H = c>>1, rr = c&1.  Byte ql[64H + 32rr + t] holds, in its low
// nibble, element 128H + 32rr + t and, in its high nibble, element 128H + 32(rr+2) + t;
// their top two bits are bits 2rr..2rr+1 / 2rr+4..2rr+5 of qh[32H + t].  The 6-bit
// fields are assembled in the low bits of each half; the -32 offset is removed with the
// activation sums of the four 16-element scale groups.  Blocks are 210 bytes (2-byte
// aligned), so quant words are read as 16-bit pairs.
struct DecQ6K {
  static constexpr int kSB = 210, kSB2 = 0;
  static constexpr bool kBf16X = false;
  uint32_t xr[32];
  float xs[4];  // 32 * 2^-24 * sums of groups (lo t<16, lo t>=16, hi t<16, hi t>=16)
  int c;
  uint32_t s_lo, s_hi;  // shifts bringing qh bits 2rr / 2rr+4 to bit 4 of each byte

  __device__ __forceinline__ static int run0(int c) { return 128 * (c >> 1) + 32 * (c & 1); }
  __device__ __forceinline__ static int run1(int c) { return 128 * (c >> 1) + 32 * (c & 1) + 64; }
  __device__ __forceinline__ static constexpr int xloc(int k, int h) { return DecQ4K::xloc(k, h); }
  __device__ __forceinline__ static constexpr int xsum(int k, int) { return ((k & 3) < 2 ? 0 : 2) + ((k >> 2) >= 4 ? 1 : 0); }
  __device__ __forceinline__ static float xsum_scale() { return 32.0f / kTwo24; }
  __device__ __forceinline__ void load_x(const uint16_t* __restrict__ x, int64_t sb, int c_, bool active) {
    load_x_f16(*this, x, sb, c_, active);
  }

  __device__ __forceinline__ void init(int c_) {
    c = c_;
    const int rr = c & 1;
    s_lo = 2 * rr;
    s_hi = 2 * rr + 4;
  }

  __device__ __forceinline__ float row(const uint8_t* blk, const uint8_t*) const {
    const int H = c >> 1, rr = c & 1;
    const uint8_t* ql = blk + 64 * H + 32 * rr;
    const uint8_t* qh = blk + 128 + 32 * H;
    float acc[4][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t l = ld_u32_a2(ql + 4 * u), e = ld_u32_a2(qh + 4 * u);
      const uint32_t lo6 = (l & 0x0F0F0F0Fu) | (((e >> s_lo) & 0x03030303u) << 4);
      const uint32_t hi6 = ((l >> 4) & 0x0F0F0F0Fu) | (((e >> s_hi) & 0x03030303u) << 4);
      const int g = u >> 2;
      fma2h(acc[g][0], acc[g][1], xr[4 * u + 0], lo6 & 0x003F003Fu);
      fma2h(acc[g][0], acc[g][1], xr[4 * u + 1], (lo6 >> 8) & 0x003F003Fu);
      fma2h(acc[2 + g][0], acc[2 + g][1], xr[4 * u + 2], hi6 & 0x003F003Fu);
      fma2h(acc[2 + g][0], acc[2 + g][1], xr[4 * u + 3], (hi6 >> 8) & 0x003F003Fu);
    }
    const int8_t* sc = reinterpret_cast<const int8_t*>(blk + 192 + 8 * H + 2 * rr);
    const float d = h2f(ld_u16(blk + 208));
    float r = 0.f;
    const int si[4] = {0, 1, 4, 5};
#pragma unroll
    for (int g = 0; g < 4; ++g)
      r = fmaf(static_cast<float>(sc[si[g]]), (acc[g][0] + acc[g][1]) - xs[g], r);
    return d * r * kTwo24;
  }
};

// ------------------------------------------------------------------------------- Q8_0
// A superblock is eight 34-byte blocks; lane piece c = blocks 2c and 2c+1.  Signed bytes
// are biased to unsigned (q + 128) in the mask itself and the bias is removed with the
// block's activation sum.  Register k of block e holds x pairs (t, t+2) / (t+1, t+3).
struct DecQ80 {
  static constexpr int kSB = 272, kSB2 = 0;
  static constexpr bool kBf16X = false;
  uint32_t xr[32];
  float xs[4];  // 128 * 2^-24 * sum of block 2c / 2c+1 activations
  int c;

  __device__ __forceinline__ static int run0(int c) { return 64 * c; }
  __device__ __forceinline__ static int run1(int c) { return 64 * c + 32; }
  __device__ __forceinline__ static constexpr int xloc(int k, int h) { return 32 * (k >> 4) + 4 * ((k >> 1) & 7) + (k & 1) + 2 * h; }
  __device__ __forceinline__ static constexpr int xsum(int k, int) { return k >> 4; }
  __device__ __forceinline__ static float xsum_scale() { return 128.0f / kTwo24; }
  __device__ __forceinline__ void init(int c_) { c = c_; }
  __device__ __forceinline__ void load_x(const uint16_t* __restrict__ x, int64_t sb, int c_, bool active) {
    load_x_f16(*this, x, sb, c_, active);
  }

  __device__ __forceinline__ float row(const uint8_t* sblk, const uint8_t*) const {
    float r = 0.f;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint8_t* blk = sblk + 34 * (2 * c + e);
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t wd = ld_u32_a2(blk + 2 + 4 * u) ^ 0x80808080u;
        fma2h(a0, a1, xr[16 * e + 2 * u], wd & 0x00FF00FFu);
        fma2h(a2, a3, xr[16 * e + 2 * u + 1], (wd >> 8) & 0x00FF00FFu);
      }
      const float d = h2f(ld_u16(blk));
      r = fmaf(d, ((a0 + a1) + (a2 + a3)) - xs[e], r);
    }
    return r * kTwo24;
  }
};

// ------------------------------------------------------------------------------- NVFP4
// Superblock = 256 elements: 128 nibble bytes (stream 1) and 16 E4M3 scales (stream 2).
// Lane piece c = nibble bytes [32c, 32c+32) and scales [4c, 4c+4); register k holds the
// activations of nibble byte k (elements 2k, 2k+1: low nibble = even element).  E2M1 and
// E4M3 are decoded by the hardware conversions to f16 (exact for every code).  The bf16
// activations are staged as f16 times a power of two chosen per CTA from max |x|, so the
// f16 x E2M1 products stay exact; the power of two is removed from the result.
struct DecNVFP4 {
  static constexpr int kSB = 128, kSB2 = 16;
  static constexpr bool kBf16X = true;
  uint32_t xr[32];
  float xs[4];
  int c;

  float inv_scale;  // the activations are held as f16(x * 2^e); partial sums are scaled back

  __device__ __forceinline__ void init(int c_) { c = c_; }
  // bf16 activations of the lane's 64 elements as f16 pairs, times one power of two chosen
  // from their largest magnitude so that every value is below 2^14 and f16 holds it exactly
  // (values 2^28 times smaller than the largest lose low bits).
  __device__ __forceinline__ void load_x(const uint16_t* __restrict__ x, int64_t sb, int c_, bool active) {
    uint32_t v[32];
    load_runs(x, sb * 256 + 64 * c_, sb * 256 + 64 * c_ + 32, active, v);
    float mx = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fmaxf(fabsf(bf2f(v[i])), fabsf(bf2f(v[i] >> 16))));
    float scale = 1.0f;
    if (mx > 0.f && mx < 3.0e38f) {
      const int e = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFF) - 127 + 1;  // 2^(e-1) <= mx < 2^e
      scale = p2(max(-126, min(127, 14 - e)));
    }
    inv_scale = 1.0f / scale;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const __half2 h2 = __floats2half2_rn(bf2f(v[k]) * scale, bf2f(v[k] >> 16) * scale);
      xr[k] = *reinterpret_cast<const uint32_t*>(&h2);
    }
  }

  __device__ __forceinline__ static uint32_t e2m1x2(uint32_t byte) {
    uint32_t h;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h) : "r"(byte));
    return h;
  }
  __device__ __forceinline__ static uint32_t e4m3x2(uint32_t two) {
    uint32_t h;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h) : "r"(two));
    return h;
  }

  __device__ __forceinline__ float row(const uint8_t* nib, const uint8_t* sc) const {
    const uint4 q0 = *reinterpret_cast<const uint4*>(nib + 32 * c);
    const uint4 q1 = *reinterpret_cast<const uint4*>(nib + 32 * c + 16);
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const uint32_t s4 = *reinterpret_cast<const uint32_t*>(sc + 4 * c) & 0x7F7F7F7Fu;  // |scale|
    float r = 0.f;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t wd = w[2 * b + u];
        fma2h(a0, a1, xr[8 * b + 4 * u + 0], e2m1x2(wd & 0xFFu));
        fma2h(a2, a3, xr[8 * b + 4 * u + 1], e2m1x2((wd >> 8) & 0xFFu));
        fma2h(a0, a1, xr[8 * b + 4 * u + 2], e2m1x2((wd >> 16) & 0xFFu));
        fma2h(a2, a3, xr[8 * b + 4 * u + 3], e2m1x2(wd >> 24));
      }
      const float sv = h2f(e4m3x2((s4 >> (8 * b)) & 0xFFu));
      r = fmaf(sv, (a0 + a1) + (a2 + a3), r);
    }
    return r * inv_scale;
  }
};

// ------------------------------------------------------------------------------- TQ1_0
// Lane piece c = payload bytes [13c, 13c+13) of qs[48] ++ qh[4].  For a byte b whose
// digits n = 0..4 weigh activations y_0..y_4: sum_n y_n t_n(b) = sum_{k=1..5} g_k F_k(b)
// with F_k(b) = floor(3^k b / 256), g_k = y_{k-1} - 3 y_k, y_5 = 0; qh bytes carry four
// digits, so their y_4 is 0 ("metal: TQ1_0 kernel performance", section 1).  F_k is one
// round-toward-minus-infinity FMA: 2^23 + b * 3^k / 256 rounded down is 2^23 + F_k.  The
// 65 coefficients g of a lane piece are staged in shared memory as fp32.
struct DecTQ10 {
  static constexpr int kSB = 54, kSB2 = 0;
  float g[13][5];
  float xsum;
  int c;

  __device__ __forceinline__ static int elem_of(int p, int n) {
    if (p < 32) return 32 * n + p;
    if (p < 48) return 160 + 16 * n + (p - 32);
    return 240 + 4 * n + (p - 48);
  }
  __device__ __forceinline__ void init(int c_) { c = c_; }
  __device__ __forceinline__ void load_x(const uint16_t* __restrict__ x, int64_t sb, int c_, bool active) {
    xsum = 0.f;
#pragma unroll
    for (int i = 0; i < 13; ++i) {
      const int p = 13 * c_ + i;
      float y[6];
#pragma unroll
      for (int n = 0; n < 5; ++n) {
        const bool has = active && !(p >= 48 && n == 4);
        y[n] = has ? h2f(__ldg(x + sb * 256 + elem_of(p, n))) : 0.f;
        xsum += y[n];
      }
      y[5] = 0.f;
#pragma unroll
      for (int k = 1; k <= 5; ++k) g[i][k - 1] = y[k - 1] - 3.f * y[k];
    }
  }

  __device__ __forceinline__ float row(const uint8_t* blk, const uint8_t*) const {
    constexpr float kMagic = 8388608.0f;  // 2^23
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int i = 0; i < 13; ++i) {
      const float b = static_cast<float>(blk[13 * c + i]);
      float& a = (i & 1) ? a1 : a0;
      a = fmaf(g[i][0], __fmaf_rd(b, 3.f / 256.f, kMagic) - kMagic, a);
      a = fmaf(g[i][1], __fmaf_rd(b, 9.f / 256.f, kMagic) - kMagic, a);
      a = fmaf(g[i][2], __fmaf_rd(b, 27.f / 256.f, kMagic) - kMagic, a);
      a = fmaf(g[i][3], __fmaf_rd(b, 81.f / 256.f, kMagic) - kMagic, a);
      a = fmaf(g[i][4], __fmaf_rd(b, 243.f / 256.f, kMagic) - kMagic, a);
    }
    const float d = h2f(ld_u16(blk + 52));
    return d * ((a0 + a1) - xsum);
  }
};

}  // namespace qg
