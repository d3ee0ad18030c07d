// Per-format register decoders for the streaming GEMV kernel.
//
// Work split (all formats): a row is cut into 256-element "superblocks" (one Q4_K / Q5_K /
// Q6_K / TQ1_0 block, eight Q8_0 blocks, or 256 NVFP4 elements with their 16 scales).
// Four lanes share a superblock and each lane owns a fixed 64-element piece of it, so the
// activations a lane needs never change while it walks down the rows: they are loaded
// once, pre-transformed, and kept in registers (`xs`).
//
// Exact nibble/byte -> float decode without shifts or int->float conversions: for a
// 32-bit word w and a field mask covering bits [p, p+n) with p+n <= 24, the float whose
// bit pattern is (w & mask) equals field * 2^(p-149) exactly (a subnormal or the smallest
// binade, both linear in the bit pattern; FFMA keeps subnormal inputs, nothing here is
// built with flush-to-zero).  The activation that multiplies the field is pre-scaled by
// 2^(149-p-64) so every product is field * x * 2^-64 exactly, and the block scale is
// multiplied by 2^64 once per block.  Fields in the top byte of a word are first moved
// down by 8 bits (one shift per word).  This is the GPU form of the "multiply by the
// masked but unshifted nibble and correct once at the end" idea of the Q4_K page
// (section "Compute").
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
__device__ __forceinline__ float fbits(uint32_t b) { return __uint_as_float(b); }

// Power-of-two float from its unbiased exponent (normal range).
__device__ __forceinline__ float p2(int e) { return __uint_as_float(static_cast<uint32_t>(e + 127) << 23); }

__device__ __forceinline__ uint32_t ld_u16(const uint8_t* p) { return *reinterpret_cast<const uint16_t*>(p); }
// 32-bit little-endian load from a 2-byte aligned shared/global address.
__device__ __forceinline__ uint32_t ld_u32_a2(const uint8_t* p) { return ld_u16(p) | (ld_u16(p + 2) << 16); }

// Pre-scale exponent for a field whose lowest bit sits at bit `pos` of the word it is
// decoded from (after the optional 8-bit shift): x * 2^(85 - pos) * field * 2^(pos-149)
// = x * field * 2^-64.
__device__ __forceinline__ float xscale(int pos) { return p2(85 - pos); }
constexpr float kTwo64 = 18446744073709551616.0f;

// Loads the NV fp16 activations x[base .. base+NV-1] (base a multiple of 8) as floats.
template <int NV>
__device__ __forceinline__ void load_x_f16(const uint16_t* __restrict__ x, int64_t base, float (&v)[NV]) {
  const uint4* p = reinterpret_cast<const uint4*>(x + base);
#pragma unroll
  for (int i = 0; i < NV / 8; ++i) {
    const uint4 q = __ldg(p + i);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * i + 2 * j] = h2f(w[j]);
      v[8 * i + 2 * j + 1] = h2f(w[j] >> 16);
    }
  }
}

// ------------------------------------------------------------------------------- Q4_K
// Lane piece c (0..3) = quant bytes [32c, 32c+32) of the block: low nibbles are elements
// 64c + t (group 2c), high nibbles 64c + 32 + t (group 2c+1), t = 0..31.
struct DecQ4K {
  static constexpr int kSB = 144;   // bytes per superblock (stream 1)
  static constexpr int kSB2 = 0;    // bytes per superblock (stream 2)
  float xs[64];                     // xs[2t] low-nibble activation of byte t, xs[2t+1] high
  float xlo, xhi;                   // plain sums of the low / high activations
  int c;

  __device__ __forceinline__ void load_x(const uint16_t* __restrict__ x, int64_t sb, int c_, bool active) {
    c = c_;
    xlo = xhi = 0.f;
    float v[64];
    if (active) {
      load_x_f16<64>(x, sb * 256 + 64 * c, v);
    } else {
#pragma unroll
      for (int j = 0; j < 64; ++j) v[j] = 0.f;
    }
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      const int b = t & 3;
      const int plo = (b == 3) ? 16 : 8 * b;  // bit position of the low nibble after the shift
      xs[2 * t] = v[t] * xscale(plo);
      xs[2 * t + 1] = v[32 + t] * xscale(plo + 4);
      xlo += v[t];
      xhi += v[32 + t];
    }
  }

  // Partial dot of this lane's 64 weights of one block with its activations.
  __device__ __forceinline__ float row(const uint8_t* blk, const uint8_t*) const {
    const uint4 h = *reinterpret_cast<const uint4*>(blk);
    const uint4 q0 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
    const uint4 q1 = *reinterpret_cast<const uint4*>(blk + 32 + 32 * c);
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t wd = w[u], ws = wd >> 8;
      float& al = (u & 1) ? a1 : a0;
      float& ah = (u & 1) ? b1 : b0;
      const int t = 4 * u;
      al = fmaf(xs[2 * t + 0], fbits(wd & 0x0000000Fu), al);
      ah = fmaf(xs[2 * t + 1], fbits(wd & 0x000000F0u), ah);
      al = fmaf(xs[2 * t + 2], fbits(wd & 0x00000F00u), al);
      ah = fmaf(xs[2 * t + 3], fbits(wd & 0x0000F000u), ah);
      al = fmaf(xs[2 * t + 4], fbits(wd & 0x000F0000u), al);
      ah = fmaf(xs[2 * t + 5], fbits(wd & 0x00F00000u), ah);
      al = fmaf(xs[2 * t + 6], fbits(ws & 0x000F0000u), al);
      ah = fmaf(xs[2 * t + 7], fbits(ws & 0x00F00000u), ah);
    }
    const float acc_lo = a0 + a1, acc_hi = b0 + b1;
    // 6-bit scales / mins of groups 2c, 2c+1 (packed layout of the block's 12 scale bytes:
    // groups 0..3 low 6 bits of bytes 0..3 / 4..7; groups 4..7 nibbles of bytes 8..11 plus
    // the top two bits of bytes 0..3 / 4..7).
    const uint32_t sw_a = h.y & 0x3F3F3F3Fu, mw_a = h.z & 0x3F3F3F3Fu;
    const uint32_t sw_b = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
    const uint32_t mw_b = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
    const uint32_t sw = (c < 2) ? sw_a : sw_b, mw = (c < 2) ? mw_a : mw_b;
    const int sh = (c & 1) * 16;
    const float s_lo = static_cast<float>((sw >> sh) & 0xFFu), s_hi = static_cast<float>((sw >> (sh + 8)) & 0xFFu);
    const float m_lo = static_cast<float>((mw >> sh) & 0xFFu), m_hi = static_cast<float>((mw >> (sh + 8)) & 0xFFu);
    const float d = h2f(h.x) * kTwo64, dmin = h2f(h.x >> 16);
    return fmaf(d, fmaf(s_lo, acc_lo, s_hi * acc_hi), -dmin * fmaf(m_lo, xlo, m_hi * xhi));
  }
};

// ------------------------------------------------------------------------------- Q5_K
// Same piece split as Q4_K (quants at byte 48); the fifth bit of element j of chunk c
// (low / high nibble) is bit 2c / 2c+1 of qh[j].  Its contribution 16*x is accumulated
// from the same pre-scaled activations through the bit's own float value, which differs
// from the nibble's scale by the lane constant 2^(4-2c) (low) or 2^(7-2c) (high).
struct DecQ5K {
  static constexpr int kSB = 176;
  static constexpr int kSB2 = 0;
  DecQ4K q4;  // activations and lane constants are the same as Q4_K's

  __device__ __forceinline__ void load_x(const uint16_t* __restrict__ x, int64_t sb, int c_, bool active) {
    q4.load_x(x, sb, c_, active);
  }

  __device__ __forceinline__ float row(const uint8_t* blk, const uint8_t*) const {
    const int c = q4.c;
    const uint4 h = *reinterpret_cast<const uint4*>(blk);
    const uint4 e0 = *reinterpret_cast<const uint4*>(blk + 16);
    const uint4 e1 = *reinterpret_cast<const uint4*>(blk + 32);
    const uint4 q0 = *reinterpret_cast<const uint4*>(blk + 48 + 32 * c);
    const uint4 q1 = *reinterpret_cast<const uint4*>(blk + 64 + 32 * c);
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const uint32_t e[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
    const uint32_t m0 = 1u << (2 * c), m1 = m0 << 8, m2 = m0 << 16;
    float al = 0.f, ah = 0.f, el = 0.f, eh = 0.f;
    const float* xs = q4.xs;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t wd = w[u], ws = wd >> 8, ed = e[u], es = ed >> 8;
      const int t = 4 * u;
      al = fmaf(xs[2 * t + 0], fbits(wd & 0x0000000Fu), al);
      ah = fmaf(xs[2 * t + 1], fbits(wd & 0x000000F0u), ah);
      al = fmaf(xs[2 * t + 2], fbits(wd & 0x00000F00u), al);
      ah = fmaf(xs[2 * t + 3], fbits(wd & 0x0000F000u), ah);
      al = fmaf(xs[2 * t + 4], fbits(wd & 0x000F0000u), al);
      ah = fmaf(xs[2 * t + 5], fbits(wd & 0x00F00000u), ah);
      al = fmaf(xs[2 * t + 6], fbits(ws & 0x000F0000u), al);
      ah = fmaf(xs[2 * t + 7], fbits(ws & 0x00F00000u), ah);
      el = fmaf(xs[2 * t + 0], fbits(ed & m0), el);
      eh = fmaf(xs[2 * t + 1], fbits(ed & (m0 << 1)), eh);
      el = fmaf(xs[2 * t + 2], fbits(ed & m1), el);
      eh = fmaf(xs[2 * t + 3], fbits(ed & (m1 << 1)), eh);
      el = fmaf(xs[2 * t + 4], fbits(ed & m2), el);
      eh = fmaf(xs[2 * t + 5], fbits(ed & (m2 << 1)), eh);
      el = fmaf(xs[2 * t + 6], fbits(es & m2), el);
      eh = fmaf(xs[2 * t + 7], fbits(es & (m2 << 1)), eh);
    }
    const float acc_lo = fmaf(p2(4 - 2 * c), el, al), acc_hi = fmaf(p2(7 - 2 * c), eh, ah);
    const uint32_t sw_a = h.y & 0x3F3F3F3Fu, mw_a = h.z & 0x3F3F3F3Fu;
    const uint32_t sw_b = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
    const uint32_t mw_b = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
    const uint32_t sw = (c < 2) ? sw_a : sw_b, mw = (c < 2) ? mw_a : mw_b;
    const int sh = (c & 1) * 16;
    const float s_lo = static_cast<float>((sw >> sh) & 0xFFu), s_hi = static_cast<float>((sw >> (sh + 8)) & 0xFFu);
    const float m_lo = static_cast<float>((mw >> sh) & 0xFFu), m_hi = static_cast<float>((mw >> (sh + 8)) & 0xFFu);
    const float d = h2f(h.x) * kTwo64, dmin = h2f(h.x >> 16);
    return fmaf(d, fmaf(s_lo, acc_lo, s_hi * acc_hi), -dmin * fmaf(m_lo, q4.xlo, m_hi * q4.xhi));
  }
};

// ------------------------------------------------------------------------------- Q6_K
// Lane piece c: half H = c>>1, rr = c&1.  Bytes ql[64H + 32rr + t] hold, in their low
// nibble, element 128H + 32rr + t and, in their high nibble, element 128H + 32(rr+2) + t;
// the top two bits come from qh[32H + t] bits 2rr / 2rr+4.  Blocks are 210 bytes, so
// loads are 16-bit.  Weight = d * sc * (q - 32); the -32 uses per-group activation sums.
struct DecQ6K {
  static constexpr int kSB = 210;
  static constexpr int kSB2 = 0;
  float xs[64];  // xs[2t] low-nibble element of byte t, xs[2t+1] high
  float xg[4];   // activation sums of the 4 scale groups: lo t<16, lo t>=16, hi t<16, hi t>=16
  int c;

  __device__ __forceinline__ void load_x(const uint16_t* __restrict__ x, int64_t sb, int c_, bool active) {
    c = c_;
    const int H = c >> 1, rr = c & 1;
    float lo[32], hi[32];
    if (active) {
      load_x_f16<32>(x, sb * 256 + 128 * H + 32 * rr, lo);
      load_x_f16<32>(x, sb * 256 + 128 * H + 32 * (rr + 2), hi);
    } else {
#pragma unroll
      for (int t = 0; t < 32; ++t) lo[t] = hi[t] = 0.f;
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) xg[g] = 0.f;
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      const int b = t & 3;
      const int pos = (b == 3) ? 16 : 8 * b;
      xs[2 * t] = lo[t] * xscale(pos);
      xs[2 * t + 1] = hi[t] * xscale(pos);
      xg[t >> 4] += lo[t];
      xg[2 + (t >> 4)] += hi[t];
    }
  }

  __device__ __forceinline__ float row(const uint8_t* blk, const uint8_t*) const {
    const int H = c >> 1, rr = c & 1;
    const uint8_t* ql = blk + 64 * H + 32 * rr;
    const uint8_t* qh = blk + 128 + 32 * H;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t l = ld_u32_a2(ql + 4 * u), e = ld_u32_a2(qh + 4 * u);
      const uint32_t lo6 = (l & 0x0F0F0F0Fu) | (((e >> (2 * rr)) & 0x03030303u) << 4);
      const uint32_t hi6 = ((l >> 4) & 0x0F0F0F0Fu) | (((e >> (2 * rr + 4)) & 0x03030303u) << 4);
      const uint32_t los = lo6 >> 8, his = hi6 >> 8;
      const int t = 4 * u;
      float& al = acc[u >> 2];
      float& ah = acc[2 + (u >> 2)];
      al = fmaf(xs[2 * t + 0], fbits(lo6 & 0x0000003Fu), al);
      ah = fmaf(xs[2 * t + 1], fbits(hi6 & 0x0000003Fu), ah);
      al = fmaf(xs[2 * t + 2], fbits(lo6 & 0x00003F00u), al);
      ah = fmaf(xs[2 * t + 3], fbits(hi6 & 0x00003F00u), ah);
      al = fmaf(xs[2 * t + 4], fbits(lo6 & 0x003F0000u), al);
      ah = fmaf(xs[2 * t + 5], fbits(hi6 & 0x003F0000u), ah);
      al = fmaf(xs[2 * t + 6], fbits(los & 0x003F0000u), al);
      ah = fmaf(xs[2 * t + 7], fbits(his & 0x003F0000u), ah);
    }
    const int8_t* sc = reinterpret_cast<const int8_t*>(blk + 192 + 8 * H + 2 * rr);
    const float d = h2f(ld_u16(blk + 208));
    float r = 0.f;
    r = fmaf(static_cast<float>(sc[0]), fmaf(kTwo64, acc[0], -32.f * xg[0]), r);
    r = fmaf(static_cast<float>(sc[1]), fmaf(kTwo64, acc[1], -32.f * xg[1]), r);
    r = fmaf(static_cast<float>(sc[4]), fmaf(kTwo64, acc[2], -32.f * xg[2]), r);
    r = fmaf(static_cast<float>(sc[5]), fmaf(kTwo64, acc[3], -32.f * xg[3]), r);
    return d * r;
  }
};

// ------------------------------------------------------------------------------- Q8_0
// A superblock is eight 34-byte blocks; lane piece c = blocks 2c and 2c+1.  Signed bytes
// are biased to unsigned (q + 128) so they decode with the same masks; the bias is removed
// with the block's activation sum.
struct DecQ80 {
  static constexpr int kSB = 272;
  static constexpr int kSB2 = 0;
  float xs[64];  // xs[32e + j], block e in {0,1}, element j
  float xb[2];
  int c;

  __device__ __forceinline__ void load_x(const uint16_t* __restrict__ x, int64_t sb, int c_, bool active) {
    c = c_;
    float v[64];
    if (active) {
      load_x_f16<64>(x, sb * 256 + 64 * c, v);
    } else {
#pragma unroll
      for (int j = 0; j < 64; ++j) v[j] = 0.f;
    }
    xb[0] = xb[1] = 0.f;
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      const int b = j & 3;
      xs[j] = v[j] * xscale(b == 3 ? 16 : 8 * b);
      xb[j >> 5] += v[j];
    }
  }

  __device__ __forceinline__ float row(const uint8_t* sblk, const uint8_t*) const {
    float r = 0.f;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint8_t* blk = sblk + 34 * (2 * c + e);
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t wd = ld_u32_a2(blk + 2 + 4 * u) ^ 0x80808080u, ws = wd >> 8;
        const float* xx = xs + 32 * e + 4 * u;
        float& a = (u & 1) ? a1 : a0;
        a = fmaf(xx[0], fbits(wd & 0x000000FFu), a);
        a = fmaf(xx[1], fbits(wd & 0x0000FF00u), a);
        a = fmaf(xx[2], fbits(wd & 0x00FF0000u), a);
        a = fmaf(xx[3], fbits(ws & 0x00FF0000u), a);
      }
      const float d = h2f(ld_u16(blk));
      r = fmaf(d, fmaf(kTwo64, a0 + a1, -128.f * xb[e]), r);
    }
    return r;
  }
};

// ------------------------------------------------------------------------------- TQ1_0
// Lane piece c = payload bytes [13c, 13c+13) of qs[48] ++ qh[4].  For a byte b whose
// digits n = 0..4 weigh activations y_0..y_4, sum_n y_n t_n(b) = sum_{k=1..5} g_k F_k(b)
// with F_k(b) = floor(3^k b / 256), g_k = y_{k-1} - 3 y_k, y_5 = 0; qh bytes carry four
// digits, so their y_4 is 0 ("metal: TQ1_0 kernel performance", section 1).  F_k is one
// round-toward-minus-infinity FMA: 2^23 + b * 3^k / 256 rounded down is 2^23 + F_k.
struct DecTQ10 {
  static constexpr int kSB = 54;
  static constexpr int kSB2 = 0;
  float g[13][5];
  float xsum;
  int c;

  __device__ __forceinline__ static int elem_of(int p, int n) {
    if (p < 32) return 32 * n + p;
    if (p < 48) return 160 + 16 * n + (p - 32);
    return 240 + 4 * n + (p - 48);
  }

  __device__ __forceinline__ void load_x(const uint16_t* __restrict__ x, int64_t sb, int c_, bool active) {
    c = c_;
    xsum = 0.f;
#pragma unroll
    for (int i = 0; i < 13; ++i) {
      const int p = 13 * c + i;
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

// ------------------------------------------------------------------------------- NVFP4
// Superblock = 256 elements: 128 nibble bytes (stream 1) and 16 E4M3 scales (stream 2).
// Lane piece c = nibble bytes [32c, 32c+32) (elements 64c..64c+63, low nibble = even
// element) and scales [4c, 4c+4).  E2M1 and E4M3 decode through the hardware conversions
// to f16 (exact for every code), products and sums in fp32, the |scale| applied once per
// 16-element block (Mojo fp4_gemv page, "Structure").
struct DecNVFP4 {
  static constexpr int kSB = 128;
  static constexpr int kSB2 = 16;
  float xs[64];
  int c;

  __device__ __forceinline__ void load_x(const uint16_t* __restrict__ x, int64_t sb, int c_, bool active) {
    c = c_;
    if (active) {
      const uint4* p = reinterpret_cast<const uint4*>(x + sb * 256 + 64 * c);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 q = __ldg(p + i);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          xs[8 * i + 2 * j] = bf2f(w[j]);
          xs[8 * i + 2 * j + 1] = bf2f(w[j] >> 16);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 64; ++j) xs[j] = 0.f;
    }
  }

  __device__ __forceinline__ static float2 e2m1x2(uint32_t byte) {
    uint32_t h;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h) : "r"(byte));
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
  }
  __device__ __forceinline__ static float2 e4m3x2(uint32_t two) {
    uint32_t h;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h) : "r"(two));
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
  }

  __device__ __forceinline__ float row(const uint8_t* nib, const uint8_t* sc) const {
    const uint4 q0 = *reinterpret_cast<const uint4*>(nib + 32 * c);
    const uint4 q1 = *reinterpret_cast<const uint4*>(nib + 32 * c + 16);
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const uint32_t s4 = *reinterpret_cast<const uint32_t*>(sc + 4 * c);
    const float2 s01 = e4m3x2(s4 & 0xFFFFu), s23 = e4m3x2(s4 >> 16);
    const float s[4] = {fabsf(s01.x), fabsf(s01.y), fabsf(s23.x), fabsf(s23.y)};
    float r = 0.f;
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t wd = w[2 * blk + u];
#pragma unroll
        for (int by = 0; by < 4; ++by) {
          const float2 e = e2m1x2((wd >> (8 * by)) & 0xFFu);
          const int j = 16 * blk + 8 * u + 2 * by;
          a0 = fmaf(xs[j], e.x, a0);
          a1 = fmaf(xs[j + 1], e.y, a1);
        }
      }
      r = fmaf(s[blk], a0 + a1, r);
    }
    return r;
  }
};

}  // namespace qg
