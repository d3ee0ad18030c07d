// Plain kernels of the qgemv library.
//
//  rowwarp_kernel<F>  path for shapes the streaming kernel does not take (rows that do not
//                     start on 16 bytes, K not a multiple of 256, very long K): one warp per
//                     row, byte loads, the dequantisation formula evaluated weight by weight
//                     in fp32.
//  unpack_kernel<F>   codes / scales / mins of every weight (bit-exact debug view).
#pragma once
#include <cuda_fp16.h>

#include <cstdint>

#include "qgemv_decode.cuh"
#include "qgemv_epilogue.cuh"
#include "qgemv_ptx.cuh"

namespace qg {

// ------------------------------------------------------------------ plain per-row path
struct RowArgs {
  const uint8_t* W;
  const uint16_t* x;
  void* y;
  int64_t N, K;
  // Epilogue (see emit_out): y[n] = alpha r + beta y[n] as ydt; with pair = 1, r =
  // silu(row n of W . x) * (row n of WB . x).  The plain GEMV uses 1, 0, fp32, no pair.
  float alpha, beta;
  int ydt, pair;
  const uint8_t* WB;
};

__device__ __forceinline__ void kq_scale_min(const uint8_t* S, int g, int& s, int& m) {
  if (g < 4) {
    s = S[g] & 63;
    m = S[g + 4] & 63;
  } else {
    s = (S[g + 4] & 0x0F) | ((S[g - 4] >> 6) << 4);
    m = (S[g + 4] >> 4) | ((S[g] >> 6) << 4);
  }
}

__device__ __forceinline__ int tq1_digit(uint32_t b, int n) {
  uint32_t p = 1;
  for (int i = 0; i < n; ++i) p *= 3;
  return static_cast<int>((3 * p * b) / 256 - 3 * ((p * b) / 256));
}

__device__ __forceinline__ float e2m1_f(uint32_t code) {
  const uint32_t m = code & 7u;
  const float v = (m < 2) ? 0.5f * m : static_cast<float>((2u | (m & 1u)) << ((m >> 1) - 1)) * 0.5f;
  return (code & 8u) ? -v : v;
}

__device__ __forceinline__ float e4m3_f(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  float v;
  if (e == 15u && m == 7u)
    v = __int_as_float(0x7fc00000);
  else if (e == 0u)
    v = static_cast<float>(m) * p2(-9);
  else
    v = static_cast<float>(8u | m) * p2(static_cast<int>(e) - 10);
  return (b & 0x80u) ? -v : v;
}

// Code, scale and min of element i of block p so that w = scale * code - min exactly in fp32.
template <int F>
__device__ __forceinline__ void elem_code(const uint8_t* p, int i, int& code, float& scale, float& mn) {
  if constexpr (F == F_Q4K || F == F_Q5K) {
    const int c = i >> 6, h = (i >> 5) & 1, j = i & 31, g = i >> 5;
    int s, m;
    kq_scale_min(p + 4, g, s, m);
    if constexpr (F == F_Q4K) {
      code = (p[16 + 32 * c + j] >> (4 * h)) & 15;
    } else {
      code = ((p[48 + 32 * c + j] >> (4 * h)) & 15) | (((p[16 + j] >> (2 * c + h)) & 1) << 4);
    }
    scale = h2f(p[0] | (p[1] << 8)) * static_cast<float>(s);
    mn = h2f(p[2] | (p[3] << 8)) * static_cast<float>(m);
  } else if constexpr (F == F_Q6K) {
    const int H = i >> 7, r = (i & 127) >> 5, l = i & 31;
    const int lo = (p[64 * H + l + 32 * (r & 1)] >> (4 * (r >> 1))) & 15;
    const int hi = (p[128 + 32 * H + l] >> (2 * r)) & 3;
    code = (lo | (hi << 4)) - 32;
    scale = h2f(p[208] | (p[209] << 8)) * static_cast<float>(static_cast<int8_t>(p[192 + 8 * H + 2 * r + l / 16]));
    mn = 0.f;
  } else if constexpr (F == F_Q80) {
    code = static_cast<int8_t>(p[2 + i]);
    scale = h2f(p[0] | (p[1] << 8));
    mn = 0.f;
  } else if constexpr (F == F_TQ10) {
    int t;
    if (i < 160)
      t = tq1_digit(p[i & 31], i >> 5);
    else if (i < 240)
      t = tq1_digit(p[32 + ((i - 160) & 15)], (i - 160) >> 4);
    else
      t = tq1_digit(p[48 + ((i - 240) & 3)], (i - 240) >> 2);
    code = t - 1;
    scale = h2f(p[52] | (p[53] << 8));
    mn = 0.f;
  }
}

template <int F>
struct FmtGeom;
template <> struct FmtGeom<F_Q4K> { static constexpr int BW = 256, BB = 144; };
template <> struct FmtGeom<F_Q5K> { static constexpr int BW = 256, BB = 176; };
template <> struct FmtGeom<F_Q6K> { static constexpr int BW = 256, BB = 210; };
template <> struct FmtGeom<F_Q80> { static constexpr int BW = 32, BB = 34; };
template <> struct FmtGeom<F_TQ10> { static constexpr int BW = 256, BB = 54; };
template <> struct FmtGeom<F_NVFP4> { static constexpr int BW = 16, BB = 8; };  // stream-1 bytes

// Row n of matrix W (N x K) dotted with x by one warp; every lane returns the total.
template <int F>
__device__ float row_dot(const uint8_t* W, const RowArgs& a, int64_t n, int lane) {
  constexpr int BW = FmtGeom<F>::BW, BB = FmtGeom<F>::BB;
  const int64_t nb = a.K / BW;
  float acc = 0.f;
  for (int64_t b = lane; b < nb; b += 32) {
    if constexpr (F == F_NVFP4) {
      const uint8_t* nib = W + n * (a.K / 2) + b * 8;
      const float s = fabsf(e4m3_f(W[a.N * (a.K / 2) + n * (a.K / 16) + b]));
      float part = 0.f;
      for (int j = 0; j < 16; ++j) {
        const uint32_t code = (nib[j >> 1] >> (4 * (j & 1))) & 15u;
        part = fmaf(bf2f(a.x[b * 16 + j]), e2m1_f(code) * s, part);
      }
      acc += part;
    } else {
      const uint8_t* p = W + (n * nb + b) * BB;
      for (int i = 0; i < BW; ++i) {
        int code;
        float scale, mn;
        elem_code<F>(p, i, code, scale, mn);
        const float w = fmaf(scale, static_cast<float>(code), -mn);
        acc = fmaf(h2f(a.x[b * BW + i]), w, acc);
      }
    }
  }
  return warp_sum(acc);
}

template <int F>
__global__ void __launch_bounds__(256) rowwarp_kernel(const RowArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t n = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); n < a.N; n += warps) {
    float r = row_dot<F>(a.W, a, n, lane);
    if (a.pair) r = silu_f(r) * row_dot<F>(a.WB, a, n, lane);
    if (lane == 0) emit_out(a.y, a.ydt, a.alpha, a.beta, n, r);
  }
}

// ------------------------------------------------------------------ unpack (debug)
struct UnpackArgs {
  const uint8_t* W;
  int8_t* codes;
  float* scales;
  float* mins;  // may be null
  int64_t N, K;
  int G;  // group length of scales / mins
};

// One thread per (row, group of G elements).
template <int F>
__global__ void __launch_bounds__(256) unpack_kernel(const UnpackArgs a) {
  const int64_t ng = a.K / a.G;
  const int64_t total = a.N * ng;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t n = t / ng, g = t % ng;
    const int64_t k0 = g * a.G;
    float scale = 0.f, mn = 0.f;
    if constexpr (F == F_NVFP4) {
      const uint8_t* nib = a.W + n * (a.K / 2);
      const uint32_t sb = a.W[a.N * (a.K / 2) + n * (a.K / 16) + g];
      const uint32_t sh = DecNVFP4::e4m3x2(sb);
      scale = fabsf(__half22float2(*reinterpret_cast<const __half2*>(&sh)).x) * 0.5f;
      for (int j = 0; j < 16; j += 2) {
        const uint32_t eh = DecNVFP4::e2m1x2(nib[(k0 + j) >> 1]);
        const float2 e = __half22float2(*reinterpret_cast<const __half2*>(&eh));
        a.codes[n * a.K + k0 + j] = static_cast<int8_t>(__float2int_rn(2.f * e.x));
        a.codes[n * a.K + k0 + j + 1] = static_cast<int8_t>(__float2int_rn(2.f * e.y));
      }
    } else {
      constexpr int BW = FmtGeom<F>::BW, BB = FmtGeom<F>::BB;
      for (int j = 0; j < a.G; ++j) {
        const int64_t k = k0 + j;
        const uint8_t* p = a.W + (n * (a.K / BW) + k / BW) * BB;
        int code;
        float s, m;
        elem_code<F>(p, static_cast<int>(k % BW), code, s, m);
        a.codes[n * a.K + k] = static_cast<int8_t>(code);
        if (j == 0) {
          scale = s;
          mn = m;
        }
      }
    }
    a.scales[t] = scale;
    if (a.mins) a.mins[t] = mn;
  }
}

}  // namespace qg
