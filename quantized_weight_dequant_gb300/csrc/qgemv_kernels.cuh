// Kernels of the qgemv library.
//
//  stream_kernel<Dec>  the main path: per-warp rings of 1-D bulk copies (global -> shared,
//                      mbarrier completion) stream the packed rows once; lanes decode from
//                      shared memory into registers against activations held in registers.
//  rowwarp_kernel<F>   plain path for shapes the bulk copies cannot take (rows that do not
//                      start on 16 bytes, K not a multiple of 256): one warp per row, byte
//                      loads, the dequantisation formula evaluated weight by weight in fp32.
//  unpack_kernel<F>    codes / scales / mins of every weight (bit-exact debug view).
//  splitk_reduce       y[n] = sum_s ws[s][n] in fixed order.
#pragma once
#include <cuda_fp16.h>

#include <cstdint>

#include "qgemv_decode.cuh"
#include "qgemv_ptx.cuh"

namespace qg {

constexpr int kDevErrTimeout = 1;
constexpr uint64_t kDrainNs = 2000000000ull;  // bound for draining copies after a timeout

struct StreamArgs {
  const uint8_t* W;    // stream 1 (all formats): rows of packed blocks / NVFP4 nibbles
  const uint8_t* W2;   // stream 2: NVFP4 scales (null otherwise)
  const uint16_t* x;   // activations (fp16 / bf16 bits)
  float* out;          // y [N], or the split-K workspace [S][N]
  int64_t N;
  int64_t row_bytes;   // stream-1 bytes per row (multiple of 16)
  int64_t row_bytes2;  // stream-2 bytes per row (multiple of 16)
  int nsb;             // 256-element superblocks per row
  int sb_per_split;    // superblocks per K slice (8 * Wk)
  int Wk;              // warps per row = slices of 8 superblocks
  int P;               // row groups per CTA (warps = P * Wk)
  int R;               // rows per stage
  int D;               // stages per warp
  int slot_bytes;      // bytes of one stage = R * slice_stride
  int slice_stride;    // bytes of one row inside a stage
  int red_rows;        // rows of the cross-warp reduction buffer (>= rows of any CTA)
  int* err;            // device error word
  uint64_t spin_ns;    // bound of every wait
  int test_stall;      // 1: warp 0 of CTA 0 waits on a barrier nothing completes
  int pdl;             // launched with programmatic dependent launch
};

// Shared memory layout: [rings: warps * D * slot_bytes][mbarriers: warps * D + 1][red].
__host__ __device__ inline size_t stream_smem_bytes(int warps, int D, int slot_bytes, int Wk, int red_rows) {
  size_t s = static_cast<size_t>(warps) * D * slot_bytes;
  s += (static_cast<size_t>(warps) * D + 1) * 8;
  s = (s + 15) & ~static_cast<size_t>(15);
  if (Wk > 1) s += static_cast<size_t>(red_rows) * Wk * 4;
  return s;
}

template <class Dec>
__global__ void __launch_bounds__(512, 1) stream_kernel(const StreamArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int SB = Dec::kSB, SB2 = Dec::kSB2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int p = warp / a.Wk, wk = warp % a.Wk;
  const int split = blockIdx.y;

  // Rows of this CTA and of this warp's row group.
  const int64_t G = gridDim.x;
  const int64_t r_lo = static_cast<int64_t>(blockIdx.x) * a.N / G;
  const int64_t r_hi = (static_cast<int64_t>(blockIdx.x) + 1) * a.N / G;
  const int64_t ncta = r_hi - r_lo;
  const int64_t p_lo = r_lo + ncta * p / a.P, p_hi = r_lo + ncta * (p + 1) / a.P;
  const int64_t nrows = p_hi - p_lo;

  // This warp's K slice: superblocks [sb0, sb0 + ncols).
  const int sbs0 = split * a.sb_per_split;
  const int sbs1 = min(a.nsb, sbs0 + a.sb_per_split);
  const int sb0 = sbs0 + 8 * wk;
  const int ncols = max(0, min(8, sbs1 - sb0));
  const int col = lane >> 2, c = lane & 3;
  const bool active = col < ncols;

  uint8_t* ring = smem + static_cast<size_t>(warp) * a.D * a.slot_bytes;
  uint64_t* bars_all = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(nwarps) * a.D * a.slot_bytes);
  uint64_t* bars = bars_all + warp * a.D;
  uint64_t* never_bar = bars_all + nwarps * a.D;
  float* red = reinterpret_cast<float*>(
      smem + ((static_cast<size_t>(nwarps) * a.D * a.slot_bytes + (static_cast<size_t>(nwarps) * a.D + 1) * 8 + 15) &
              ~static_cast<size_t>(15)));
  float* out = a.out + static_cast<int64_t>(split) * a.N;

  const int64_t nunits = ncols > 0 ? (nrows + a.R - 1) / a.R : 0;
  const uint32_t bytes1 = static_cast<uint32_t>(ncols) * SB, bytes2 = static_cast<uint32_t>(ncols) * SB2;
  const uint64_t policy = policy_evict_first();

  if (lane == 0) {
    for (int j = 0; j < a.D; ++j) mbar_init(smem_u32(bars + j), 1);
    if (warp == 0) mbar_init(smem_u32(never_bar), 1);
    fence_mbar_init();
  }
  __syncwarp();

  // Stage u of this warp: rows p_lo + u*R .. (+R), each row's slice copied on its own.
  auto issue = [&](int64_t u) {
    const int slot = static_cast<int>(u % a.D);
    const int64_t row0 = p_lo + u * a.R;
    const int nr = static_cast<int>(min(static_cast<int64_t>(a.R), nrows - u * a.R));
    const uint32_t bar = smem_u32(bars + slot);
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nr) * (bytes1 + bytes2));
    uint8_t* dst = ring + static_cast<size_t>(slot) * a.slot_bytes;
    for (int r = 0; r < nr; ++r) {
      const int64_t row = row0 + r;
      bulk_g2s(smem_u32(dst + r * a.slice_stride), a.W + row * a.row_bytes + static_cast<int64_t>(sb0) * SB, bytes1,
               bar, policy);
      if (SB2 > 0)
        bulk_g2s(smem_u32(dst + r * a.slice_stride + 8 * SB), a.W2 + row * a.row_bytes2 + static_cast<int64_t>(sb0) * SB2,
                 bytes2, bar, policy);
    }
  };

  // The packed weights are never written by the work this launch may overlap, so their
  // copies start before the dependency wait; the activations are read after it.
  if (lane == 0) {
    const int64_t pro = min(static_cast<int64_t>(a.D), nunits);
    for (int64_t u = 0; u < pro; ++u) issue(u);
  }
  if (a.pdl) pdl_wait();

  Dec dec;
  dec.load_x(a.x, sb0 + col, c, active);

  bool ok = true;
  if (a.test_stall && blockIdx.x == 0 && blockIdx.y == 0 && warp == 0)
    ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(never_bar), 0, a.spin_ns));

  int64_t u = 0;
  for (; ok && u < nunits; ++u) {
    const int slot = static_cast<int>(u % a.D);
    const uint32_t parity = static_cast<uint32_t>((u / a.D) & 1);
    ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(bars + slot), parity, a.spin_ns));
    if (!ok) break;
    const uint8_t* sp = ring + static_cast<size_t>(slot) * a.slot_bytes;
    const int nr = static_cast<int>(min(static_cast<int64_t>(a.R), nrows - u * a.R));
    for (int r = 0; r < nr; ++r) {
      const uint8_t* rp = sp + r * a.slice_stride;
      float v = active ? dec.row(rp + col * SB, rp + 8 * SB + col * SB2) : 0.f;
      v = warp_sum(v);
      const int64_t row = p_lo + u * a.R + r;
      if (lane == 0) {
        if (a.Wk == 1)
          out[row] = v;
        else
          red[(row - r_lo) * a.Wk + wk] = v;
      }
    }
    __syncwarp();
    if (lane == 0 && u + a.D < nunits) {
      fence_proxy_async_smem();
      issue(u + a.D);
    }
  }
  if (!ok) {
    // Record the timeout, then let every copy still in flight land before the CTA exits.
    if (lane == 0) {
      atomicOr(a.err, kDevErrTimeout);
      const int64_t last = min(nunits, u + a.D);
      for (int64_t v = u; v < last; ++v)
        mbar_wait_bounded(smem_u32(bars + (v % a.D)), static_cast<uint32_t>((v / a.D) & 1), kDrainNs);
    }
    __syncwarp();
  }
  if (ncols == 0 && a.Wk > 1) {
    for (int64_t row = p_lo + lane; row < p_hi; row += 32) red[(row - r_lo) * a.Wk + wk] = 0.f;
  }
  if (a.pdl) pdl_launch_dependents();
  if (a.Wk > 1) {
    named_bar_sync(1, blockDim.x);
    for (int64_t i = threadIdx.x; i < ncta; i += blockDim.x) {
      float s = 0.f;
      for (int w = 0; w < a.Wk; ++w) s += red[i * a.Wk + w];
      out[r_lo + i] = s;
    }
  }
}

// ------------------------------------------------------------------ plain per-row path
struct RowArgs {
  const uint8_t* W;
  const uint16_t* x;
  float* y;
  int64_t N, K;
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

template <int F>
__global__ void __launch_bounds__(256) rowwarp_kernel(const RowArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  constexpr int BW = FmtGeom<F>::BW, BB = FmtGeom<F>::BB;
  const int64_t nb = a.K / BW;
  for (int64_t n = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); n < a.N; n += warps) {
    float acc = 0.f;
    for (int64_t b = lane; b < nb; b += 32) {
      if constexpr (F == F_NVFP4) {
        const uint8_t* nib = a.W + n * (a.K / 2) + b * 8;
        const float s = fabsf(e4m3_f(a.W[a.N * (a.K / 2) + n * (a.K / 16) + b]));
        float part = 0.f;
        for (int j = 0; j < 16; ++j) {
          const uint32_t code = (nib[j >> 1] >> (4 * (j & 1))) & 15u;
          part = fmaf(bf2f(a.x[b * 16 + j]), e2m1_f(code) * s, part);
        }
        acc += part;
      } else {
        const uint8_t* p = a.W + (n * nb + b) * BB;
        for (int i = 0; i < BW; ++i) {
          int code;
          float scale, mn;
          elem_code<F>(p, i, code, scale, mn);
          const float w = fmaf(scale, static_cast<float>(code), -mn);
          acc = fmaf(h2f(a.x[b * BW + i]), w, acc);
        }
      }
    }
    acc = warp_sum(acc);
    if (lane == 0) a.y[n] = acc;
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
      const float2 s = DecNVFP4::e4m3x2(sb);
      scale = fabsf(s.x) * 0.5f;
      for (int j = 0; j < 16; j += 2) {
        const float2 e = DecNVFP4::e2m1x2(nib[(k0 + j) >> 1]);
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

// y[n] = ws[0][n] + ws[1][n] + ... in that order.
__global__ void __launch_bounds__(256) splitk_reduce(const float* __restrict__ ws, float* __restrict__ y, int64_t N,
                                                     int S) {
  for (int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; n < N;
       n += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float s = 0.f;
    for (int i = 0; i < S; ++i) s += ws[static_cast<int64_t>(i) * N + n];
    y[n] = s;
  }
}

}  // namespace qg
