// Streaming GEMV kernel.
//
// The row range of a CTA is covered by P row groups x Wk K-columns of warps.  Warp (p, wk)
// owns K-column wk (2048 elements = 8 superblocks): each lane keeps the activations of its
// 64-element piece in registers for the whole kernel, and the warp walks down the rows of
// its row group, R rows per stage, streaming only its own slice of each row.
//  * Weights reach shared memory through a private ring of D stages per warp, filled with
//    16-byte cp.async copies (cache-global) issued by all 32 lanes.  A stage is consumed
//    after cp.async.wait_group, which the hardware tracks per thread: a warp waiting for
//    data stalls on its scoreboard and takes no issue slots from warps that are decoding.
//  * Each lane decodes its piece of each row (qgemv_decode.cuh); the warp adds its 32
//    lanes; the Wk partial sums of a row are added in a fixed order in shared memory at the
//    end, so results are bitwise reproducible.
//  * The first stages are requested before the programmatic-dependent-launch wait (they
//    are weights, which the kernel this launch may overlap does not write); the
//    activations are read after it.
#pragma once
#include <cuda_fp16.h>

#include <cstdint>

#include "qgemv_decode.cuh"
#include "qgemv_ptx.cuh"

namespace qg {

constexpr int kDevErrTimeout = 1;

struct StreamArgs {
  const uint8_t* W;     // stream 1: rows of packed blocks / NVFP4 nibbles
  const uint8_t* W2;    // stream 2: NVFP4 scales (null otherwise)
  const uint16_t* x;    // activations (fp16, bf16 for NVFP4)
  float* y;
  int64_t N;
  int64_t row_bytes, row_bytes2;  // bytes per row of stream 1 / 2 (multiples of 16)
  int nsb;              // superblocks per row
  int Wk;               // K-columns (warps per row group) = ceil(nsb / 8)
  int P;                // row groups per CTA
  int D;                // stages per warp: 2, 3, 4 or 6
  int red_rows;         // rows of the reduction buffer (>= rows of any CTA)
  int* err;
  uint64_t spin_ns;
  int test_stall;       // 1: warp 0 of CTA 0 also waits, bounded, on a barrier nothing completes
};

template <class Dec>
__host__ __device__ constexpr int slice_bytes() {
  return 8 * Dec::kSB + 8 * Dec::kSB2;
}

// Shared memory: [rings: warps * D * R * slice][reduction buffer][never-completing barrier]
__host__ __device__ inline size_t stream_ring_bytes(int warps, int D, int R, int slice) {
  return static_cast<size_t>(warps) * D * R * slice;
}
__host__ __device__ inline size_t stream_bar_offset(int warps, int D, int R, int slice, int Wk, int red_rows) {
  size_t s = stream_ring_bytes(warps, D, R, slice);
  if (Wk > 1) s += static_cast<size_t>(red_rows) * Wk * 4;
  return (s + 15) & ~static_cast<size_t>(15);
}
__host__ __device__ inline size_t stream_smem_bytes(int warps, int D, int R, int slice, int Wk, int red_rows) {
  return stream_bar_offset(warps, D, R, slice, Wk, red_rows) + 16;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// One warp's whole life after set-up: prologue copies, activations, then the stage loop.
template <class Dec, int R, int D>
__device__ __forceinline__ void warp_stream(const StreamArgs& a, Dec& dec, uint8_t* ring, float* red, int64_t r_lo,
                                            int64_t p_lo, int64_t nrows, int wk, int ncols, int lane) {
  constexpr int SB = Dec::kSB, SB2 = Dec::kSB2, SLICE = slice_bytes<Dec>();
  constexpr int STAGE = R * SLICE;
  const int col = lane >> 2, c = lane & 3;
  const bool active = col < ncols;
  const int n1 = ncols * SB / 16, n2 = ncols * SB2 / 16;  // 16-byte copies per row
  const int nst = static_cast<int>((nrows + R - 1) / R);
  const uint32_t ring_s = smem_u32(ring);
  const uint8_t* src1 = a.W + p_lo * a.row_bytes + static_cast<int64_t>(wk) * 8 * SB;
  const uint8_t* src2 = (SB2 > 0) ? a.W2 + p_lo * a.row_bytes2 + static_cast<int64_t>(wk) * 8 * SB2 : a.W;

  auto issue = [&](int st) {
    if (st < nst) {
      const int r0 = st * R;
      const int nr = static_cast<int>(min(static_cast<int64_t>(R), nrows - r0));
      const uint32_t dst = ring_s + (st % D) * STAGE;
      for (int r = 0; r < nr; ++r) {
        const uint8_t* s1 = src1 + static_cast<int64_t>(r0 + r) * a.row_bytes;
        for (int i = lane; i < n1; i += 32) cp_async16(dst + r * SLICE + 16 * i, s1 + 16 * i);
        if (SB2 > 0) {
          const uint8_t* s2 = src2 + static_cast<int64_t>(r0 + r) * a.row_bytes2;
          for (int i = lane; i < n2; i += 32) cp_async16(dst + r * SLICE + 8 * SB + 16 * i, s2 + 16 * i);
        }
      }
    }
    cp_async_commit();
  };

#pragma unroll
  for (int s = 0; s < D - 1; ++s) issue(s);
  pdl_wait();
  dec.load_x(a.x, 8 * wk + col, c, active);

  for (int st = 0; st < nst; ++st) {
    issue(st + D - 1);
    cp_async_wait<D - 1>();
    __syncwarp();
    const uint8_t* s1 = ring + (st % D) * STAGE + col * SB;
    const uint8_t* s2 = ring + (st % D) * STAGE + 8 * SB + col * SB2;
    const int r0 = st * R;
    const int nr = static_cast<int>(min(static_cast<int64_t>(R), nrows - r0));
    float v[R];
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] = 0.f;
    if (active) {
      if (nr == R) {
#pragma unroll
        for (int r = 0; r < R; ++r) v[r] = dec.row(s1 + r * SLICE, s2 + r * SLICE);
      } else {  // last, partial stage of the row group
#pragma unroll
        for (int r = 0; r < R; ++r)
          if (r < nr) v[r] = dec.row(s1 + r * SLICE, s2 + r * SLICE);
      }
    }
    __syncwarp();  // every lane is done with this slot before it is refilled
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (r < nr) {
        const float sum = warp_sum(v[r]);
        if (lane == 0) {
          const int64_t row = p_lo + r0 + r;
          if (a.Wk == 1)
            a.y[row] = sum;
          else
            red[(row - r_lo) * a.Wk + wk] = sum;
        }
      }
    }
  }
  cp_async_wait<0>();
}

template <class Dec, int R>
__global__ void __launch_bounds__(512, 1) stream_kernel(const StreamArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int SLICE = slice_bytes<Dec>();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int p = warp / a.Wk, wk = warp % a.Wk;

  const int64_t G = gridDim.x;
  const int64_t r_lo = static_cast<int64_t>(blockIdx.x) * a.N / G;
  const int64_t r_hi = (static_cast<int64_t>(blockIdx.x) + 1) * a.N / G;
  const int64_t ncta = r_hi - r_lo;
  const int64_t p_lo = r_lo + ncta * p / a.P, p_hi = r_lo + ncta * (p + 1) / a.P;
  const int ncols = min(8, a.nsb - 8 * wk);

  uint8_t* ring = smem + static_cast<size_t>(warp) * a.D * R * SLICE;
  float* red = reinterpret_cast<float*>(smem + stream_ring_bytes(nwarps, a.D, R, SLICE));
  uint64_t* never_bar = reinterpret_cast<uint64_t*>(smem + stream_bar_offset(nwarps, a.D, R, SLICE, a.Wk, a.red_rows));

  pdl_launch_dependents();  // the next kernel may start copying its weights right away
  if (a.test_stall && blockIdx.x == 0 && warp == 0) {
    if (lane == 0) {
      mbar_init(smem_u32(never_bar), 1);
      fence_mbar_init();
      if (!mbar_wait_bounded(smem_u32(never_bar), 0, a.spin_ns)) atomicOr(a.err, kDevErrTimeout);
    }
    __syncwarp();
  }
  Dec dec;
  dec.init(lane & 3);
  const int64_t nrows = p_hi - p_lo;
  switch (a.D) {
    case 2: warp_stream<Dec, R, 2>(a, dec, ring, red, r_lo, p_lo, nrows, wk, ncols, lane); break;
    case 3: warp_stream<Dec, R, 3>(a, dec, ring, red, r_lo, p_lo, nrows, wk, ncols, lane); break;
    case 4: warp_stream<Dec, R, 4>(a, dec, ring, red, r_lo, p_lo, nrows, wk, ncols, lane); break;
    default: warp_stream<Dec, R, 6>(a, dec, ring, red, r_lo, p_lo, nrows, wk, ncols, lane); break;
  }
  if (a.Wk > 1) {
    __syncthreads();
    for (int64_t i = threadIdx.x; i < ncta; i += blockDim.x) {
      float s = 0.f;
      for (int w = 0; w < a.Wk; ++w) s += red[i * a.Wk + w];
      a.y[r_lo + i] = s;
    }
  }
}

}  // namespace qg
