// NVFP4 W4A16 GEMM for many activation rows (prefill): Y[t, n] = sum_k X[t, k] * w[n, k],
// w = e2m1(code) * |e4m3 block scale| ("fp4_gemv" page: the matmul role next to the GEMV,
// where a whole prompt's tokens meet each weight), on the fifth-generation tensor cores.
//
// The weights are block-scaled FP4 and the activations bf16.  A block-scaled FP4 MMA would
// need the activations in FP4 too, which changes the result; instead the weights are
// dequantised into the MMA's A operand in tensor memory.  e2m1 times an e4m3 scale has at
// most 6 significant bits and lies within [2^-10, 2688], so the bf16 operand is the exact
// weight and the tensor core's fp32 accumulation is the only rounding.
//
//  * Tile: 128 weight rows (the MMA's M, TMEM lanes) x BT tokens (its N), in stages of BK along
//    K (128 for BT <= 128, 64 for BT = 256: shared memory).  D = W_tile . X_tile^T: the
//    dequantised weights are the A operand in tensor memory (each lane a weight row, two bf16
//    per column), X the B operand in shared memory, K-major in the 128-byte swizzle layout
//    (BK / 64 sub-tiles of 128-byte rows).  When the tiles do not fill the GPU (few tokens),
//    K is split over the ks CTAs of a thread-block cluster: each leaves its partial tile in its
//    own shared memory, and CTA q of the cluster adds column slice q of all ks partials through
//    distributed shared memory, in rank order (so the result does not depend on which CTA
//    finishes first).
//  * Warp 0: allocates TMEM, then one lane loads the X tile of each stage with a 2-D TMA copy
//    (rows past T read as zeros).  Warp 1: one lane issues tcgen05.mma (BK / 16 steps of K 16 per
//    stage) once the stage's one full barrier has the X copy's bytes and the arrivals of its
//    256 dequantising threads, and frees the stage with tcgen05.commit.  Warps 2..17
//    dequantise in two groups of eight that take the even and the odd stages: the thread of
//    TMEM lane r and half hh copies its BK / 4 bytes of codes and 4 scale bytes of each of its
//    stages into a private ring with cp.async (three stages ahead), then writes the BK / 2
//    weights as bf16 pairs into the stage's A columns with tcgen05.st.  Afterwards the 16
//    warps read the accumulator with tcgen05.ld (each its TMEM lane quarter and a quarter of
//    the columns).
//  * Shared memory carries only X and the raw codes: the weights never round-trip through it.
//  * Each CTA starts its K loop at its own offset, so that concurrent CTAs ask for different
//    K-blocks of X (no measured change on the shapes timed, where the MMA-issuing thread's
//    loop is the limit; it costs nothing).
//  * Every wait on an mbarrier is bounded; a wait that gives up sets the error word, and the
//    CTA still waits for its copies and MMAs and frees its TMEM before it returns.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "qgemv_decode.cuh"
#include "qgemv_ptx.cuh"
#include "qgemv_stream.cuh"

namespace qg {

constexpr int kTcRows = 128;        // weight rows per tile: the MMA's M and the TMEM lanes
constexpr int kTcGroupWarps = 8;    // dequantising warps per group (two groups: even and odd stages)
constexpr int kTcThreads = 32 * (2 + 2 * kTcGroupWarps);
constexpr int kTcRawDepth = 4;      // raw stages per group (cp.async ring, three in flight)

struct TcArgs {
  const uint8_t* W;  // e2m1 codes [N, K/2], low nibble first
  const uint8_t* S;  // e4m3 block scales [N, K/16]
  float* y;          // [T, N] fp32
  int64_t N;
  int T, K;
  int n_ttiles;      // token tiles: ceil(T / BT)
  int ks, kb_per;    // K splits per tile (the cluster size) and K-blocks (of tc_bk) per split
  int* err;
  uint64_t spin_ns;
  int stall;         // test hook: CTA 0's dequantisers withhold their arrival for its first stage
};

// K per stage: 128 (two 128-byte swizzle rows of bf16, eight MMAs per barrier round trip) for
// tiles of up to 128 tokens; 64 for 256-token tiles, whose X stages would not fit otherwise.
__host__ __device__ constexpr int tc_bk(int BT) { return BT > 128 ? 64 : 128; }
// Stages (X in shared memory, A in TMEM), within 227 KB of shared memory and 512 TMEM columns.
__host__ __device__ constexpr int tc_stages(int BT) { return BT > 128 ? 5 : BT > 64 ? 4 : 6; }
// Raw stage: codes [half][128 rows][BK / 4 bytes], scales [half][128 rows][4 bytes].
__host__ __device__ constexpr int tc_raw_bytes(int BT) { return 2 * kTcRows * (tc_bk(BT) / 4) + 2 * kTcRows * 4; }
// TMEM columns: the accumulator [0, BT), A stage s at BT + (BK / 2) s (a power of 2)
__host__ __device__ constexpr int tc_tmem_cols(int BT) {
  return BT + tc_stages(BT) * (tc_bk(BT) / 2) <= 256 ? 256 : 512;
}
__host__ __device__ constexpr size_t tc_smem_bytes(int BT) {
  return 1024 + static_cast<size_t>(tc_stages(BT)) * BT * 2 * tc_bk(BT) +
         static_cast<size_t>(2 * kTcRawDepth) * tc_raw_bytes(BT) + 256;
}

// ------------------------------------------------------------------ tcgen05 / TMA wrappers
__device__ __forceinline__ void tmem_alloc(uint32_t slot_sa, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_sa), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// The mbarrier gets one arrival once every MMA this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
// 16 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 16 consecutive 32-bit TMEM columns of this thread's lane <- v.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// D (TMEM) = A B^T (+ D when acc != 0): A from TMEM columns, B from a shared-memory descriptor.
__device__ __forceinline__ void tc_mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                               uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major tile in the 128-byte swizzle layout: rows of
// 128 bytes, 8-row groups 1024 bytes apart (stride byte offset), tile base 1024-byte aligned;
// the K = 16 slices of a row are 32 bytes apart (start address advanced by 32 k).
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both K-major, M x N.
__host__ __device__ constexpr uint32_t tc_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
// Every thread of every CTA of the cluster arrives; this CTA's earlier shared-memory writes are
// visible to the cluster after the wait.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// fp32 at shared address `a` of cluster CTA `rank`
__device__ __forceinline__ float ld_dsmem_f32(uint32_t a, uint32_t rank) {
  uint32_t ra;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t tc_hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// fp16 pair -> bf16 pair (exact for the dequantised weights: 6 significant bits, normal range)
__device__ __forceinline__ uint32_t h2_to_bf2(uint32_t h) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
  return *reinterpret_cast<const uint32_t*>(&b);
}

template <int BT>
__global__ void __launch_bounds__(kTcThreads, 1) tc_nvfp4_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                 const __grid_constant__ TcArgs a) {
  static_assert(BT == 64 || BT == 128 || BT == 256, "MMA N");
  constexpr int TC = tc_tmem_cols(BT);
  constexpr int RD = kTcRawDepth;
  constexpr int kTcStages = tc_stages(BT);
  constexpr int BK = tc_bk(BT), NSUB = BK / 64;    // K per stage, 128-byte swizzle rows per X row
  constexpr int XSTAGE = BT * 2 * BK;               // bytes of an X stage: NSUB sub-tiles of BT x 128
  constexpr int ACOLS = BK / 2;                     // TMEM columns of an A stage
  constexpr int RAW = tc_raw_bytes(BT), CODES = BK / 4;  // raw stage bytes, code bytes per half row
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t xs0 = base;                                 // X stages: NSUB x BT rows x 128 bytes
  const uint32_t rs0 = base + kTcStages * XSTAGE;            // raw stages: [group][RD]
  const uint32_t bars = rs0 + 2 * RD * RAW;                  // full[S], empty[S], accum
  const uint32_t accum = bars + 8 * 2 * kTcStages;
  const uint32_t tslot = accum + 8;                          // TMEM base written by tcgen05.alloc
  // full[s]: the X copy (one arrival with its transaction bytes) and the stage's 256
  // dequantising threads; empty[s]: the MMAs that read stage s have completed
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (kTcStages + s); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // block = (weight tile, token tile, split): the splits of a tile form one cluster
  const unsigned ntt = static_cast<unsigned>(a.n_ttiles), uks = static_cast<unsigned>(a.ks);
  const int ksi = static_cast<int>(blockIdx.x % uks);
  const unsigned tile = blockIdx.x / uks;
  const int tt = static_cast<int>(tile % ntt), wt = static_cast<int>(tile / ntt);
  const int t0 = tt * BT;
  const int64_t n0 = static_cast<int64_t>(wt) * kTcRows;
  const int kb0 = ksi * a.kb_per;
  const int nkb = min(a.K / BK - kb0, a.kb_per);  // K-blocks of this CTA (>= 1)
  // The CTA walks its K-blocks from a rotated start, so CTAs that run at the same time ask for
  // different K-blocks of X and of the weight tiles that token tiles share.  The order is
  // fixed per CTA, so results are reproducible.
  const int rot = static_cast<int>((static_cast<unsigned>(wt) * 17u + static_cast<unsigned>(tt) * 5u) %
                                   static_cast<unsigned>(nkb));
  auto kb_at = [&](int i) { return kb0 + (i + rot < nkb ? i + rot : i + rot - nkb); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(full(s), 1 + kTcGroupWarps * 32);
      mbar_init(empty(s), 1);
    }
    mbar_init(accum, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, TC);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = lds_u32(tslot);  // accumulator at column 0, A stage s at BT + ACOLS s
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {  // ---- X tiles by TMA
      int i = 0;
      for (; i < nkb; ++i) {
        const int s = i % kTcStages;
        const uint32_t ph = (i / kTcStages) & 1;
        if (i >= kTcStages && !mbar_wait_bounded(empty(s), ph ^ 1, a.spin_ns)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(full(s), XSTAGE);
#pragma unroll
        for (int u = 0; u < NSUB; ++u)
          tma_load_2d(xs0 + s * XSTAGE + u * BT * 128, &xmap, kb_at(i) * BK + 64 * u, t0, full(s));
      }
      // the copies issued last have landed before the CTA may leave (their stages' full phases
      // complete once the copy and the stage's dequantisers are in)
      for (int j = i > kTcStages ? i - kTcStages : 0; j < i; ++j)
        if (!mbar_wait_bounded(full(j % kTcStages), (j / kTcStages) & 1, a.spin_ns)) ok = false;
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issue
      constexpr uint32_t idesc = tc_idesc_bf16(kTcRows, BT);
      // descriptor of stage 0; K-step k of stage s starts at byte s XSTAGE + (k / 4) BT 128 +
      // 32 (k % 4), a sixteenth of that added to the start-address field (no carry: addresses
      // stay below 2^18)
      const uint64_t xd0 = tc_desc_sw128(xs0);
      int s = 0;
      uint32_t ph = 0;
      for (int i = 0; i < nkb; ++i) {
        if (!mbar_wait_bounded(full(s), ph, a.spin_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t xd = xd0 + static_cast<uint64_t>(s * (XSTAGE / 16));
        const uint32_t ta = tmem + BT + ACOLS * s;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          tc_mma_bf16_ta(tmem, ta + 8 * k, xd + static_cast<uint64_t>((k >> 2) * (BT * 8) + 2 * (k & 3)), idesc,
                         k == 0 ? static_cast<uint32_t>(i) : 1u);
        tc_commit(empty(s));
        if (++s == kTcStages) s = 0, ph ^= 1;
      }
      tc_commit(accum);  // also after a failure: the epilogue then finds the MMAs complete
    }
  } else {
    // ---- dequantisation: warp group g takes stages g, g + 2, ...; the thread of TMEM lane r
    // (row r of the tile) and half hh writes A columns hh BK / 4 .. (hh + 1) BK / 4 - 1 of each
    const int dw = warp - 2, q4 = warp & 3, hh = (dw >> 2) & 1, g = dw >> 3;
    const int r = 32 * q4 + lane;
    const int64_t n = n0 + r;
    const bool rv = n < a.N;
    const uint8_t* wrow = a.W + (rv ? n : 0) * static_cast<int64_t>(a.K / 2) + CODES * hh;
    // scales: BK = 128 takes the 4 bytes of its half (blocks 4 hh .. 4 hh + 3); BK = 64 the
    // row's 4 bytes of the stage, of which its half uses 2
    const uint8_t* srow = a.S + (rv ? n : 0) * static_cast<int64_t>(a.K / 16) + (BK == 128 ? 4 * hh : 0);
    // raw slot: codes [half][row][CODES] (a warp's 32 rows of one half are contiguous),
    // scales [half][row][4 B]
    const uint32_t rq = static_cast<uint32_t>((hh * kTcRows + r) * CODES);
    const uint32_t rsc = static_cast<uint32_t>(2 * kTcRows * CODES + (hh * kTcRows + r) * 4);
    const uint32_t ring = rs0 + static_cast<uint32_t>(g * RD) * RAW;
    const uint32_t lane_a = tmem + (static_cast<uint32_t>(32 * q4) << 16) + BT + (ACOLS / 2) * hh;
    const int nj = (nkb - g + 1) / 2;  // this group's stages
    auto issue = [&](int j) {
      const uint32_t slot = ring + static_cast<uint32_t>(j % RD) * RAW;
      if (j < nj && rv) {
        const int64_t kb = kb_at(g + 2 * j);
#pragma unroll
        for (int u = 0; u < CODES / 16; ++u) cp_async16(slot + rq + 16 * u, wrow + kb * (BK / 2) + 16 * u);
        cp_async4(slot + rsc, srow + kb * (BK / 16));
      }
      cp_async_commit();
    };
#pragma unroll 1
    for (int j = 0; j < RD - 1; ++j) issue(j);
    for (int j = 0; j < nj; ++j) {
      const int i = g + 2 * j, s = i % kTcStages;
      const uint32_t ph = (i / kTcStages) & 1;
      issue(j + RD - 1);
      if (i >= kTcStages && !mbar_wait_bounded(empty(s), ph ^ 1, a.spin_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();  // the MMAs that read A stage s are complete
      cp_async_wait<RD - 1>();
      const uint32_t slot = ring + static_cast<uint32_t>(j % RD) * RAW;
      uint32_t c = lds_u32(slot + rsc);
      if (BK == 64) c >>= 16 * hh;  // the half's two scale bytes
      if (!rv) c = 0;
      // |scale| of the half's blocks as fp16 pairs (block b in both halves of sc[b])
      uint32_t sc[CODES / 8];
#pragma unroll
      for (int b = 0; b < CODES / 8; b += 2) {
        const uint32_t s2 = DecNVFP4::e4m3x2((c >> (8 * b)) & 0x7F7Fu);
        sc[b] = __byte_perm(s2, s2, 0x1010);
        sc[b + 1] = __byte_perm(s2, s2, 0x3232);
      }
#pragma unroll
      for (int part = 0; part < CODES / 16; ++part) {  // 16 code bytes = 32 weights = 16 columns
        uint4 qv = lds_v4(slot + rq + 16 * part);
        if (!rv) qv = make_uint4(0u, 0u, 0u, 0u);
        const uint32_t wv[4] = {qv.x, qv.y, qv.z, qv.w};
        uint32_t v[16];
#pragma unroll
        for (int w = 0; w < 4; ++w) {  // word w: 8 elements (columns 4 w .. 4 w + 3 of the part)
          uint32_t hv[4];
          DecNVFP4::e2m1x8(wv[w], hv);
          const uint32_t sj = sc[2 * part + (w >> 1)];
#pragma unroll
          for (int u = 0; u < 4; ++u) v[4 * w + u] = h2_to_bf2(tc_hmul2(hv[u], sj));
        }
        tmem_st16(lane_a + ACOLS * s + 16 * part, v);
      }
      tmem_st_wait();
      tc_fence_before();
      if (!(a.stall && blockIdx.x == 0 && i == 0)) mbar_arrive(full(s));
    }
    cp_async_wait<0>();

    // ---- epilogue: TMEM lane quarter q4, column quarter dw / 4
    if (!mbar_wait_bounded(accum, 0, a.spin_ns)) ok = false;
    tc_fence_after();
    const int part = dw >> 2;
    const int64_t nrow = n0 + r;
    const bool nv = nrow < a.N;
    const bool split = a.ks > 1;
#pragma unroll 1
    for (int c = part * (BT / 4); c < (part + 1) * (BT / 4); c += 16) {
      uint32_t v[16];
      tmem_ld16(tmem + (static_cast<uint32_t>(32 * q4) << 16) + static_cast<uint32_t>(c), v);
      tmem_ld_wait();
      if (split) {  // partial tile into this CTA's (now idle) X stages: red[column][row]
#pragma unroll
        for (int j = 0; j < 16; ++j)
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(xs0 + ((c + j) * kTcRows + r) * 4), "r"(v[j]) : "memory");
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = t0 + c + j;
          if (nv && t < a.T) a.y[static_cast<int64_t>(t) * a.N + nrow] = __uint_as_float(v[j]);
        }
      }
    }
  }

  if (a.ks > 1) {
    // ---- split K: the cluster's partial tiles are complete after the first barrier; CTA ksi
    // adds columns [ksi BT / ks, (ksi + 1) BT / ks) of all of them, in rank order, then the
    // second barrier keeps every CTA's shared memory alive until the others are done with it.
    __syncwarp();
    cluster_sync();
    const int c_lo = (ksi * BT) / a.ks, c_hi = ((ksi + 1) * BT) / a.ks;
    const int per = (c_hi - c_lo) * kTcRows;
    for (int e = threadIdx.x; e < per; e += kTcThreads) {
      const int c = c_lo + e / kTcRows, rr = e % kTcRows;
      const int t = t0 + c;
      const int64_t nr = n0 + rr;
      float acc = 0.f;
      for (int q = 0; q < a.ks; ++q) acc += ld_dsmem_f32(xs0 + (c * kTcRows + rr) * 4, static_cast<uint32_t>(q));
      if (t < a.T && nr < a.N) a.y[static_cast<int64_t>(t) * a.N + nr] = acc;
    }
    cluster_sync();
  }

  if (!ok) atomicOr(a.err, kDevErrTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TC);
  }
}

template <int BT>
const void* tc_kernel_ptr() {
  return reinterpret_cast<const void*>(&tc_nvfp4_kernel<BT>);
}

}  // namespace qg
