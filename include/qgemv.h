/*
 * qgemv: batch-1 GEMV with block-quantised weights dequantised on the fly, for GB300
 * (sm_103a).
 *
 *     y[n] = sum_k x[k] * dequant(W)[n, k],   n < N, k < K        (M = 1, alpha = 1, beta = 0)
 *
 * The operation is the GEMV of "Writing a high performant GEMV + dequant for Metal"
 * (section "What is a GEMV": y = alpha x.W^T + beta C with x:(1,K), W:(M,K), alpha = 1,
 * beta = 0; that page's M is N here) and of the Mojo "fp4_gemv" page (out = x @ dequant(W)^T
 * at M = 1).  Weights stay in their packed block format in device memory; every kernel
 * streams the packed bytes once, decodes them in registers and accumulates in fp32.
 *
 * Conventions for every entry point:
 *  - Pointers named x, W, y, codes, scales, mins are DEVICE pointers owned by the caller.
 *    The library never frees, keeps or retains them past the call's stream work.
 *  - Calls are asynchronous on `stream`; nothing is allocated and nothing synchronises
 *    inside qgemv_run / qgemv_unpack.  Results are ready when the stream's work is done.
 *  - Errors are reported only through the returned status; arguments are validated before
 *    anything is launched, so an error status means no kernel was enqueued (except
 *    QGEMV_ERR_CUDA, which means the launch itself failed).
 *  - A handle may be used from one host thread at a time.
 */
#ifndef QGEMV_H_
#define QGEMV_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Weight formats.  Byte layouts (offsets inside one block, fp16 little-endian):
 *  QGEMV_Q4_K  256 weights / 144 B: d@0, dmin@2, 12 B packed 6-bit scales+mins@4,
 *              qs[128]@16.  w_i = d*s_g*q_i - dmin*m_g, g = i/32 (Metal GEMV page,
 *              sections "What is a weight block?" and "Compute").  x fp16.
 *  QGEMV_NVFP4 W4A16 (Mojo fp4_gemv page, "Structure"): E2M1 nibbles [N, K/2] (low nibble
 *              = even k) immediately followed, in the SAME buffer, by E4M3 scales
 *              [N, K/16]; w = e2m1 * |e4m3 scale of its 16-element block|.  x bf16.
 *  QGEMV_TQ1_0 256 weights / 54 B: qs[48]@0 (5 base-3 digits per byte), qh[4]@48
 *              (4 digits per byte), d@52; digit n of byte b = floor(3^(n+1) b/256) -
 *              3 floor(3^n b/256); w = d*(t-1) ("metal: TQ1_0 kernel performance",
 *              sections 1, 2 and "Not applicable").  x fp16.
 *  QGEMV_Q5_K  256 weights / 176 B: d@0, dmin@2, scales[12]@4, qh[32]@16, qs[128]@48.
 *  QGEMV_Q6_K  256 weights / 210 B: ql[128]@0, qh[64]@128, int8 scales[16]@192, d@208.
 *  QGEMV_Q8_0   32 weights /  34 B: d@0, int8 qs[32]@2.
 *  (Q5_K, Q6_K and Q8_0 are named on the Metal GEMV page, section "UD-Q4_K_XL"; their
 *  standard ggml layouts are used.)  x fp16 for all of them. */
typedef enum {
  QGEMV_Q4_K = 0,
  QGEMV_NVFP4 = 1,
  QGEMV_TQ1_0 = 2,
  QGEMV_Q5_K = 3,
  QGEMV_Q6_K = 4,
  QGEMV_Q8_0 = 5
} qgemv_format_t;

typedef enum {
  QGEMV_OK = 0,
  QGEMV_ERR_INVALID_ARG = 1,        /* null pointer / handle, bad option value */
  QGEMV_ERR_UNSUPPORTED_FORMAT = 2, /* format id not in qgemv_format_t */
  QGEMV_ERR_BAD_SHAPE = 3,          /* N < 1, K < 1, K not a multiple of the block length */
  QGEMV_ERR_MISALIGNED = 4,         /* x, W or y not 16-byte aligned */
  QGEMV_ERR_CUDA = 5,               /* a CUDA runtime call or kernel launch failed */
  QGEMV_ERR_TIMEOUT = 6,            /* a kernel gave up on a bounded wait (see check_error) */
  QGEMV_ERR_OOM = 7,                /* qgemv_create could not allocate its workspace */
  QGEMV_ERR_NO_DEVICE = 8,          /* no usable CUDA device / not an sm_103 device */
  QGEMV_ERR_TOO_LARGE = 9           /* shape needs more than qgemv_run_noalloc's fixed scratch */
} qgemv_status_t;

typedef struct qgemv_handle_s* qgemv_handle_t;

/* Create a handle on CUDA device `device` (made current for the call).  Queries the SM
 * count and L2 size and allocates the handle's device memory: a 4-byte error word, a 16 MiB
 * workspace for split-K column sums and 4 KiB of per-range counters (zeroed here; every
 * launch leaves them at zero).  *h receives the handle.  Returns QGEMV_ERR_NO_DEVICE when
 * the device is missing or is not compute capability 10.3, QGEMV_ERR_OOM when an allocation
 * fails. */
qgemv_status_t qgemv_create(qgemv_handle_t* h, int device);

/* Free the handle's device memory and the handle.  Waits for nothing: the caller must
 * make sure no work using the handle is still pending.  NULL is accepted. */
qgemv_status_t qgemv_destroy(qgemv_handle_t h);

/* y = x . dequant(W)^T  (overwrites y).
 *   x        device, K elements: fp16 bits (bf16 for QGEMV_NVFP4), 16-byte aligned.
 *   packed_W device, qgemv_packed_bytes(fmt, N, K) bytes, rows contiguous, 16-byte aligned.
 *   y        device, N fp32 values, 16-byte aligned; must not overlap x or packed_W.
 *   N >= 1; K >= 1 and a multiple of 256 (Q4_K, Q5_K, Q6_K, TQ1_0), 32 (Q8_0) or 16 (NVFP4).
 * The call is asynchronous on `stream` (0 = legacy default stream), allocates nothing and
 * does not synchronise.  It may use the handle's workspace, so calls on one handle must not
 * run at the same time on the GPU: calls ordered on one stream are fine; concurrent streams
 * need one handle each.  Results are deterministic: the same inputs and shape give
 * bitwise-identical y on every call (every sum is taken in a fixed order; the one atomic,
 * a per-range arrival count, only picks which CTA adds the column sums). */
qgemv_status_t qgemv_run(qgemv_handle_t h, qgemv_format_t fmt, const void* x, const void* packed_W,
                         int64_t N, int64_t K, float* y, cudaStream_t stream);

/* Debug unpack for bit-exact checks: for every weight (n, k)
 *     dequant(W)[n, k] = scales[n, k/G] * codes[n, k] - mins[n, k/G]      (exactly, in fp32)
 * with G = qgemv_group_size(fmt) and
 *   Q4_K, Q5_K: codes = q (0..15 / 0..31), scales = d*s_g, mins = dmin*m_g   (G = 32)
 *   Q6_K:       codes = q-32 (-32..31),    scales = d*sc,    mins = 0        (G = 16)
 *   Q8_0:       codes = int8 q,            scales = d,       mins = 0        (G = 32)
 *   TQ1_0:      codes = t-1 (-1..1),       scales = d,       mins = 0        (G = 256)
 *   NVFP4:      codes = 2*e2m1 (-12..12),  scales = |e4m3|/2, mins = 0       (G = 16)
 * All scales and mins are exact in fp32.  codes: device int8 [N, K]; scales: device fp32
 * [N, K/G]; mins: device fp32 [N, K/G] or NULL.  Same validation as qgemv_run (codes,
 * scales, mins need no 16-byte alignment).  Asynchronous on `stream`. */
qgemv_status_t qgemv_unpack(qgemv_handle_t h, qgemv_format_t fmt, const void* packed_W, int64_t N,
                            int64_t K, int8_t* codes, float* scales, float* mins, cudaStream_t stream);

/* Synchronise `stream`, then read and clear the handle's device error word.  Returns
 * QGEMV_ERR_TIMEOUT if any kernel since the last check gave up on a bounded wait (its y
 * is then undefined), QGEMV_ERR_CUDA if the stream reported an error, else QGEMV_OK. */
qgemv_status_t qgemv_check_error(qgemv_handle_t h, cudaStream_t stream);

/* Static description of a status code (never NULL). */
const char* qgemv_status_string(qgemv_status_t status);

/* Bytes of a packed N x K matrix in `fmt` (0 for an unknown format or a bad shape). */
size_t qgemv_packed_bytes(qgemv_format_t fmt, int64_t N, int64_t K);

/* Group length G of qgemv_unpack's scales for `fmt` (0 for an unknown format). */
int qgemv_group_size(qgemv_format_t fmt);

/* Tuning and test options (per handle).  Values are validated; bad ones give
 * QGEMV_ERR_INVALID_ARG and change nothing.
 *   QGEMV_OPT_FORCE_PATH      0 auto, 1 the cp.async streaming kernels (falls back to 0
 *                             when the shape does not meet their alignment rule) and, in
 *                             qgemv_run_batch, the batch kernel for every M >= 2 it takes
 *                             (whatever N), 2 the plain warp-per-row kernels.
 *   QGEMV_OPT_RING_DEPTH      0 auto, else 2..8: copy stages per warp of the streaming
 *                             kernel (2, 3 or 4 are used, larger values mean 4; fewer
 *                             if they do not fit in shared memory).
 *   QGEMV_OPT_ROWS_PER_STAGE  0 auto, else 1..8 rows per stage (1, 2 or 4 are used).
 *   QGEMV_OPT_SPIN_LIMIT_NS   bound, in ns, of every spin-wait on a barrier in the kernels
 *                             (default 1e9); 0 makes such a wait give up at once.  (The
 *                             streaming kernel waits for its own copies with
 *                             cp.async.wait_group, which the hardware completes.)
 *   QGEMV_OPT_PDL             1 launches the streaming kernels with programmatic dependent
 *                             launch: they may start while the previous kernel on the stream
 *                             is still running, and they request their first weight stages
 *                             before waiting for it; activations are read only after it
 *                             completes.  packed_W must therefore not be written by the kernel
 *                             launched just before.  0 (default) launches them normally.
 *   QGEMV_OPT_TEST_STALL      test hook, default 0.  1 makes warp 0 of the first CTA of every
 *                             streaming launch also wait on a barrier that nothing completes,
 *                             bounded by the spin limit, so the timeout path (error word,
 *                             draining of in-flight copies, QGEMV_ERR_TIMEOUT from
 *                             qgemv_check_error) can be exercised without hanging a GPU; in
 *                             qgemv_run_gemm's tensor-core kernel, the first CTA's
 *                             dequantising threads withhold their arrival for its first stage,
 *                             so its MMA, copy and dequantising waits all run out.
 *   QGEMV_OPT_CTAS_PER_SM     streaming kernel CTAs per SM, 1 or 2 (default 2, used when
 *                             a row needs at most 8 warps); with 1, each CTA takes about half
 *                             an SM, so the next kernel of a programmatic-dependent-launch
 *                             chain can start on the other half.
 *   QGEMV_OPT_KSPLIT          0 (default): when K > 4096 and N * ceil(K / 2048) <= 4 Mi, each
 *                             CTA of the streaming kernel takes one 2048-wide K-column of a
 *                             range of rows (so it reads only that part of x) and the column
 *                             sums of a row meet in the handle's workspace, where the last
 *                             CTA of the range adds them in column order.  1: each CTA covers
 *                             every K-column of its rows and adds them in shared memory.
 *   QGEMV_OPT_GRID_PER_SM     0 (default): as many streaming CTAs per SM as fit, except
 *                             that with QGEMV_OPT_PDL a launch that covers K in one CTA and
 *                             has at most 16 rows per warp takes one CTA per SM; 1: one per
 *                             SM; 2: two per SM.  One per SM leaves the rest of each SM to
 *                             the next kernel of a programmatic-dependent-launch chain, whose
 *                             CTAs then fetch their first weights while this one finishes. */
typedef enum {
  QGEMV_OPT_FORCE_PATH = 0,
  QGEMV_OPT_RING_DEPTH = 2,
  QGEMV_OPT_ROWS_PER_STAGE = 3,
  QGEMV_OPT_SPIN_LIMIT_NS = 4,
  QGEMV_OPT_PDL = 5,
  QGEMV_OPT_TEST_STALL = 6,
  QGEMV_OPT_CTAS_PER_SM = 7,
  QGEMV_OPT_KSPLIT = 8,
  QGEMV_OPT_GRID_PER_SM = 9
} qgemv_option_t;

qgemv_status_t qgemv_set_option(qgemv_handle_t h, qgemv_option_t opt, int64_t value);

/* Describe the launch qgemv_run would make for (fmt, N, K) into `buf` (NUL-terminated,
 * at most `len` bytes): path, grid, block, warps per row, split, ring depth, shared
 * memory.  Returns the same validation status as qgemv_run without launching. */
qgemv_status_t qgemv_describe(qgemv_handle_t h, qgemv_format_t fmt, int64_t N, int64_t K, char* buf,
                              size_t len);

/* Compile-time build marker, checked by the Python binding at load (provenance). */
const char* qgemv_build_marker(void);

/* ---------------------------------------------------------------- layer entry points
 * The general form of the GEMV, y = alpha x.W^T + beta C (Q4_K page, section "What is a
 * GEMV", with C the output's previous contents), and launches over several matrices that
 * share one activation vector: the projections of a decoder layer that read the same x
 * (Q, K and V; the MLP's gate and up), which that page names as the GEMVs of each decoder
 * layer.  The MLP's gate/up pair can be combined as SwiGLU, h = silu(x.Wg^T) * (x.Wu^T)
 * with silu(g) = g / (1 + e^-g) (the gate of Llama/Qwen-style MLPs; the pages name the MLP
 * projections but not their activation). */

/* Output element types: fp32, or fp16 / bf16 rounded to nearest even from the fp32 result. */
typedef enum { QGEMV_OUT_F32 = 0, QGEMV_OUT_F16 = 1, QGEMV_OUT_BF16 = 2 } qgemv_out_t;

/* One matrix of qgemv_run_group.  For row n < N, with r the fp32 result of the row:
 *   swiglu = 0:  r = x . dequant(packed_W)[n, :]
 *   swiglu = 1:  r = silu(x . dequant(packed_W)[n, :]) * (x . dequant(packed_W_up)[n, :])
 *   y[n] = alpha * r + beta * y[n]    (y is not read when beta == 0; one rounding to `out`)
 * packed_W (and packed_W_up): device, qgemv_packed_bytes(fmt, N, K) bytes each, 16-byte
 * aligned; packed_W_up is ignored unless swiglu = 1.  y: device, N elements of type `out`,
 * 16-byte aligned, not overlapping x, any matrix or another problem's y. */
typedef struct {
  qgemv_format_t fmt;
  const void* packed_W;
  const void* packed_W_up;
  int64_t N;
  void* y;
  float alpha;
  float beta;
  qgemv_out_t out;
  int swiglu;
} qgemv_problem_t;

/* Maximum number of matrices in one qgemv_run_group call. */
#define QGEMV_MAX_GROUP 8

/* Runs `count` (1..QGEMV_MAX_GROUP) GEMVs that share x and K, as described by problems[]
 * (host array, read during the call only).  Formats may differ, except that x is bf16 when
 * the matrices are NVFP4 and fp16 otherwise, so NVFP4 cannot be mixed with the other
 * formats (QGEMV_ERR_INVALID_ARG).  K must be a multiple of every format's block length.
 * Matrices the streaming kernel takes (K a multiple of 256 and 16-byte rows) run in ONE
 * launch, each on a share of the CTAs in proportion to its bytes; the others get a
 * warp-per-row launch each.  Validation as qgemv_run for every matrix, all before any
 * launch; also INVALID_ARG for count out of range, a NULL problems, x or y, swiglu not 0/1,
 * swiglu = 1 without packed_W_up, or `out` out of range.  Asynchronous on `stream`, no
 * allocation; uses the handle's workspace like qgemv_run (one call at a time per handle).
 * Deterministic like qgemv_run. */
qgemv_status_t qgemv_run_group(qgemv_handle_t h, const void* x, int64_t K, int count,
                               const qgemv_problem_t* problems, cudaStream_t stream);

/* y = alpha * x . dequant(W)^T + beta * y for one matrix, y of type `out`: qgemv_run_group
 * with one problem (swiglu = 0).  alpha = 1, beta = 0, out = QGEMV_OUT_F32 computes what
 * qgemv_run does (through the grouped kernel, so the last bits may differ). */
qgemv_status_t qgemv_run_ex(qgemv_handle_t h, qgemv_format_t fmt, const void* x, const void* packed_W,
                            int64_t N, int64_t K, float alpha, float beta, void* y, qgemv_out_t out,
                            cudaStream_t stream);

/* ---------------------------------------------------------------- small batches
 * Y = X . dequant(W)^T for M = 1..QGEMV_MAX_BATCH activation vectors at once (the general
 * GEMV of the Q4_K page, "What is a GEMV", with x of shape (M, K) instead of (1, K)): every
 * packed weight is read and decoded once and serves all M vectors.  Every format uses the
 * tensor cores' mma.sync path (decoded weights go straight into the A fragments; the M vectors
 * fill the B operand) when M >= 4, or M >= 2 and N >= 4096 (below that two or three
 * single-vector launches are faster), with rows whose packed length is a multiple of 16 bytes
 * (K a multiple of 2048 for TQ1_0 and Q6_K, of 256 for the others) and M * N * ceil(K / 1024)
 * within the handle's workspace (4 Mi column sums); other calls run the single-vector path
 * once per vector.  Input domain of the tensor-core path: a Q8_0 weight d q is formed in
 * fp16, so weights must be below 65504 in magnitude (quantised model weights are many orders
 * of magnitude smaller); the single-vector path has no such limit. */
#define QGEMV_MAX_BATCH 8

/* x: device, M rows of K 16-bit values (fp16; bf16 for NVFP4), row-major, 16-byte aligned.
 * y: device, M rows of N fp32 values, row-major (y[m * N + n]), 16-byte aligned.
 * packed_W, N, K: as qgemv_run.  1 <= M <= QGEMV_MAX_BATCH, else QGEMV_ERR_INVALID_ARG.
 * Validation, asynchrony, workspace use and determinism as qgemv_run.  Each output obeys the
 * GEMV tolerance of its own vector. */
qgemv_status_t qgemv_run_batch(qgemv_handle_t h, qgemv_format_t fmt, const void* x, int M,
                               const void* packed_W, int64_t N, int64_t K, float* y,
                               cudaStream_t stream);

/* ---------------------------------------------------------------- many rows (prefill)
 * Y = X . dequant(W)^T for any number M >= 1 of activation rows: the matrix-matrix product
 * that the Mojo "fp4_gemv" page sets beside its GEMV (its opening description: a whole prompt
 * goes through the prefill path, a shared-memory tile feeding the matrix unit, while decode
 * at M = 1 is the GEMV).  NVFP4 with M > QGEMV_MAX_BATCH runs on the fifth-generation tensor
 * cores (tcgen05) when K is a multiple of 128 (of 64 when M > 128): tiles of 128 weight rows x
 * 64, 128 or 256 rows of X (by M), X brought in by TMA, the weights dequantised exactly to
 * bf16 into the MMA's A operand in tensor memory (e2m1 times an e4m3 scale has at most 6
 * significant bits), fp32 accumulation in tensor memory, K split over a thread-block cluster
 * when the tiles do not fill the GPU.  Every other call goes through qgemv_run_batch in
 * chunks of QGEMV_MAX_BATCH rows.
 *
 * x: device, M rows of K 16-bit values (fp16; bf16 for NVFP4), row-major, 16-byte aligned.
 * y: device, M rows of N fp32 values, row-major (y[m * N + n]), 16-byte aligned.
 * packed_W, N, K: as qgemv_run.  M < 1 gives QGEMV_ERR_INVALID_ARG; the tensor-core path
 * needs M, K < 2^31 (else QGEMV_ERR_BAD_SHAPE).  Asynchronous on `stream`, allocates
 * nothing; each output obeys the GEMV tolerance of its own row; repeated calls give identical
 * bits.  A wait in the tensor-core kernel that runs past QGEMV_OPT_SPIN_LIMIT_NS sets the
 * handle's error word (read by qgemv_check_error). */
qgemv_status_t qgemv_run_gemm(qgemv_handle_t h, qgemv_format_t fmt, const void* x, int64_t M,
                              const void* packed_W, int64_t N, int64_t K, float* y,
                              cudaStream_t stream);

/* Capacity of qgemv_run_noalloc's scratch, in fp32 column sums: N * ceil(K / 2048) of them. */
#define QGEMV_NOALLOC_MAX_COLUMN_SUMS 262144

/* qgemv_run without a handle and without allocating anything.  (This entry point is part
 * of the library's interface only; the pages that describe the method have no
 * counterpart.)  It exists for callers that may not call cudaMalloc: code that runs under
 * a host application owning all device memory (a plug-in given fixed buffers), processes
 * whose allocator is capped or instrumented so a new allocation would fail or be refused,
 * and latency-critical paths where an allocation's implicit synchronisation is not
 * acceptable.  Those callers cannot use qgemv_create, which allocates the handle's
 * workspace.
 *
 * Computes y = x . dequant(W)^T exactly like qgemv_run with the split-K streaming kernel:
 * every CTA takes one 2048-wide K-column of a range of rows, and the column sums of a row
 * are added in column order.  Arguments, layouts and results are those of qgemv_run;
 * results are bitwise reproducible from call to call.  Shapes: K a multiple of 256 and at
 * most 32768, with packed rows a multiple of 16 bytes (K a multiple of 2048 for Q6_K and
 * TQ1_0), else QGEMV_ERR_BAD_SHAPE.  When K > 2048, N * ceil(K / 2048) must not exceed
 * QGEMV_NOALLOC_MAX_COLUMN_SUMS, else QGEMV_ERR_TOO_LARGE and nothing is launched.
 *
 * Scratch: fixed arrays in the library's device memory (1 MiB of column sums, 4 KiB of
 * counters), which every GPU that loads the library holds until the process exits.  All
 * calls on a device share them and they keep what the last call left: each call first
 * clears the counters with cudaMemsetAsync on `stream`, then launches.  Calls that may run
 * at the same time on the GPU (different streams, or host threads that do not order their
 * streams) race on the scratch and give wrong results; order them on one stream.
 *
 * The first call on a device (the current device) sets that device up: it looks up the
 * scratch arrays' device addresses with cudaGetSymbolAddress and sets the kernels'
 * shared-memory attribute.  Make that first call before any stream capture begins.
 * Asynchronous on `stream`; does not synchronise. */
qgemv_status_t qgemv_run_noalloc(qgemv_format_t fmt, const void* x, const void* packed_W, int64_t N, int64_t K,
                                 float* y, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QGEMV_H_ */
