/* A plain C caller of the library: no Python, no PyTorch.  It reads a packed weight matrix
 * and an activation vector (files written by the test), runs qgemv_run through the C ABI on
 * device buffers it allocates itself, and compares every output with the CPU oracle
 * (oracle_gemv_range, linked from the oracle's own library) within the GEMV tolerance
 * |y - y_ref| <= 2e-3 * sum|x w| + 1e-5.  It also checks that invalid arguments are refused
 * with their documented status before anything is launched.
 *
 * usage: c_abi_program FMT N K weights.bin x.bin      (exit status 0: every check passed) */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "qgemv.h"

int oracle_gemv_range(int fmt, const uint16_t* x, const uint8_t* W, int64_t N, int64_t K, int64_t r0, int64_t r1,
                      double* y, double* S);

static void* read_file(const char* path, size_t expect) {
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  void* buf = malloc(expect ? expect : 1);
  size_t got = buf ? fread(buf, 1, expect, f) : 0;
  fclose(f);
  if (got != expect) {
    free(buf);
    return NULL;
  }
  return buf;
}

#define CHECK(cond, ...)            \
  do {                              \
    if (!(cond)) {                  \
      fprintf(stderr, __VA_ARGS__); \
      fputc('\n', stderr);          \
      return 1;                     \
    }                               \
  } while (0)

int main(int argc, char** argv) {
  CHECK(argc == 6, "usage: %s FMT N K weights.bin x.bin", argv[0]);
  const qgemv_format_t fmt = (qgemv_format_t)atoi(argv[1]);
  const int64_t N = atoll(argv[2]), K = atoll(argv[3]);
  const size_t wbytes = qgemv_packed_bytes(fmt, N, K);
  CHECK(wbytes > 0, "qgemv_packed_bytes refused fmt %d N %lld K %lld", (int)fmt, (long long)N, (long long)K);
  uint8_t* W = (uint8_t*)read_file(argv[4], wbytes);
  uint16_t* x = (uint16_t*)read_file(argv[5], (size_t)K * 2);
  CHECK(W && x, "cannot read the input files");

  qgemv_handle_t h = NULL;
  CHECK(qgemv_create(&h, 0) == QGEMV_OK && h, "qgemv_create failed");
  void *dW = NULL, *dx = NULL, *dy = NULL;
  CHECK(cudaMalloc(&dW, wbytes) == cudaSuccess && cudaMalloc(&dx, (size_t)K * 2) == cudaSuccess &&
            cudaMalloc(&dy, (size_t)N * 4) == cudaSuccess,
        "cudaMalloc failed");
  CHECK(cudaMemcpy(dW, W, wbytes, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(dx, x, (size_t)K * 2, cudaMemcpyHostToDevice) == cudaSuccess,
        "cudaMemcpy to the device failed");
  cudaStream_t s;
  CHECK(cudaStreamCreate(&s) == cudaSuccess, "cudaStreamCreate failed");

  /* refused before any launch, with the documented statuses */
  CHECK(qgemv_run(h, fmt, NULL, dW, N, K, (float*)dy, s) == QGEMV_ERR_INVALID_ARG, "null x was not refused");
  CHECK(qgemv_run(h, fmt, dx, dW, 0, K, (float*)dy, s) == QGEMV_ERR_BAD_SHAPE, "N = 0 was not refused");
  CHECK(qgemv_run(h, fmt, dx, dW, N, K + 1, (float*)dy, s) == QGEMV_ERR_BAD_SHAPE, "a ragged K was not refused");
  CHECK(qgemv_run(h, fmt, (const uint8_t*)dx + 2, dW, N, K, (float*)dy, s) == QGEMV_ERR_MISALIGNED,
        "a misaligned x was not refused");
  CHECK(qgemv_status_string(QGEMV_ERR_BAD_SHAPE) != NULL, "no status string");

  CHECK(qgemv_run(h, fmt, dx, dW, N, K, (float*)dy, s) == QGEMV_OK, "qgemv_run failed");
  CHECK(qgemv_check_error(h, s) == QGEMV_OK, "device error word set");
  float* y = (float*)malloc((size_t)N * 4);
  double* yr = (double*)malloc((size_t)N * 8);
  double* S = (double*)malloc((size_t)N * 8);
  CHECK(y && yr && S, "malloc failed");
  CHECK(cudaMemcpy(y, dy, (size_t)N * 4, cudaMemcpyDeviceToHost) == cudaSuccess, "cudaMemcpy to the host failed");
  CHECK(oracle_gemv_range((int)fmt, x, W, N, K, 0, N, yr, S) == 0, "the oracle refused the inputs");
  int64_t bad = 0;
  double worst = 0.0;
  for (int64_t n = 0; n < N; ++n) {
    const double tol = 2e-3 * S[n] + 1e-5, err = fabs((double)y[n] - yr[n]);
    if (!(err <= tol)) {
      if (bad < 5) fprintf(stderr, "row %lld: %.9g against %.9g (tolerance %.3g)\n", (long long)n, y[n], yr[n], tol);
      ++bad;
    }
    if (err / tol > worst) worst = err / tol;
  }
  CHECK(bad == 0, "%lld of %lld rows outside the tolerance", (long long)bad, (long long)N);
  printf("ok: fmt %d, %lld x %lld, largest error %.3g of the tolerance\n", (int)fmt, (long long)N, (long long)K, worst);

  cudaStreamDestroy(s);
  cudaFree(dW);
  cudaFree(dx);
  cudaFree(dy);
  CHECK(qgemv_destroy(h) == QGEMV_OK, "qgemv_destroy failed");
  free(W);
  free(x);
  free(y);
  free(yr);
  free(S);
  return 0;
}
