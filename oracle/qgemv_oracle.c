/*
 * Plain CPU fp64 oracle for the batch-1 dequant GEMV  y = x . dequant(W)^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this
 * file: only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Every weight is decoded on its own, straight from the block layout, into a double,
 * and the dot product is a plain left-to-right fp64 sum.  Nothing is factored, fused,
 * reordered or vectorised; the only goal is to be easy to check against the sources:
 *
 *  - "Writing a high performant GEMV + dequant for Metal" (the Q4_K page): the GEMV
 *    y = alpha x.W^T + beta C with alpha = 1, beta = 0 ("What is a GEMV"), the 144-byte
 *    Q4_K block of 8 groups of 32 ("What is a weight block?"), the dequantised weight
 *    w_i = d s_g q_i - dmin m_g ("Compute"), and the byte/nibble/scale positions
 *    that its kernel listing reads ("Kernel code": 6-bit scale unpack with masks
 *    0x3f3f / 0x0f0f / 0xc0c0, quants at byte 16, low nibbles paired with the first
 *    32 activations of each 64, high nibbles with the next 32).
 *  - Mojo "fp4_gemv" page: NVFP4 W4A16, w = e2m1(nibble) * |e4m3 block scale|, one
 *    scale per 16 elements along K (section "Structure").
 *  - "metal: TQ1_0 kernel performance": qs[48] then qh[4] (section 1), digit n of a
 *    byte b as the floor pair floor(3^(n+1) b / 256) - 3 floor(3^n b / 256)
 *    (sections 2 and "Not applicable"), the element order of the dequantize
 *    (16 elements per index il; il < 10 in the 32-byte region at digit il/2,
 *    10 <= il < 15 in the 16-byte region at digit il-10, il = 15 the qh tail),
 *    and w = d (t - 1) for digits {0,1,2} -> {-1,0,+1}.
 *  - Q5_K, Q6_K, Q8_0: only named on the Q4_K page (section "UD-Q4_K_XL"); the
 *    standard ggml layouts are used.  PARITY UNPINNED against ggml itself: no ggml
 *    code or data is available here, so these three decoders are pinned only to the
 *    written layout (hand-built blocks and encoder round trips in the tests).
 *
 * Floating-point inputs (fp16 d, bf16 / fp16 x, E4M3 and E2M1 codes) are decoded by one
 * generic minifloat routine written from the IEEE-754-style definition; the tests pin
 * that routine against numpy/torch on every fp16, bf16, E4M3 and E5M2 code.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_Q4_K 0
#define ORACLE_NVFP4 1
#define ORACLE_TQ1_0 2
#define ORACLE_Q5_K 3
#define ORACLE_Q6_K 4
#define ORACLE_Q8_0 5

#define SPECIAL_NONE 0 /* every code is finite (E2M1) */
#define SPECIAL_IEEE 1 /* top exponent = inf / nan (fp16, bf16, E5M2) */
#define SPECIAL_FN 2   /* only S.1111.111 is nan, no inf (E4M3 "fn") */

/* value = (-1)^s * 2^(E - bias) * (1 + M / 2^m) for E > 0, (-1)^s * 2^(1 - bias) * M / 2^m
 * for E = 0 (subnormal). */
double oracle_minifloat(uint32_t bits, int ebits, int mbits, int bias, int special) {
  uint32_t sign = (bits >> (ebits + mbits)) & 1u;
  uint32_t E = (bits >> mbits) & ((1u << ebits) - 1u);
  uint32_t M = bits & ((1u << mbits) - 1u);
  uint32_t Emax = (1u << ebits) - 1u;
  double v;
  if (special == SPECIAL_IEEE && E == Emax) {
    v = M ? NAN : INFINITY;
  } else if (special == SPECIAL_FN && E == Emax && M == (1u << mbits) - 1u) {
    v = NAN;
  } else if (E == 0) {
    v = ldexp((double)M, 1 - bias - mbits);
  } else {
    v = ldexp((double)((1u << mbits) | M), (int)E - bias - mbits);
  }
  return sign ? -v : v;
}

double oracle_fp16(uint16_t h) { return oracle_minifloat(h, 5, 10, 15, SPECIAL_IEEE); }
double oracle_bf16(uint16_t h) { return oracle_minifloat(h, 8, 7, 127, SPECIAL_IEEE); }
double oracle_e4m3(uint8_t b) { return oracle_minifloat(b, 4, 3, 7, SPECIAL_FN); }
double oracle_e5m2(uint8_t b) { return oracle_minifloat(b, 5, 2, 15, SPECIAL_IEEE); }
double oracle_e2m1(uint8_t c) { return oracle_minifloat(c & 15u, 2, 1, 1, SPECIAL_NONE); }

static double rd_fp16(const uint8_t* p) { return oracle_fp16((uint16_t)(p[0] | (p[1] << 8))); }

/* TQ1_0 digit n (0-based, most significant first) of byte b: the floor pair. */
int oracle_tq1_digit(uint8_t b, int n) {
  long p = 1;
  for (int i = 0; i < n; ++i) p *= 3;
  long hi = (3 * p * (long)b) / 256; /* floor(3^(n+1) b / 256), all terms non-negative */
  long lo = (p * (long)b) / 256;     /* floor(3^n b / 256) */
  return (int)(hi - 3 * lo);
}

/* K-quant 6-bit scale s_g and min m_g of group g from the 12 packed bytes S. */
static void kquant_scale_min(const uint8_t* S, int g, int* s, int* m) {
  if (g < 4) {
    *s = S[g] & 63;
    *m = S[g + 4] & 63;
  } else {
    *s = (S[g + 4] & 0x0F) | ((S[g - 4] >> 6) << 4);
    *m = (S[g + 4] >> 4) | ((S[g] >> 6) << 4);
  }
}

/* Code, scale and min of element i of a block so that w = scale * code - min exactly. */
static void elem_q4k(const uint8_t* p, int i, int* code, double* scale, double* mn) {
  int c = i / 64, h = (i / 32) % 2, j = i % 32, g = i / 32, s, m;
  kquant_scale_min(p + 4, g, &s, &m);
  *code = (p[16 + 32 * c + j] >> (4 * h)) & 15;
  *scale = rd_fp16(p) * s;
  *mn = rd_fp16(p + 2) * m;
}

static void elem_q5k(const uint8_t* p, int i, int* code, double* scale, double* mn) {
  int c = i / 64, h = (i / 32) % 2, j = i % 32, g = i / 32, s, m;
  kquant_scale_min(p + 4, g, &s, &m);
  int lo = (p[48 + 32 * c + j] >> (4 * h)) & 15;
  int hb = (p[16 + j] >> (2 * c + h)) & 1;
  *code = lo | (hb << 4);
  *scale = rd_fp16(p) * s;
  *mn = rd_fp16(p + 2) * m;
}

static void elem_q6k(const uint8_t* p, int i, int* code, double* scale, double* mn) {
  int H = i / 128, r = (i % 128) / 32, l = i % 32;
  int lo = (p[64 * H + l + 32 * (r & 1)] >> (4 * (r >> 1))) & 15;
  int hi = (p[128 + 32 * H + l] >> (2 * r)) & 3;
  int8_t sc = (int8_t)p[192 + 8 * H + 2 * r + l / 16];
  *code = (lo | (hi << 4)) - 32;
  *scale = rd_fp16(p + 208) * sc;
  *mn = 0.0;
}

static void elem_q80(const uint8_t* p, int i, int* code, double* scale, double* mn) {
  *code = (int8_t)p[2 + i];
  *scale = rd_fp16(p);
  *mn = 0.0;
}

static void elem_tq10(const uint8_t* p, int i, int* code, double* scale, double* mn) {
  int t;
  if (i < 160) {
    t = oracle_tq1_digit(p[i % 32], i / 32);
  } else if (i < 240) {
    t = oracle_tq1_digit(p[32 + (i - 160) % 16], (i - 160) / 16);
  } else {
    t = oracle_tq1_digit(p[48 + (i - 240) % 4], (i - 240) / 4);
  }
  *code = t - 1;
  *scale = rd_fp16(p + 52);
  *mn = 0.0;
}

static int block_geometry(int fmt, int* bw, int* bb) {
  switch (fmt) {
    case ORACLE_Q4_K: *bw = 256; *bb = 144; return 0;
    case ORACLE_Q5_K: *bw = 256; *bb = 176; return 0;
    case ORACLE_Q6_K: *bw = 256; *bb = 210; return 0;
    case ORACLE_Q8_0: *bw = 32; *bb = 34; return 0;
    case ORACLE_TQ1_0: *bw = 256; *bb = 54; return 0;
    default: return -1;
  }
}

/* Group length of the per-group scale that oracle_unpack reports. */
int oracle_group_size(int fmt) {
  switch (fmt) {
    case ORACLE_Q4_K: case ORACLE_Q5_K: case ORACLE_Q8_0: return 32;
    case ORACLE_Q6_K: case ORACLE_NVFP4: return 16;
    case ORACLE_TQ1_0: return 256;
    default: return 0;
  }
}

/* code / scale / min of weight (n, k). */
static int elem(int fmt, const uint8_t* W, int64_t N, int64_t K, int64_t n, int64_t k, int* code,
                double* scale, double* mn) {
  if (fmt == ORACLE_NVFP4) {
    uint8_t byte = W[n * (K / 2) + k / 2];
    uint8_t c = (k % 2) ? (byte >> 4) : (byte & 15);
    uint8_t s = W[N * (K / 2) + n * (K / 16) + k / 16];
    *code = (int)lrint(2.0 * oracle_e2m1(c)); /* E2M1 values are multiples of 1/2 */
    *scale = fabs(oracle_e4m3(s)) * 0.5;
    *mn = 0.0;
    return 0;
  }
  int bw, bb;
  if (block_geometry(fmt, &bw, &bb)) return -1;
  const uint8_t* p = W + (n * (K / bw) + k / bw) * bb;
  int i = (int)(k % bw);
  switch (fmt) {
    case ORACLE_Q4_K: elem_q4k(p, i, code, scale, mn); break;
    case ORACLE_Q5_K: elem_q5k(p, i, code, scale, mn); break;
    case ORACLE_Q6_K: elem_q6k(p, i, code, scale, mn); break;
    case ORACLE_Q8_0: elem_q80(p, i, code, scale, mn); break;
    case ORACLE_TQ1_0: elem_tq10(p, i, code, scale, mn); break;
  }
  return 0;
}

/* The dequantised weight itself, computed by each format's own formula. */
static double weight(int fmt, const uint8_t* W, int64_t N, int64_t K, int64_t n, int64_t k) {
  if (fmt == ORACLE_NVFP4) {
    uint8_t byte = W[n * (K / 2) + k / 2];
    uint8_t c = (k % 2) ? (byte >> 4) : (byte & 15);
    uint8_t s = W[N * (K / 2) + n * (K / 16) + k / 16];
    return oracle_e2m1(c) * fabs(oracle_e4m3(s));
  }
  int code;
  double scale, mn;
  elem(fmt, W, N, K, n, k, &code, &scale, &mn);
  if (fmt == ORACLE_Q4_K || fmt == ORACLE_Q5_K) {
    /* w = d * s_g * q - dmin * m_g; scale = d * s_g and mn = dmin * m_g above. */
    return scale * code - mn;
  }
  return scale * code; /* Q6_K: d*sc*(q-32); Q8_0: d*q; TQ1_0: d*(t-1) */
}

static int check_shape(int fmt, int64_t N, int64_t K) {
  if (N < 1 || K < 1) return -1;
  if (fmt == ORACLE_NVFP4) return (K % 16) ? -1 : 0;
  int bw, bb;
  if (block_geometry(fmt, &bw, &bb)) return -1;
  return (K % bw) ? -1 : 0;
}

/* Dequantise rows[0..nrows) into w[nrows][K]. */
int oracle_dequant_rows(int fmt, const uint8_t* W, int64_t N, int64_t K, const int64_t* rows,
                        int64_t nrows, double* w) {
  if (check_shape(fmt, N, K)) return -1;
  for (int64_t r = 0; r < nrows; ++r)
    for (int64_t k = 0; k < K; ++k) w[r * K + k] = weight(fmt, W, N, K, rows[r], k);
  return 0;
}

/* codes [N,K], scales [N, K/G], mins [N, K/G] (mins may be NULL), G = oracle_group_size. */
int oracle_unpack(int fmt, const uint8_t* W, int64_t N, int64_t K, int8_t* codes, double* scales,
                  double* mins) {
  if (check_shape(fmt, N, K)) return -1;
  int G = oracle_group_size(fmt);
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) {
      int code;
      double scale, mn;
      elem(fmt, W, N, K, n, k, &code, &scale, &mn);
      codes[n * K + k] = (int8_t)code;
      if (k % G == 0) {
        scales[n * (K / G) + k / G] = scale;
        if (mins) mins[n * (K / G) + k / G] = mn;
      }
    }
  return 0;
}

/* y[r] = sum_k x_k w(rows[r], k) and S[r] = sum_k |x_k w(rows[r], k)| in fp64.
 * x holds fp16 bits, or bf16 bits for NVFP4. */
int oracle_gemv_rows(int fmt, const uint16_t* x, const uint8_t* W, int64_t N, int64_t K,
                     const int64_t* rows, int64_t nrows, double* y, double* S) {
  if (check_shape(fmt, N, K)) return -1;
  double* xv = (double*)malloc((size_t)K * sizeof(double));
  if (!xv) return -2;
  for (int64_t k = 0; k < K; ++k) xv[k] = (fmt == ORACLE_NVFP4) ? oracle_bf16(x[k]) : oracle_fp16(x[k]);
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t n = rows[r];
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      double t = xv[k] * weight(fmt, W, N, K, n, k);
      acc += t;
      mag += fabs(t);
    }
    y[r] = acc;
    if (S) S[r] = mag;
  }
  free(xv);
  return 0;
}

/* Same over a contiguous row range [r0, r1); y and S indexed from 0. */
int oracle_gemv_range(int fmt, const uint16_t* x, const uint8_t* W, int64_t N, int64_t K, int64_t r0,
                      int64_t r1, double* y, double* S) {
  if (r0 < 0 || r1 > N || r0 > r1) return -1;
  int64_t nr = r1 - r0;
  int64_t* rows = (int64_t*)malloc((size_t)(nr > 0 ? nr : 1) * sizeof(int64_t));
  if (!rows) return -2;
  for (int64_t i = 0; i < nr; ++i) rows[i] = r0 + i;
  int rc = oracle_gemv_rows(fmt, x, W, N, K, rows, nr, y, S);
  free(rows);
  return rc;
}

/* ------------------------------------------------------------------ layer epilogues
 * The general GEMV of the Q4_K page ("What is a GEMV"): y = alpha x.W^T + beta C, which
 * the page then fixes to alpha = 1, beta = 0.  Row n: y[n] = alpha * dot_n + beta * c[n]
 * (c is not read when beta == 0), S[n] = |alpha| * sum_k |x_k w(n, k)|. */
int oracle_gemv_general(int fmt, const uint16_t* x, const uint8_t* W, int64_t N, int64_t K, double alpha,
                        double beta, const double* c, double* y, double* S) {
  int rc = oracle_gemv_range(fmt, x, W, N, K, 0, N, y, S);
  if (rc) return rc;
  for (int64_t n = 0; n < N; ++n) {
    double v = alpha * y[n];
    if (beta != 0.0) v += beta * c[n];
    y[n] = v;
    if (S) S[n] = fabs(alpha) * S[n];
  }
  return 0;
}

/* SiLU (x * logistic(x)), the gate non-linearity of a SwiGLU MLP. */
double oracle_silu(double g) { return g / (1.0 + exp(-g)); }

/* The gated MLP input of a decoder layer (the Q4_K page's "MLPs" of each decoder layer,
 * read as the SwiGLU of Llama/Qwen-style models): two matrices of the same format and
 * shape share x; h[n] = silu(g_n) * u_n with g = x.Wg^T, u = x.Wu^T.  Also returns g, u and
 * their magnitude sums (any of g, u, Sg, Su may be NULL). */
int oracle_swiglu(int fmt, const uint16_t* x, const uint8_t* Wg, const uint8_t* Wu, int64_t N, int64_t K,
                  double* h, double* g, double* u, double* Sg, double* Su) {
  double* gv = (double*)malloc((size_t)N * 4 * sizeof(double));
  if (!gv) return -2;
  double *uv = gv + N, *sg = gv + 2 * N, *su = gv + 3 * N;
  int rc = oracle_gemv_range(fmt, x, Wg, N, K, 0, N, gv, sg);
  if (!rc) rc = oracle_gemv_range(fmt, x, Wu, N, K, 0, N, uv, su);
  if (!rc) {
    for (int64_t n = 0; n < N; ++n) {
      h[n] = oracle_silu(gv[n]) * uv[n];
      if (g) g[n] = gv[n];
      if (u) u[n] = uv[n];
      if (Sg) Sg[n] = sg[n];
      if (Su) Su[n] = su[n];
    }
  }
  free(gv);
  return rc;
}
