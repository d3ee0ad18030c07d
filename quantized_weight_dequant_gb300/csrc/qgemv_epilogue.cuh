// Output stage shared by the kernels: the general GEMV epilogue out = alpha r + beta out
// ("Writing a high performant GEMV + dequant for Metal", section "What is a GEMV":
// y = alpha x.W^T + beta C, with C the output's previous contents) in fp32, fp16 or bf16,
// and the SiLU of a SwiGLU gate.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

namespace qg {

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// out[n] = alpha * r + beta * out[n] in the output type (one rounding from fp32).
__device__ __forceinline__ void emit_out(void* y, int ydt, float alpha, float beta, int64_t n, float r) {
  float o = alpha * r;
  if (ydt == 0) {
    float* q = static_cast<float*>(y) + n;
    if (beta != 0.f) o = fmaf(beta, *q, o);
    *q = o;
  } else if (ydt == 1) {
    __half* q = static_cast<__half*>(y) + n;
    if (beta != 0.f) o = fmaf(beta, __half2float(*q), o);
    *q = __float2half_rn(o);
  } else {
    __nv_bfloat16* q = static_cast<__nv_bfloat16*>(y) + n;
    if (beta != 0.f) o = fmaf(beta, __bfloat162float(*q), o);
    *q = __float2bfloat16_rn(o);
  }
}
}  // namespace qg
