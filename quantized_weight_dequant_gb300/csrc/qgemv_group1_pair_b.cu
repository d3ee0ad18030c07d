// One-format grouped-kernel instantiations with SwiGLU pairs compiled in (the
// matrices of a grouped launch share one format), kept apart from the single-matrix
// kernels' translation units.
#include "qgemv_stream.cuh"

namespace qg {

const void* group_kernel_pair_q80(int R, int D) { return group_kernel_1_table<DecQ80, true>(R, D); }
const void* group_kernel_pair_tq10(int R, int D) { return group_kernel_1_table<DecTQ10, true>(R, D); }
const void* group_kernel_pair_nvfp4(int R, int D) { return group_kernel_1_table<DecNVFP4, true>(R, D); }

}  // namespace qg
