// One-format grouped-kernel instantiations (the
// matrices of a grouped launch share one format), kept apart from the single-matrix
// kernels' translation units.
#include "qgemv_stream.cuh"

namespace qg {

const void* group_kernel_q80(int R, int D) { return group_kernel_1_table<DecQ80, false>(R, D); }
const void* group_kernel_tq10(int R, int D) { return group_kernel_1_table<DecTQ10, false>(R, D); }
const void* group_kernel_nvfp4(int R, int D) { return group_kernel_1_table<DecNVFP4, false>(R, D); }

}  // namespace qg
