// One-format grouped-kernel instantiations with SwiGLU pairs compiled in (the
// matrices of a grouped launch share one format), kept apart from the single-matrix
// kernels' translation units.
#include "qgemv_stream.cuh"

namespace qg {

const void* group_kernel_pair_q4k(int R, int D) { return group_kernel_1_table<DecQ4K, true>(R, D); }
const void* group_kernel_pair_q5k(int R, int D) { return group_kernel_1_table<DecQ5K, true>(R, D); }
const void* group_kernel_pair_q6k(int R, int D) { return group_kernel_1_table<DecQ6K, true>(R, D); }

}  // namespace qg
