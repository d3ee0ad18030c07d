// One-format grouped-kernel instantiations (the
// matrices of a grouped launch share one format), kept apart from the single-matrix
// kernels' translation units.
#include "qgemv_stream.cuh"

namespace qg {

const void* group_kernel_q4k(int R, int D) { return group_kernel_1_table<DecQ4K, false>(R, D); }
const void* group_kernel_q5k(int R, int D) { return group_kernel_1_table<DecQ5K, false>(R, D); }
const void* group_kernel_q6k(int R, int D) { return group_kernel_1_table<DecQ6K, false>(R, D); }

}  // namespace qg
