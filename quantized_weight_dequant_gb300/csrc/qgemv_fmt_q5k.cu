// Streaming-kernel instantiations for one weight format (compiled on their own so the
// library's translation units build in parallel).
#include "qgemv_stream.cuh"

namespace qg {

const void* stream_kernel_q5k(int R, int D) { return stream_kernel_table<DecQ5K>(R, D); }

}  // namespace qg
