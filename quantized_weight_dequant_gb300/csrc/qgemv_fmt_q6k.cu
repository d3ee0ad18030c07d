// Streaming-kernel instantiations for one weight format (compiled on their own so the
// library's translation units build in parallel).
#include "qgemv_stream.cuh"

namespace qg {

const void* stream_kernel_q6k(int R, int D) { return stream_kernel_table<DecQ6K>(R, D); }

}  // namespace qg
