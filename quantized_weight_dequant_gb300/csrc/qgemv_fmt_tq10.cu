// Streaming-kernel instantiations for one weight format (compiled on their own so the
// library's translation units build in parallel).
#include "qgemv_stream.cuh"

namespace qg {

const void* stream_kernel_tq10(int R, int D) { return stream_kernel_table<DecTQ10>(R, D); }

}  // namespace qg
