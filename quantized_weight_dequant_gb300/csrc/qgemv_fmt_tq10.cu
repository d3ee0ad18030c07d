// Streaming-kernel instantiations for one weight format (compiled on their own so the
// library's translation units build in parallel).
#include "qgemv_stream.cuh"

namespace qg {

const void* stream_kernel_tq10(int rows_per_item) {
  switch (rows_per_item) {
    case 1: return reinterpret_cast<const void*>(&stream_kernel<DecTQ10, 1>);
    case 2: return reinterpret_cast<const void*>(&stream_kernel<DecTQ10, 2>);
    default: return reinterpret_cast<const void*>(&stream_kernel<DecTQ10, 4>);
  }
}

}  // namespace qg
