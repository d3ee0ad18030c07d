// Streaming-kernel instantiations for one weight format (compiled on their own so the
// library's translation units build in parallel).
#include "qgemv_stream.cuh"

namespace qg {

const void* stream_kernel_q4k(int rows_per_item) {
  switch (rows_per_item) {
    case 1: return reinterpret_cast<const void*>(&stream_kernel<DecQ4K, 1>);
    case 2: return reinterpret_cast<const void*>(&stream_kernel<DecQ4K, 2>);
    default: return reinterpret_cast<const void*>(&stream_kernel<DecQ4K, 4>);
  }
}

}  // namespace qg
