// Grouped-kernel instantiations with 4 rows per stage (every format in one kernel; compiled
// on their own so the library's translation units build in parallel).
#include "qgemv_stream.cuh"

namespace qg {

const void* group_kernel_r4(int D) {
  switch (D) {
    case 2: return reinterpret_cast<const void*>(&group_kernel<4, 2>);
    case 3: return reinterpret_cast<const void*>(&group_kernel<4, 3>);
    default: return reinterpret_cast<const void*>(&group_kernel<4, 4>);
  }
}

}  // namespace qg
