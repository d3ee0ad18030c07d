// Grouped-kernel instantiations with 2 rows per stage (every format in one kernel; compiled
// on their own so the library's translation units build in parallel).
#include "qgemv_stream.cuh"

namespace qg {

const void* group_kernel_r2(int D) {
  switch (D) {
    case 2: return reinterpret_cast<const void*>(&group_kernel<2, 2>);
    case 3: return reinterpret_cast<const void*>(&group_kernel<2, 3>);
    default: return reinterpret_cast<const void*>(&group_kernel<2, 4>);
  }
}

}  // namespace qg
