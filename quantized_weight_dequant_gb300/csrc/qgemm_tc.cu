// tcgen05 NVFP4 GEMM instantiations: 256, 128 or 64 tokens per tile.
#include "qgemm_tc.cuh"

namespace qg {

const void* tc_kernel_for(int BT) {
  return BT > 128 ? tc_kernel_ptr<256>() : BT > 64 ? tc_kernel_ptr<128>() : tc_kernel_ptr<64>();
}

}  // namespace qg
