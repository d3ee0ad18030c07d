// Small-batch kernel instantiations (Q4_K, Q5_K, Q8_0 and NVFP4; ring depths 2 and 3).
#include "qgemv_batch.cuh"

namespace qg {

const void* batch_kernel_for(int f, int D) {
  switch (f) {
    case F_Q4K: return batch_kernel_table<BatchQ4K>(D);
    case F_Q5K: return batch_kernel_table<BatchQ5K>(D);
    case F_Q80: return batch_kernel_table<BatchQ80>(D);
    case F_NVFP4: return batch_kernel_table<BatchNVFP4>(D);
  }
  return nullptr;
}

size_t batch_smem_bytes(int f, int warps, int D) {
  switch (f) {
    case F_Q4K: return batch_smem(warps, D, batch_slice<BatchQ4K>()).total;
    case F_Q5K: return batch_smem(warps, D, batch_slice<BatchQ5K>()).total;
    case F_Q80: return batch_smem(warps, D, batch_slice<BatchQ80>()).total;
    case F_NVFP4: return batch_smem(warps, D, batch_slice<BatchNVFP4>()).total;
  }
  return 0;
}

}  // namespace qg
