// Small-batch kernel instantiations (every format; ring depths 2 and 3).
#include "qgemv_batch.cuh"

namespace qg {

const void* batch_kernel_for(int f, int D) {
  switch (f) {
    case F_Q4K: return batch_kernel_table<BatchQ4K>(D);
    case F_Q5K: return batch_kernel_table<BatchQ5K>(D);
    case F_Q80: return batch_kernel_table<BatchQ80>(D);
    case F_NVFP4: return batch_kernel_table<BatchNVFP4>(D);
    case F_TQ10: return batch_kernel_table<BatchTQ10>(D);
    case F_Q6K: return batch_kernel_table<BatchQ6K>(D);
  }
  return nullptr;
}

size_t batch_smem_bytes(int f, int warps, int D) {
  switch (f) {
    case F_Q4K: return batch_smem(warps, D, batch_slice<BatchQ4K>()).total;
    case F_Q5K: return batch_smem(warps, D, batch_slice<BatchQ5K>()).total;
    case F_Q80: return batch_smem(warps, D, batch_slice<BatchQ80>()).total;
    case F_NVFP4: return batch_smem(warps, D, batch_slice<BatchNVFP4>()).total;
    case F_TQ10: return batch_smem(warps, D, batch_slice<BatchTQ10>()).total;
    case F_Q6K: return batch_smem(warps, D, batch_slice<BatchQ6K>()).total;
  }
  return 0;
}

}  // namespace qg
