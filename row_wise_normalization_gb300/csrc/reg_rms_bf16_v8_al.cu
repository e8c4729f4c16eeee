// Register-held kernels: RMS, BF16 storage, every row whole aligned vectors.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_rms_bf16_v8_al(int slots, int tpr) { return reg_pick<OP_RMS, __nv_bfloat16, 8, false, true>(slots, tpr); }
}  // namespace rn
