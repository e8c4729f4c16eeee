// Register-held kernels: RMS, BF16 storage, scalar accesses.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_rms_bf16_v1(int slots, int tpr) { return reg_pick<OP_RMS, __nv_bfloat16, 1, false, false>(slots, tpr); }
}  // namespace rn
