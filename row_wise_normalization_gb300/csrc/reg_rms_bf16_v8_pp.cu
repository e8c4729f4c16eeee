// Register-held kernels: RMS, BF16 storage, aligned rows, parameters held across rows.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_rms_bf16_v8_pp(int slots, int tpr) { return reg_pick<OP_RMS, __nv_bfloat16, 8, true, true>(slots, tpr); }
}  // namespace rn
