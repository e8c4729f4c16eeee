// Register-held kernels: LN, BF16 storage, aligned rows, parameters held across rows.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_ln_bf16_v8_pp(int slots, int tpr) { return reg_pick<OP_LN, __nv_bfloat16, 8, true, true>(slots, tpr); }
}  // namespace rn
