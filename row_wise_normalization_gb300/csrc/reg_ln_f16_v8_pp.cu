// Register-held kernels: LN, F16 storage, aligned rows, parameters held across rows.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_ln_f16_v8_pp(int slots, int tpr) { return reg_pick<OP_LN, __half, 8, true, true>(slots, tpr); }
}  // namespace rn
