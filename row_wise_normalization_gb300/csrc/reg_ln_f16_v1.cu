// Register-held kernels: LN, F16 storage, scalar accesses.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_ln_f16_v1(int slots, int tpr) { return reg_pick<OP_LN, __half, 1, false, false>(slots, tpr); }
}  // namespace rn
