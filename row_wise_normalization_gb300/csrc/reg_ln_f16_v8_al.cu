// Register-held kernels: LN, F16 storage, every row whole aligned vectors.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_ln_f16_v8_al(int slots, int tpr) { return reg_pick<OP_LN, __half, 8, false, true>(slots, tpr); }
}  // namespace rn
