// Register-held kernels: LN, F16 storage, 128-bit vectors, any row phase.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_ln_f16_v8(int slots, int tpr) { return reg_pick<OP_LN, __half, 8, false, false>(slots, tpr); }
}  // namespace rn
