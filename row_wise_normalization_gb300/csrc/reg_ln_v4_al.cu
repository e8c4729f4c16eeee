// Register-held kernels: LN, every row 16-byte aligned whole vectors, parameters per row.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_ln_v4_al(int slots, int tpr) { return reg_pick<OP_LN, float, 4, false, true>(slots, tpr); }
}  // namespace rn
