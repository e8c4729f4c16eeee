// Register-held kernels: LN, every row 16-byte aligned, parameters per row,
// compiled without prefetch (the one-wave instances).
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_ln_v4_al_nopf(int slots, int tpr) { return reg_pick<OP_LN, float, 4, false, true, false, true>(slots, tpr); }
}  // namespace rn
