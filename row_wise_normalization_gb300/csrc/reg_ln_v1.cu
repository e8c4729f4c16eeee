// Register-held kernels: LN, scalar accesses (x and y in different 16-byte phases).
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_ln_v1(int slots, int tpr) { return reg_pick<OP_LN, float, 1, false, false>(slots, tpr); }
}  // namespace rn
