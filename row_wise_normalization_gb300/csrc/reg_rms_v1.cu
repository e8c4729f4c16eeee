// Register-held kernels: RMS, scalar accesses (x and y in different 16-byte phases).
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_rms_v1(int slots, int tpr) { return reg_pick<OP_RMS, float, 1, false, false>(slots, tpr); }
}  // namespace rn
