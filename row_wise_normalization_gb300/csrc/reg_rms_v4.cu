// Register-held kernels: RMS, 128-bit vectors, any row phase (head peel, scalar tail).
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_rms_v4(int slots, int tpr) { return reg_pick<OP_RMS, float, 4, false, false>(slots, tpr); }
}  // namespace rn
