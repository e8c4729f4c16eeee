// Register-held kernels with a residual add: RMS, family v4.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_rms_v4_res(int slots, int tpr) { return reg_pick<OP_RMS, float, 4,false,false, true>(slots, tpr); }
}  // namespace rn
