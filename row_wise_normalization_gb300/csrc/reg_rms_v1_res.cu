// Register-held kernels with a residual add: RMS, family v1.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_rms_v1_res(int slots, int tpr) { return reg_pick<OP_RMS, float, 1,false,false, true>(slots, tpr); }
}  // namespace rn
