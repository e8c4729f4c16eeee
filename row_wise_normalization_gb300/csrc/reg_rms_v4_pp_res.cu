// Register-held kernels with a residual add: RMS, family v4_pp.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_rms_v4_pp_res(int slots, int tpr) { return reg_pick<OP_RMS, float, 4,true,true, true>(slots, tpr); }
}  // namespace rn
