// Register-held kernels: RMS, F16 storage, aligned rows, parameters held across rows.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_rms_f16_v8_pp(int slots, int tpr) { return reg_pick<OP_RMS, __half, 8, true, true>(slots, tpr); }
}  // namespace rn
