// Register-held kernels: RMS, F16 storage, every row whole aligned vectors.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_rms_f16_v8_al(int slots, int tpr) { return reg_pick<OP_RMS, __half, 8, false, true>(slots, tpr); }
}  // namespace rn
