// Register-held kernels: RMS, VEC = 4, every (slots, threads-per-row) pair.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_rms_v4(int slots, int tpr) { return reg_pick<OP_RMS, 4>(slots, tpr); }
}  // namespace rn
