// Register-held kernels: RMS, VEC = 1, every (slots, threads-per-row) pair.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_rms_v1(int slots, int tpr) { return reg_pick<OP_RMS, 1>(slots, tpr); }
}  // namespace rn
