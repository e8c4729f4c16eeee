// Register-held kernels: RMS, every row 16-byte aligned, parameters held,
// compiled without prefetch (the one-wave instances).
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_rms_v4_pp_nopf(int slots, int tpr) { return reg_pick<OP_RMS, float, 4, true, true, false, true>(slots, tpr); }
}  // namespace rn
