// Warp-per-row kernels with the parameters staged in shared memory (aligned
// rows, no prefetch: the one-wave instances), f32 storage.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_ps_f32(int op, int slots) {
    return op == OP_LN ? reg_pick_ps<OP_LN, float, 4>(slots) : reg_pick_ps<OP_RMS, float, 4>(slots);
}
}  // namespace rn
