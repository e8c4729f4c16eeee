// Warp-per-row kernels with the parameters staged in shared memory (aligned
// rows, no prefetch: the one-wave instances), f16 storage.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_ps_f16(int op, int slots) {
    return op == OP_LN ? reg_pick_ps<OP_LN, __half, 8>(slots) : reg_pick_ps<OP_RMS, __half, 8>(slots);
}
}  // namespace rn
