// Warp-per-row kernels with the parameters staged in shared memory (aligned
// rows, no prefetch: the one-wave instances), f32 storage.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_ps_f32(int op, int slots) {
    return op == OP_LN ? reg_pick_ps<OP_LN, float, 4>(slots) : reg_pick_ps<OP_RMS, float, 4>(slots);
}
// The same with prefetch, for LayerNorm rows of 5-6 quads a lane (calls of
// more than one wave's worth of rows).
const KernelEntry* reg_entry_pfps_f32(int op, int slots) {
    if (op != OP_LN) return nullptr;
    if (slots == 5) return reg_ps_entry<OP_LN, float, 4, 5, false>();
    if (slots == 6) return reg_ps_entry<OP_LN, float, 4, 6, false>();
    return nullptr;
}
}  // namespace rn
