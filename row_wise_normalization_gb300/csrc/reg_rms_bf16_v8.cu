// Register-held kernels: RMS, BF16 storage, 128-bit vectors, any row phase.
#include "rn_reg.cuh"

namespace rn {
const KernelEntry* reg_entry_rms_bf16_v8(int slots, int tpr) { return reg_pick<OP_RMS, __nv_bfloat16, 8, false, false>(slots, tpr); }
}  // namespace rn
