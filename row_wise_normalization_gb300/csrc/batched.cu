// Batched small problems: one launch for many independent normalizations.
#include "rn_batched.cuh"

namespace rn {

const BatchEntry* batched_entry(int op, int dtype, int slots) {
    if (op == OP_LN) {
        switch (dtype) {
            case DT_F32: return batch_pick<OP_LN, float>(slots);
            case DT_BF16: return batch_pick<OP_LN, __nv_bfloat16>(slots);
            case DT_F16: return batch_pick<OP_LN, __half>(slots);
            default: return nullptr;
        }
    }
    switch (dtype) {
        case DT_F32: return batch_pick<OP_RMS, float>(slots);
        case DT_BF16: return batch_pick<OP_RMS, __nv_bfloat16>(slots);
        case DT_F16: return batch_pick<OP_RMS, __half>(slots);
        default: return nullptr;
    }
}

}  // namespace rn
