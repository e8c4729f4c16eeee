// Backward kernels with FP16 storage (FP32 arithmetic and partials).
#include "rn_bwd.cuh"

namespace rn {

const BwdEntry* bwd_entry_f16(int op, int vec, int slots, int tpr, bool pg) {
    return bwd_pick_type<__half>(op, vec, slots, tpr, pg);
}

const BwdEntry* bwd_staged_entry_f16(int op, int slots, int tpr, bool pg) {
    return bwd_staged_pick_type<__half>(op, slots, tpr, pg);
}

cudaError_t column_reduce_f16(const float* ws, int64_t rows, int64_t width, int64_t d,
                               void* out0, void* out1, cudaStream_t s) {
    return column_reduce_t<__half>(ws, rows, width, d, out0, out1, s);
}

}  // namespace rn
