// Backward kernels (FP32 storage), the dispatch over storage types and the
// column reduction of parameter-gradient partials.
#include "rn_bwd.cuh"

namespace rn {

const BwdEntry* bwd_entry_bf16(int op, int vec, int slots, int tpr, bool pg);
const BwdEntry* bwd_entry_f16(int op, int vec, int slots, int tpr, bool pg);
const BwdEntry* bwd_staged_entry_bf16(int op, int slots, int tpr, bool pg);
const BwdEntry* bwd_staged_entry_f16(int op, int slots, int tpr, bool pg);
cudaError_t column_reduce_bf16(const float* ws, int64_t rows, int64_t width, int64_t d,
                               void* out0, void* out1, cudaStream_t s);
cudaError_t column_reduce_f16(const float* ws, int64_t rows, int64_t width, int64_t d,
                              void* out0, void* out1, cudaStream_t s);

const BwdEntry* bwd_entry(int op, int dtype, int vec, int slots, int tpr, bool pg) {
    switch (dtype) {
        case DT_F32: return bwd_pick_type<float>(op, vec, slots, tpr, pg);
        case DT_BF16: return bwd_entry_bf16(op, vec, slots, tpr, pg);
        case DT_F16: return bwd_entry_f16(op, vec, slots, tpr, pg);
        default: return nullptr;
    }
}

const BwdEntry* bwd_staged_entry(int op, int dtype, int slots, int tpr, bool pg) {
    switch (dtype) {
        case DT_F32: return bwd_staged_pick_type<float>(op, slots, tpr, pg);
        case DT_BF16: return bwd_staged_entry_bf16(op, slots, tpr, pg);
        case DT_F16: return bwd_staged_entry_f16(op, slots, tpr, pg);
        default: return nullptr;
    }
}

cudaError_t column_reduce(int dtype, const float* ws, int64_t rows, int64_t width, int64_t d,
                          void* out0, void* out1, cudaStream_t s) {
    switch (dtype) {
        case DT_BF16: return column_reduce_bf16(ws, rows, width, d, out0, out1, s);
        case DT_F16: return column_reduce_f16(ws, rows, width, d, out0, out1, s);
        default: return column_reduce_t<float>(ws, rows, width, d, out0, out1, s);
    }
}

}  // namespace rn
