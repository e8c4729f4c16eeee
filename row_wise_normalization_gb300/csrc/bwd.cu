// Backward kernels and the column reduction of parameter-gradient partials.
#include "rn_bwd.cuh"

namespace rn {

const BwdEntry* bwd_entry(int op, int vec, int slots, int tpr, bool pg) {
    if (op == OP_LN) {
        if (vec == 4) return pg ? bwd_pick<OP_LN, 4, true>(slots, tpr) : bwd_pick<OP_LN, 4, false>(slots, tpr);
        return pg ? bwd_pick<OP_LN, 1, true>(slots, tpr) : bwd_pick<OP_LN, 1, false>(slots, tpr);
    }
    if (vec == 4) return pg ? bwd_pick<OP_RMS, 4, true>(slots, tpr) : bwd_pick<OP_RMS, 4, false>(slots, tpr);
    return pg ? bwd_pick<OP_RMS, 1, true>(slots, tpr) : bwd_pick<OP_RMS, 1, false>(slots, tpr);
}

cudaError_t column_reduce(const float* ws, int64_t rows, int64_t width, int64_t d, float* out0,
                          float* out1, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((width + kReduceCols - 1) / kReduceCols));
    cfg.blockDim = dim3(kReduceCols * kReduceSlices);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, column_reduce_kernel, ws, rows, width, d, out0, out1);
}

}  // namespace rn
