// Streaming (two-read) kernels for any width.
#include "rn_stream.cuh"

namespace rn {
template <int OP, bool RES>
const KernelEntry* stream_pick(int vec) {
    return vec == 4 ? &StreamInst<OP, float, 4, RES>::entry : &StreamInst<OP, float, 1, RES>::entry;
}

template <int OP, typename T>
const KernelEntry* stream_pick16(int vec) {
    return vec == 8 ? &StreamInst<OP, T, 8, false>::entry : &StreamInst<OP, T, 1, false>::entry;
}

const KernelEntry* stream_entry(int op, int dtype, int vec, bool res) {
    if (dtype == DT_BF16) {
        if (res) return nullptr;
        return op == OP_LN ? stream_pick16<OP_LN, __nv_bfloat16>(vec)
                           : stream_pick16<OP_RMS, __nv_bfloat16>(vec);
    }
    if (dtype == DT_F16) {
        if (res) return nullptr;
        return op == OP_LN ? stream_pick16<OP_LN, __half>(vec) : stream_pick16<OP_RMS, __half>(vec);
    }
    if (op == OP_LN) return res ? stream_pick<OP_LN, true>(vec) : stream_pick<OP_LN, false>(vec);
    return res ? stream_pick<OP_RMS, true>(vec) : stream_pick<OP_RMS, false>(vec);
}
}  // namespace rn
