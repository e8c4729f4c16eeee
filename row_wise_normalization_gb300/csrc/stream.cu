// Streaming (two-read) kernels for any width.
#include "rn_stream.cuh"

namespace rn {
template <int OP, bool RES>
const KernelEntry* stream_pick(int vec) {
    return vec == 4 ? &StreamInst<OP, 4, RES>::entry : &StreamInst<OP, 1, RES>::entry;
}

const KernelEntry* stream_entry(int op, int vec, bool res) {
    if (op == OP_LN) return res ? stream_pick<OP_LN, true>(vec) : stream_pick<OP_LN, false>(vec);
    return res ? stream_pick<OP_RMS, true>(vec) : stream_pick<OP_RMS, false>(vec);
}
}  // namespace rn
