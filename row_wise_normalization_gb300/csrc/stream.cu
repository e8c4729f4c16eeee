// Streaming (two-read) kernels for any width.
#include "rn_stream.cuh"

namespace rn {
const KernelEntry* stream_entry(int op, int vec) {
    if (op == OP_LN) return vec == 4 ? &StreamInst<OP_LN, 4>::entry : &StreamInst<OP_LN, 1>::entry;
    return vec == 4 ? &StreamInst<OP_RMS, 4>::entry : &StreamInst<OP_RMS, 1>::entry;
}
}  // namespace rn
