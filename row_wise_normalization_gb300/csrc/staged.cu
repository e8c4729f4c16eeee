// Shared-memory-staged (bulk-copy) kernels and the device error word.
#include "rn_staged.cuh"

namespace rn {

template <int OP>
const KernelEntry* staged_pick(int stages) {
    switch (stages) {
        case 1: return &StagedInst<OP, kStagedThreads, 1>::entry;
        case 2: return &StagedInst<OP, kStagedThreads, 2>::entry;
        case 3: return &StagedInst<OP, kStagedThreads, 3>::entry;
        case 4: return &StagedInst<OP, kStagedThreads, 4>::entry;
        default: return nullptr;
    }
}

const KernelEntry* staged_entry(int op, int stages) {
    return op == OP_LN ? staged_pick<OP_LN>(stages) : staged_pick<OP_RMS>(stages);
}

cudaError_t bounded_wait_selftest(unsigned long long limit_ns, cudaStream_t s) {
    bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns);
    return cudaGetLastError();
}

cudaError_t device_error_word(unsigned int* out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_device_error, sizeof(unsigned int));
    if (e != cudaSuccess || !clear) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int));
}

// Looked up once per CUDA context and kept, so that later calls (a stream
// capture among them) make no runtime query; a context created anew (after a
// device reset) gets a fresh lookup.
cudaError_t device_error_address(unsigned int** out) {
    static SymbolAddressCache cache;
    void* p = nullptr;
    const cudaError_t e = cache.get(&p, [](void** q) {
        return cudaGetSymbolAddress(q, g_device_error);
    });
    if (e != cudaSuccess) return e;
    *out = static_cast<unsigned int*>(p);
    return cudaSuccess;
}

}  // namespace rn
