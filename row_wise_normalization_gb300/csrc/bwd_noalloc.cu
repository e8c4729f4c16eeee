// ln_bwd_noalloc: LayerNorm backward with the parameter-gradient partials in
// a static device array instead of a caller-supplied workspace.
//
// Some callers cannot allocate device memory at the point where they need
// the backward: a serving or training process whose caching allocator has
// already reserved nearly all of HBM (a fresh cudaMalloc would fail or
// fragment that pool), a latency-sensitive loop where cudaFree's device-wide
// synchronisation would stall the other streams, or plain C code with no
// allocator of its own. This entry point takes the same inputs and outputs
// as ln_bwd and uses, as its workspace, one file-scope array that every GPU
// loading the library holds until the process exits.
//
// Set-up: the first call that needs the array in a CUDA context (with that
// context's device current) looks up the array's device address with
// cudaGetSymbolAddress, checks the result and keeps the address for that
// context; make that first call before any stream capture on the device. A
// context created anew for the device (after cudaDeviceReset, say) gets a
// lookup of its own, since the address is kept per context, not per device
// number. No call here allocates: no cudaMalloc, no cudaFree, no allocating
// library routine.
//
// Every call shares the one array, which keeps whatever the last call left
// there. Nothing in it needs to start at zero: the row kernel writes every
// partial row that the column reduction then reads. Calls whose kernels can
// overlap on the GPU (different streams, or different host threads, on the
// same device) race on the array; serialise them, e.g. on one stream.
#include "rn_params.h"
#include "rownorm.h"

namespace {

static __device__ __align__(256) float g_noalloc_scratch[RN_NOALLOC_SCRATCH_BYTES / 4];

// The array's address in the current context (looked up once per context).
int scratch_on_current_device(void** out) {
    static rn::SymbolAddressCache cache;
    const cudaError_t err = cache.get(out, [](void** p) {
        return cudaGetSymbolAddress(p, g_noalloc_scratch);
    });
    return err == cudaSuccess ? RN_OK : rn::record_cuda_error(err);
}

}  // namespace

extern "C" int ln_bwd_noalloc(const float* dy, const float* x, const float* gamma,
                              const float* mean, const float* rstd, float* dx, float* dgamma,
                              float* dbeta, int64_t rows, int64_t d, void* stream) {
    // the checks every backward call makes come first, so that errors (and
    // rows == 0, which only zeroes the requested gradients) are reported as
    // ln_bwd reports them
    const int st = rn::ln_bwd_check_args(dy, x, gamma, mean, rstd, dx, dgamma, dbeta, rows, d);
    if (st != RN_OK) return st;
    const bool pg = dgamma || dbeta;
    if (rows == 0 || !pg)   // no partials: the scratch is not needed
        return ln_bwd(dy, x, gamma, mean, rstd, dx, dgamma, dbeta, rows, d, nullptr, 0, stream);
    if (d > RN_NOALLOC_MAX_D) return RN_ERR_SCRATCH;
    void* scratch = nullptr;
    const int sst = scratch_on_current_device(&scratch);
    if (sst != RN_OK) return sst;
    return ln_bwd(dy, x, gamma, mean, rstd, dx, dgamma, dbeta, rows, d, scratch,
                  (size_t)RN_NOALLOC_SCRATCH_BYTES, stream);
}
