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
// Set-up: the first call on each device (with that device current) looks up
// the array's device address with cudaGetSymbolAddress and keeps it; make
// that first call before any stream capture on the device. No call here
// allocates: no cudaMalloc, no cudaFree, no allocating library routine.
//
// Every call shares the one array, which keeps whatever the last call left
// there. Nothing in it needs to start at zero: the row kernel writes every
// partial row that the column reduction then reads. Calls whose kernels can
// overlap on the GPU (different streams, or different host threads, on the
// same device) race on the array; serialise them, e.g. on one stream.
#include <atomic>
#include <mutex>

#include "rn_params.h"
#include "rownorm.h"

namespace {

static __device__ __align__(256) float g_noalloc_scratch[RN_NOALLOC_SCRATCH_BYTES / 4];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_ptr[kMaxDevices];
std::mutex g_setup_mu;

// The array's address on the current device, looked up once per device.
int scratch_on_current_device(void** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return rn::record_cuda_error(err);
    if (dev < 0 || dev >= kMaxDevices) return rn::record_cuda_error(cudaErrorInvalidDevice);
    void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lk(g_setup_mu);
        p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
        if (!p) {
            err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (err != cudaSuccess || !p)
                return rn::record_cuda_error(err != cudaSuccess ? err : cudaErrorInvalidSymbol);
            g_scratch_ptr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return RN_OK;
}

}  // namespace

extern "C" int ln_bwd_noalloc(const float* dy, const float* x, const float* gamma,
                              const float* mean, const float* rstd, float* dx, float* dgamma,
                              float* dbeta, int64_t rows, int64_t d, void* stream) {
    if (d > RN_NOALLOC_MAX_D) return RN_ERR_SCRATCH;
    void* scratch = nullptr;
    const int st = scratch_on_current_device(&scratch);
    if (st != RN_OK) return st;
    return ln_bwd(dy, x, gamma, mean, rstd, dx, dgamma, dbeta, rows, d, scratch,
                  (size_t)RN_NOALLOC_SCRATCH_BYTES, stream);
}
