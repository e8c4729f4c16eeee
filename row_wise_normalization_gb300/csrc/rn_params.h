// rn_params.h -- kernel arguments and the launcher registry shared by the
// C-ABI translation unit and the kernel instantiation units.
#pragma once

#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

namespace rn {

enum Op : int { OP_LN = 0, OP_RMS = 1 };

// Storage types of x, y and the parameters (statistics are always FP32).
enum Dtype : int { DT_F32 = 0, DT_BF16 = 1, DT_F16 = 2 };
constexpr int dtype_size(int dt) { return dt == DT_F32 ? 4 : 2; }

// Arguments of every row-normalization kernel. For RMSNorm p0 = w, p1 = NULL,
// mean = rstd = NULL. With a residual (r != NULL) the kernels normalise
// h = x + r and write h to `h` when it is not NULL.
struct Params {
    const float* x;
    float* y;
    const float* r;    // residual added to x (residual variants only)
    float* h;          // x + r written back (may be NULL)
    const float* p0;   // gamma or w
    const float* p1;   // beta (LN only)
    float* mean;       // may be NULL
    float* rstd;       // may be NULL
    int64_t rows;
    int64_t d;
    int64_t ldx, ldy;  // row strides of x and y, in elements (>= d; d when contiguous)
    int64_t ldr, ldh;  // row strides of r and h
    float eps;
    unsigned int* err = nullptr;   // device error word (the cluster kernel's bounded waits)
};

// Launches a forward kernel with programmatic stream serialization (see
// pdl_wait in rn_device.cuh): stream order is kept, since the kernel waits
// for the one ahead of it before its first global access, but its launch
// overlaps that kernel's tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned threads, size_t smem,
                       cudaStream_t s, const Args&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// One compiled kernel configuration.
struct KernelEntry {
    const void* fn;        // the __global__ function (for occupancy queries)
    int threads;           // threads per CTA
    int rows_per_cta;      // rows a CTA handles per iteration of its row loop
    int smem_bytes;        // dynamic shared memory per CTA (0: set per launch)
    cudaError_t (*launch)(const Params&, int grid, cudaStream_t);
    // Raises the kernel's dynamic shared memory limit (NULL if not needed).
    cudaError_t (*prepare)(int smem_bytes);
};

// Register-held kernels (warp per row when tpr == 32, a CTA per row above).
// al: x, y and the parameters are 16-byte aligned and d % 4 == 0 (no head or
// tail scalars); pp: the parameter vectors are held in registers across rows
// (requires al, tpr <= 128 and slots <= 6). Returns NULL if the
// configuration was not compiled.
const KernelEntry* reg_entry(int op, int dtype, int vec, int slots, int tpr, bool pp, bool al,
                             bool res);

// Register-held configurations, measured on GB300 (cold L2, same-session
// device-to-device copy as the reference):
//  * warp per row: 4 rows (128 threads) per CTA, prefetching the next row;
//  * CTA per row: the fewest threads (a power of two >= 64) that hold the row
//    in at most kMaxSlots vectors each, prefetching except for the widest
//    slices on 256 threads, where doubling the held registers costs more
//    resident warps than the overlap wins (a thread then holds 32 floats and
//    3 CTAs of 256 per SM keep enough bytes in flight), and where two rows
//    would not fit the 64 registers a thread of a 1024-thread CTA can have
//    (512-thread rows of 8 vectors do prefetch, one CTA per SM: 3-4% faster
//    than two CTAs without, e.g. LayerNorm 4096 x 16384 94.4 -> 90.3 us);
//  * with a residual the prefetched row holds x and the residual apart until
//    it is processed (three slices live), so only slices of <= 4 vectors
//    prefetch;
//  * 16-bit storage moves half the bytes per held float, so for slices of
//    24+ floats on rows of 128+ threads the resident threads (1024 per SM)
//    keep more bytes in flight than a prefetched second row does: no
//    prefetch there (LayerNorm BF16 32768 x 4096: 123 -> 96 us);
//  * parameters held across rows for rows of up to 128 threads holding at
//    most 6 vectors each, when every row starts at the same 16-byte phase
//    (with 8 vectors the held parameters cost a resident CTA per SM) --
//    except the 16-bit slices of 24 floats on 128-thread rows, which run at
//    1024 resident threads per SM where the held parameters would spill
//    (LayerNorm BF16 32768 x 3072: 90.4 -> 76.2 us without them).
constexpr bool reg_prefetch(int vec, int slots, int tpr, bool res = false) {
    return vec > 1 && !(slots * vec >= 32 && tpr == 256) && (!res || slots <= 4) &&
           !(vec == 8 && slots * vec >= 24 && tpr >= 128) &&   // 16-bit: occupancy wins
           (52 + 2 * slots * vec) * tpr <= 65536;   // both rows fit the registers of one CTA
}
// (16-bit warp-per-row rows load their parameters per row: holding them cost
// LayerNorm BF16 4096 x 768 10.8 -> 9.8 us, 8192 x 768 14.4 -> 12.3 us)
constexpr bool reg_may_hold_params(int vec, int slots, int tpr) {
    return vec > 1 && tpr <= 128 && slots * vec <= 24 && !(vec == 8 && tpr == 32) &&
           !(vec == 8 && slots * vec >= 24 && tpr >= 128);   // 16-bit: occupancy wins
}

// Streaming two-read kernels (any width); res: with a residual add (FP32).
const KernelEntry* stream_entry(int op, int dtype, int vec, bool res);

// Shared-memory-staged kernels with `stages` row buffers (1..kMaxStages).
const KernelEntry* staged_entry(int op, int stages);

// Rows split across a thread-block cluster of `cl` CTAs of `threads` threads,
// each holding `slots` quads of the row per thread.
struct ClusterEntry {
    int cl;
    int threads;
    int slots;
    cudaError_t (*launch)(const Params&, int grid, cudaStream_t);
    cudaError_t (*prepare)(int);
    cudaError_t (*max_clusters)(int* n);
};
const ClusterEntry* cluster_entry(int op, int slots, int threads, int cl, bool al);
constexpr int kMaxCluster = 16;
constexpr int kClusterMaxQuads = 1024 * 8 * kMaxCluster;   // 524288 floats per row

// Batched small problems (rn_batched.cuh): one launch over the rows of up to
// kBatchMax independent problems of width <= kBatchMaxD whose x and y share a
// 16-byte phase. The table is the kernel's (__grid_constant__) parameter.
constexpr int kBatchMax = 128;
constexpr int kBatchMaxD = 1024;
constexpr int kBatchThreads = 128;
struct BatchProblem {
    const void* x;     // [rows][d], contiguous
    const void* p0;    // gamma or w
    const void* p1;    // beta (LN) or NULL
    void* y;
    float* mean;       // may be NULL
    float* rstd;       // may be NULL
    int64_t rows;
    int d;             // <= kBatchMaxD
    int al;            // x, y and the parameters 16-byte aligned, d % vector == 0
};
struct BatchParams {
    int n;                         // problems in the table (>= 1, each with rows > 0)
    float eps;
    int64_t start[kBatchMax + 1];  // start[k]: first global row of problem k
    BatchProblem pr[kBatchMax];
};
struct BatchEntry {
    const void* fn;
    int threads;
    cudaError_t (*launch)(const BatchParams&, int grid, cudaStream_t);
};
// slots: vectors per lane, 1, 2, 4 or 8 (FP32) / 1, 2 or 4 (16-bit).
const BatchEntry* batched_entry(int op, int dtype, int slots);

// Arguments of the backward kernels (rn_bwd.cuh). dy, x, dx and p0 are of the
// call's storage type (the float pointers are reinterpreted).
struct BwdParams {
    const float* dy;
    const float* x;
    const float* p0;      // gamma or w
    const float* mean;    // LN: saved mean
    const float* rstd;    // LN: saved rstd
    float* dx;
    float* ws;            // [grid][ws_width] partial column sums (NULL: no parameter grads)
    int64_t rows;
    int64_t d;
    int64_t ws_width;     // 2d (LN: dbeta part, dgamma part) or d (RMS: dw)
    float eps;            // RMS only
    unsigned int* err;    // the device error word (the staged instances' bounded waits)
    int stages;           // staged instances: row buffers in the ring (2..kBwdMaxStages)
};

// Backward kernels. slots: 1-4 (FP32 vectors), 1-2 (16-bit vectors), 1-4 and 8
// (scalars).
struct BwdEntry {
    const void* fn;
    int threads;
    int rows_per_cta;
    int smem_bytes;       // dynamic shared memory per CTA (the 1024-thread instances)
    cudaError_t (*launch)(const BwdParams&, int grid, cudaStream_t);
    // Raises the kernel's dynamic shared memory limit (NULL if not needed).
    cudaError_t (*prepare)();
    int staged;           // 1: a staged instance (ring depth set per call)
};
const BwdEntry* bwd_entry(int op, int dtype, int vec, int slots, int tpr, bool pg);
// The staged form of a CTA-per-row backward instance (vector layout, 256 or
// 512 threads): x and dy rows reach shared memory by bulk copies, ahead of
// the row being reduced. NULL where no staged instance is compiled.
const BwdEntry* bwd_staged_entry(int op, int dtype, int slots, int tpr, bool pg);
// Bytes of shared memory one stage of the staged backward holds: a row of x
// and a row of dy, each padded to 128 bytes.
constexpr int64_t bwd_stage_bytes(int64_t d, int es) { return 2 * ((d * es + 127) / 128 * 128); }
constexpr int kBwdMaxStages = 8;    // row buffers of the staged backward, at most
constexpr int kBwdRingStages = 4;   // the depth the planner asks for (when it fits)
constexpr int kBwdStagedSmemBudget = 232448 - 2048;   // per CTA, dynamic
// out0/out1: the parameter gradients in the storage type `dtype` (or NULL).
cudaError_t column_reduce(int dtype, const float* ws, int64_t rows, int64_t width, int64_t d,
                          void* out0, void* out1, cudaStream_t s);
constexpr int kBwdHeld = 16;   // floats of a row a backward thread holds (x and dy each)
constexpr int kBwdMinRowsPerGroup = 4;   // rows a backward row group takes at least (with grads)

// Records err as this thread's last CUDA error; returns RN_ERR_CUDA.
int record_cuda_error(cudaError_t err);

// ln_bwd's argument checks (sizes, null pointers, alignment, aliasing) for an
// FP32 call, without those of the workspace; returns an rn_status.
int ln_bwd_check_args(const float* dy, const float* x, const float* gamma, const float* mean,
                      const float* rstd, float* dx, float* dgamma, float* dbeta, int64_t rows,
                      int64_t d);

// Launches the bounded-wait self-test (one CTA, a wait nothing completes).
cudaError_t bounded_wait_selftest(unsigned long long limit_ns, cudaStream_t s);

// Reads (and optionally clears) the device error word of the current device.
cudaError_t device_error_word(unsigned int* out, bool clear);
// The device address of that word on the current device (for kernels built in
// other translation units, which receive it as a parameter).
cudaError_t device_error_address(unsigned int** out);

// A process-unique identifier of the CUDA context current on this thread (0
// if none is). A device's primary context gets a new identifier when it is
// created again (after cudaDeviceReset, say), so caches of device addresses
// are keyed on it rather than on the device number.
cudaError_t current_context_id(unsigned long long* id);

// A __device__ variable's address in the current context: `lookup` (which
// calls cudaGetSymbolAddress in the translation unit that defines the
// variable, with the device current) runs the first time the address is
// needed in each context, and the address is kept for later calls, so that
// a call inside a stream capture makes no lookup once one call in that
// context has run outside it.
class SymbolAddressCache {
  public:
    cudaError_t get(void** out, cudaError_t (*lookup)(void**)) {
        int dev = 0;
        cudaError_t err = cudaGetDevice(&dev);
        if (err != cudaSuccess) return err;
        if (dev < 0 || dev >= kDevices) return cudaErrorInvalidDevice;
        unsigned long long ctx = 0;
        if ((err = current_context_id(&ctx)) != cudaSuccess) return err;
        std::lock_guard<std::mutex> lk(mu_);
        Entry& en = e_[dev];
        if (ctx != 0 && en.ctx == ctx && en.ptr) {
            *out = en.ptr;
            return cudaSuccess;
        }
        void* p = nullptr;
        if ((err = lookup(&p)) != cudaSuccess) return err;
        if (!p) return cudaErrorInvalidSymbol;
        // the lookup made the device's primary context current if none was
        if ((err = current_context_id(&ctx)) != cudaSuccess) return err;
        en.ctx = ctx;
        en.ptr = p;
        *out = p;
        return cudaSuccess;
    }

  private:
    static constexpr int kDevices = 64;
    struct Entry {
        unsigned long long ctx = 0;
        void* ptr = nullptr;
    };
    std::mutex mu_;
    Entry e_[kDevices];
};

// Compiled configuration space of the register-held kernels.
constexpr int kMaxSlots = 8;
constexpr int kWarpRowsPerCta = 4;  // rows (warps) per CTA in the warp variant

// Row groups per CTA of the register-held kernels: 4 warp rows, and 3 rows
// of 256 threads for aligned FP32 LayerNorm rows of 8 vectors a thread
// (d 7169-8192). Those run one 768-thread CTA per SM instead of three of
// 256, so that the SM stages gamma and beta in shared memory once (64 KB)
// rather than three times. Everything else: one row per CTA.
constexpr int reg_rows_per_cta(int op, int vec, int slots, int tpr, bool res, bool al) {
    return tpr == 32 ? kWarpRowsPerCta
                     : ((op == 0 && vec == 4 && slots == 8 && tpr == 256 && !res && al) ? 3 : 1);
}
constexpr int kStreamThreads = 512;
constexpr int kStagedThreads = 512;
constexpr int kMaxStages = 4;
// Dynamic shared memory the staged kernel may use for its row buffers: the
// 227 KiB per-CTA limit of sm_100-class GPUs less room for static shared data.
constexpr int kStagedSmemBudget = 232448 - 1024;

}  // namespace rn
