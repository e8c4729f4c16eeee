// rn_params.h -- kernel arguments and the launcher registry shared by the
// C-ABI translation unit and the kernel instantiation units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace rn {

enum Op : int { OP_LN = 0, OP_RMS = 1 };

// Arguments of every row-normalization kernel. For RMSNorm p0 = w, p1 = NULL,
// mean = rstd = NULL.
struct Params {
    const float* x;
    float* y;
    const float* p0;   // gamma or w
    const float* p1;   // beta (LN only)
    float* mean;       // may be NULL
    float* rstd;       // may be NULL
    int64_t rows;
    int64_t d;
    float eps;
};

// One compiled kernel configuration.
struct KernelEntry {
    const void* fn;        // the __global__ function (for occupancy queries)
    int threads;           // threads per CTA
    int rows_per_cta;      // rows a CTA handles per iteration of its row loop
    int smem_bytes;        // dynamic shared memory per CTA
    cudaError_t (*launch)(const Params&, int grid, cudaStream_t);
};

// Register-held kernels (warp per row when tpr == 32, a CTA per row above).
// Returns NULL if the configuration was not compiled.
const KernelEntry* reg_entry(int op, int vec, int slots, int tpr);

// Streaming two-read kernels (any width).
const KernelEntry* stream_entry(int op, int vec);

// Compiled configuration space of the register-held kernels.
constexpr int kMaxSlots = 8;
constexpr int kWarpRowsPerCta = 4;  // rows (warps) per CTA in the warp variant
constexpr int kStreamThreads = 512;

}  // namespace rn
