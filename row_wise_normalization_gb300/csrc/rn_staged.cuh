// rn_staged.cuh -- rows staged in shared memory by the bulk-copy (TMA) engine.
//
// A persistent CTA owns rows blockIdx.x, blockIdx.x + gridDim.x, ... and keeps
// a ring of STAGES row buffers in shared memory. One thread issues a 1-D
// cp.async.bulk (global -> shared, completion counted in bytes on the stage's
// mbarrier) for the 16-byte-aligned body of a row; the <= 6 scalars of the
// unaligned head and tail are read with plain loads. While the CTA reduces
// and writes row i, the copies of rows i+1 .. i+STAGES-1 are in flight, so
// the bytes in flight per SM do not depend on how many threads hold data --
// the point of staging rows too wide for registers (the pages' kernels hold
// at most 1024 elements per row in registers, "LayerNorm [4096,768] is about
// 10% behind Triton's kernel", wide-row comment).
//
// Per row: pass 1 sums the staged row (shifted by its first element),
// reduce -> mean; pass 2 sums squared deviations about the mean, reduce ->
// rstd (the centred two-pass form of the statistics equation); pass 3 writes
// y from shared memory with streaming 128-bit stores. Each reduction is one
// xor-shuffle tree per warp and one exchange through shared memory.
//
// Every mbarrier wait is bounded (about one second of %globaltimer); a wait
// that runs out sets bit 0 of the device error word, waits (bounded) for the
// CTA's copies still in flight, and the CTA returns.
#pragma once

#include "rn_async.cuh"

namespace rn {

// The device error word (one per device, per loaded library). This header is
// compiled into one translation unit only (staged.cu), which also holds the
// host accessor.
__device__ unsigned int g_device_error = 0;

// Self-test of the bounded wait: thread 0 waits on an mbarrier that nothing
// arrives at, through the wait above, and records the timeout exactly as a
// staged kernel does. Touches no data.
__global__ void bounded_wait_selftest_kernel(unsigned long long limit_ns) {
    __shared__ __align__(8) unsigned long long bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_bounded(smem_addr(&bar), 0, limit_ns))
        atomicOr(&g_device_error, kErrStagedTimeout);
}

// Sum of one float per thread over the CTA; every thread gets the result.
// `slot` has one float per warp; the caller guarantees it is not being read.
template <int TPB>
__device__ __forceinline__ float block_sum(float v, float* slot, int lane, int w) {
    constexpr int W = TPB / 32;
    v = warp_sum(v);
    if (lane == 0) slot[w] = v;
    __syncthreads();
    float s;
    if constexpr (W <= 8) {
        s = 0.f;
#pragma unroll
        for (int k = 0; k < W; ++k) s += slot[k];
    } else {
        s = warp_sum(lane < W ? slot[lane] : 0.f);
    }
    return s;
}

// Bytes of shared memory one stage needs for a row of width d (the aligned
// body is at most 4 * (d / 4) bytes).
__host__ __device__ constexpr int staged_stage_bytes(int64_t d) {
    return (int)(((d / 4) * 16 + 127) / 128 * 128);
}

template <int OP, int TPB, int STAGES>
__global__ void __launch_bounds__(TPB, 1) staged_kernel(const Params p) {
    constexpr int W = TPB / 32;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ __align__(8) unsigned long long bars[STAGES];
    __shared__ float red[3][W];     // three rotating exchange slots
    __shared__ int abort_flag;

    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int d = (int)p.d;
    const float fd = (float)d;
    const int stage_bytes = staged_stage_bytes(d);
    const int64_t first = blockIdx.x;
    const int64_t stride = gridDim.x;
    const int64_t nmine = first < p.rows ? (p.rows - 1 - first) / stride + 1 : 0;

    pdl_launch_dependents();
    if (t == 0) {
        abort_flag = 0;
        for (int s = 0; s < STAGES; ++s) mbar_init(smem_addr(&bars[s]), 1);
        mbar_fence_init();
    }
    __syncthreads();
    pdl_wait();   // no global access (bulk copies included) before this

    // Issue the copy of my i-th row into stage i % STAGES (thread 0 only).
    auto issue = [&](int64_t i) {
        const int64_t row = first + i * stride;
        const float* xr = p.x + row * p.ldx;
        const int h = head_peel(xr, d);
        const int nv = (d - h) >> 2;
        const int s = (int)(i % STAGES);
        const uint32_t bar = smem_addr(&bars[s]);
        if (nv > 0) {
            mbar_arrive_expect_tx(bar, (uint32_t)nv * 16u);
            bulk_g2s(smem_addr(smem_raw + (size_t)s * stage_bytes), xr + h, (uint32_t)nv * 16u,
                     bar);
        } else {
            mbar_arrive(bar);
        }
    };

    if (t == 0)
        for (int64_t i = 0; i < STAGES && i < nmine; ++i) issue(i);

    int rot = 0;
    for (int64_t i = 0; i < nmine; ++i) {
        const int64_t row = first + i * stride;
        const float* xr = p.x + row * p.ldx;
        float* yr = p.y + row * p.ldy;
        const int h = head_peel(xr, d);
        const int nv = (d - h) >> 2;
        const int tl = d - h - 4 * nv;
        const int s = (int)(i % STAGES);
        const uint32_t parity = (uint32_t)((i / STAGES) & 1);
        const float4* buf = reinterpret_cast<const float4*>(smem_raw + (size_t)s * stage_bytes);

        // head/tail scalars with plain loads while the body lands
        const bool has_e = t < h + tl;
        const int ei = (t < h) ? t : h + 4 * nv + (t - h);
        const float e = has_e ? ld_x1(xr + ei) : 0.f;

        if (!mbar_wait_bounded(smem_addr(&bars[s]), parity)) {
            atomicOr(&g_device_error, kErrStagedTimeout);
            abort_flag = 1;
        }
        __syncthreads();
        if (abort_flag) break;

        float mu = 0.f, rs, K = 0.f, mus = 0.f;   // mus = mu - K
        if constexpr (OP == OP_LN) {
            // pass 1: mean (shifted by the row's first element); the output
            // is formed in the shifted frame too, (x - K) - mus
            K = d > 0 ? ld_x1(xr) : 0.f;
            float s1 = has_e ? e - K : 0.f;
            for (int q = t; q < nv; q += TPB) {
                const float4 v = buf[q];
                s1 += ((v.x - K) + (v.y - K)) + ((v.z - K) + (v.w - K));
            }
            mus = block_sum<TPB>(s1, red[rot], lane, w) / fd;
            mu = K + mus;
            rot = rot == 2 ? 0 : rot + 1;
            // pass 2: centred sum of squares
            float s2 = has_e ? ((e - K) - mus) * ((e - K) - mus) : 0.f;
            for (int q = t; q < nv; q += TPB) {
                const float4 v = buf[q];
                const float a = (v.x - K) - mus, b = (v.y - K) - mus, c = (v.z - K) - mus,
                            dd = (v.w - K) - mus;
                s2 = fmaf(a, a, s2);
                s2 = fmaf(b, b, s2);
                s2 = fmaf(c, c, s2);
                s2 = fmaf(dd, dd, s2);
            }
            rs = rsqrtf(block_sum<TPB>(s2, red[rot], lane, w) / fd + p.eps);
            rot = rot == 2 ? 0 : rot + 1;
        } else {
            float s2 = has_e ? e * e : 0.f;
            for (int q = t; q < nv; q += TPB) {
                const float4 v = buf[q];
                s2 = fmaf(v.x, v.x, s2);
                s2 = fmaf(v.y, v.y, s2);
                s2 = fmaf(v.z, v.z, s2);
                s2 = fmaf(v.w, v.w, s2);
            }
            rs = rsqrtf(block_sum<TPB>(s2, red[rot], lane, w) / fd + p.eps);
            rot = rot == 2 ? 0 : rot + 1;
        }

        // pass 3: write y
        bool pa = ((((uintptr_t)p.p0 >> 2) + h) & 3) == 0;
        if constexpr (OP == OP_LN) pa = pa && ((((uintptr_t)p.p1 >> 2) + h) & 3) == 0;
        for (int q = t; q < nv; q += TPB) {
            const float4 v = buf[q];
            const int j = h + 4 * q;
            Vec<4> a, o;
            ld_p(a, p.p0 + j, pa);
            if constexpr (OP == OP_LN) {
                Vec<4> b;
                ld_p(b, p.p1 + j, pa);
                o.v[0] = fmaf(((v.x - K) - mus) * rs, a.v[0], b.v[0]);
                o.v[1] = fmaf(((v.y - K) - mus) * rs, a.v[1], b.v[1]);
                o.v[2] = fmaf(((v.z - K) - mus) * rs, a.v[2], b.v[2]);
                o.v[3] = fmaf(((v.w - K) - mus) * rs, a.v[3], b.v[3]);
            } else {
                o.v[0] = v.x * rs * a.v[0];
                o.v[1] = v.y * rs * a.v[1];
                o.v[2] = v.z * rs * a.v[2];
                o.v[3] = v.w * rs * a.v[3];
            }
            st_y(yr + j, o);
        }
        if (has_e) {
            const float a = ld_p1(p.p0 + ei);
            float o;
            if constexpr (OP == OP_LN)
                o = fmaf(((e - K) - mus) * rs, a, ld_p1(p.p1 + ei));
            else
                o = e * rs * a;
            st_y1(yr + ei, o);
        }
        if constexpr (OP == OP_LN) {
            if (t == 0) {
                if (p.mean) p.mean[row] = mu;
                if (p.rstd) p.rstd[row] = rs;
            }
        }

        // every thread is done with stage s: refill it with row i + STAGES
        __syncthreads();
        if (t == 0 && i + STAGES < nmine) {
            fence_proxy_async_smem();
            issue(i + STAGES);
        }
    }

    if (abort_flag && t == 0) {
        // drain: wait (bounded) for every copy this CTA may still have in flight
        for (int s = 0; s < STAGES; ++s) {
            const uint32_t bar = smem_addr(&bars[s]);
            for (uint32_t par = 0; par < 2; ++par) (void)mbar_wait_bounded(bar, par);
        }
    }
}

template <int OP, int TPB, int STAGES>
struct StagedInst {
    static cudaError_t launch(const Params& p, int grid, cudaStream_t s) {
        const int smem = STAGES * staged_stage_bytes(p.d);
        return launch_pdl(staged_kernel<OP, TPB, STAGES>, (unsigned)grid, TPB, (size_t)smem, s, p);
    }
    // The limit is per function and process-wide, so it is raised once to the
    // whole budget (never lowered to one launch's need, which would break a
    // later launch that needs more).
    static cudaError_t prepare(int /*smem*/) {
        return cudaFuncSetAttribute(staged_kernel<OP, TPB, STAGES>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kStagedSmemBudget);
    }
    static const KernelEntry entry;
};

template <int OP, int TPB, int STAGES>
const KernelEntry StagedInst<OP, TPB, STAGES>::entry = {
    (const void*)&staged_kernel<OP, TPB, STAGES>, TPB, 1, 0, &StagedInst<OP, TPB, STAGES>::launch,
    &StagedInst<OP, TPB, STAGES>::prepare};

}  // namespace rn
