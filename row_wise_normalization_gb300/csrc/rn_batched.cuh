// rn_batched.cuh -- many small, independent normalization problems in one
// launch.
//
// A tiny problem (512 x 128, say) finishes in a few microseconds of DRAM
// time but pays a whole launch; a model step that normalises many such
// tensors is launch-bound. Here the table of up to kBatchMax problems travels
// in the kernel's parameter space (a __grid_constant__ struct: no device
// allocation, no copy), the rows of all problems form one index space
// [0, start[n]), and every warp takes a contiguous chunk of it, finding its
// first problem by binary search over the row offsets and then walking
// forward (the problem's fields stay in registers while its rows last). A
// row is handled exactly as in
// the warp-per-row kernel: held in registers as 128-bit vectors after a
// head peel to the row's 16-byte boundary (x and y share that phase -- the
// host sends other problems to their own launches), mean then centred sum
// of squares by xor shuffles, output from the registers. Rows are at most
// 1024 elements; the kernel is compiled for 1, 2, 4 or 8 vectors per lane
// (SLOTS; up to 4 for 16-bit types) and the host picks the fewest that hold
// the widest row of the table, so narrow batches keep few registers and many
// rows in flight.
#pragma once

#include "rn_reg.cuh"

namespace rn {

// One row, as the warp-per-row kernel computes it (the same operations in
// the same order, so the results match a single call's bit for bit). AL: the
// problem's arrays are 16-byte aligned and d is a multiple of the vector.
template <int OP, typename T, int SLOTS, bool AL>
__device__ __forceinline__ void batched_row_held(HeldRow<Elem<T>::kVec, SLOTS, false>& cur,
                                                 T* yr, const T* P0, const T* P1, float* mean,
                                                 float* rstd, int64_t row, int d, float eps,
                                                 int lane) {
    constexpr int VEC = Elem<T>::kVec;
    const float fd = (float)d;
    const int h = cur.h, nv = cur.nv, tl = cur.tl;
    const bool has_e = !AL && lane < h + tl;
    const int ei = (lane < h) ? lane : h + VEC * nv + (lane - h);

    // slices of at most 8 floats load the parameters with the row, before
    // the reduction (as the single-call kernel does); wider ones after it
    constexpr bool EP = SLOTS * VEC <= 8;
    bool pa = true;
    if constexpr (!AL) {
        pa = aligned16(P0, h);
        if constexpr (OP == OP_LN) pa = pa && aligned16(P1, h);
    }
    Vec<VEC> pa0[SLOTS], pa1[OP == OP_LN ? SLOTS : 1];
    float pe0 = 0.f, pe1 = 0.f;
    if constexpr (EP)
        load_row_params<OP, T, VEC, SLOTS, 32>(pa0, pa1, pe0, pe1, P0, P1, h, nv, has_e, ei, pa,
                                               lane);

    // the statistics as the warp-per-row kernel takes them (FP32 vector rows
    // leave centred in place: (x - K) - mu_s)
    constexpr bool SHIFT = OP == OP_LN && sizeof(T) == 4;
    constexpr bool PK = VEC % 2 == 0;   // FP32 and 16-bit vector rows
    float mu = 0.f, rs, K = 0.f, mu_s = 0.f;
    warp_row_stats<OP, T, VEC, SLOTS, false>(cur, lane, has_e, fd, eps, K, mu_s, mu, rs);

#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        const int q = lane + s * 32;
        if (q < nv) {
            const int j = h + q * VEC;
            Vec<VEC> a, b, o;
            if constexpr (EP) {
                a = pa0[s];
                if constexpr (OP == OP_LN) b = pa1[s];
            } else {
                ldt_p(a, P0 + j, pa);
                if constexpr (OP == OP_LN) ldt_p(b, P1 + j, pa);
            }
            if constexpr (PK) {
                o = out_pairs<OP, false, VEC>(cur.v[s], a, b, 0.f, rs);
            } else if constexpr (OP == OP_LN) {
#pragma unroll
                for (int k = 0; k < VEC; ++k)
                    o.v[k] = SHIFT ? fmaf(((cur.v[s].v[k] - K) - mu_s) * rs, a.v[k], b.v[k])
                                   : fmaf((cur.v[s].v[k] - mu) * rs, a.v[k], b.v[k]);
            } else {
#pragma unroll
                for (int k = 0; k < VEC; ++k) o.v[k] = cur.v[s].v[k] * rs * a.v[k];
            }
            stt_y(yr + j, o);
        }
    }
    if constexpr (!EP) {
        if (has_e) {
            pe0 = ldt_p1(P0 + ei);
            if constexpr (OP == OP_LN) pe1 = ldt_p1(P1 + ei);
        }
    }
    if (has_e) {
        float o;
        if constexpr (OP == OP_LN)
            o = fmaf((SHIFT ? (cur.e - K) - mu_s : cur.e - mu) * rs, pe0, pe1);
        else
            o = cur.e * rs * pe0;
        stt_y1(yr + ei, o);
    }
    if constexpr (OP == OP_LN) {
        if (lane == 0) {
            if (mean) mean[row] = mu;
            if (rstd) rstd[row] = rs;
        }
    }
}

// Rows [r0, r1) of one problem. Narrow FP32 slices (at most 16 floats a
// lane) issue the loads of the next row before the current one is reduced
// and written, as the warp-per-row kernel's prefetch does (FP32 128 problems
// of 2048 x 64 70.1 -> 60.1 us, 64 x 512 x 128 17.0 -> 16.4 us; 16-bit rows,
// at fewer resident CTAs, were slower with it: 64 x 512 x 128 19.0 -> 22.6 us).
template <int OP, typename T, int SLOTS, bool AL>
__device__ __forceinline__ void batched_rows(const T* X, T* Y, const T* P0, const T* P1,
                                             float* mean, float* rstd, int64_t r0, int64_t r1,
                                             int d, float eps, int lane) {
    constexpr int VEC = Elem<T>::kVec;
    constexpr bool BPF = sizeof(T) == 4 && SLOTS * VEC <= 16;
    HeldRow<VEC, SLOTS, false> cur;
    load_row<T, VEC, SLOTS, 32, AL, false>(cur, X + r0 * d, nullptr, d, lane);
    for (int64_t row = r0; row < r1; ++row) {
        HeldRow<VEC, SLOTS, false> nxt;
        if constexpr (BPF) {
            if (row + 1 < r1)
                load_row<T, VEC, SLOTS, 32, AL, false>(nxt, X + (row + 1) * d, nullptr, d, lane);
        }
        batched_row_held<OP, T, SLOTS, AL>(cur, Y + row * d, P0, P1, mean, rstd, row, d, eps,
                                           lane);
        if constexpr (BPF) {
            cur = nxt;
        } else if (row + 1 < r1) {
            load_row<T, VEC, SLOTS, 32, AL, false>(cur, X + (row + 1) * d, nullptr, d, lane);
        }
    }
}

// Register budget per SLOTS: about 12 per held float and 52 fixed (the
// problem's fields, the row's head/tail and alignment state), plus the
// early-loaded parameters of slices of at most 8 floats and the prefetched
// row of FP32 slices of at most 16.
constexpr int batch_min_ctas(int slots, int vec) {
    const int regs = 52 + 12 * slots * vec / 4 + (slots * vec <= 8 ? 2 * slots * vec : 0) +
                     (vec == 4 && slots * vec <= 16 ? 2 * slots * vec : 0);   // prefetched row
    const int n = 65536 / (((regs + 7) / 8) * 8 * kBatchThreads);
    return n < 1 ? 1 : (n > 16 ? 16 : n);
}

template <int OP, typename T, int SLOTS>
__global__ void __launch_bounds__(kBatchThreads, batch_min_ctas(SLOTS, Elem<T>::kVec))
    batched_kernel(const __grid_constant__ BatchParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t total = p.start[p.n];
    // a contiguous chunk of rows per warp: the problem is looked up once and
    // then advanced as the chunk crosses into the next problem
    const int64_t chunk = (total + nwarps - 1) / nwarps;
    int64_t r = warp * chunk;
    const int64_t r_end = r + chunk < total ? r + chunk : total;
    pdl_launch_dependents();
    if (r >= r_end) return;
    pdl_wait();   // no global access before this (the table is a kernel parameter)
    int k = 0, hi = p.n - 1;   // the last k with start[k] <= r
    while (k < hi) {
        const int mid = (k + hi + 1) >> 1;
        if (p.start[mid] <= r)
            k = mid;
        else
            hi = mid - 1;
    }
    for (;;) {
        const BatchProblem& pr = p.pr[k];
        const int64_t first = p.start[k];
        const int64_t last = p.start[k + 1] < r_end ? p.start[k + 1] : r_end;
        const int d = pr.d;
        const T* X = reinterpret_cast<const T*>(pr.x);
        T* Y = reinterpret_cast<T*>(pr.y);
        const T* P0 = reinterpret_cast<const T*>(pr.p0);
        const T* P1 = reinterpret_cast<const T*>(pr.p1);
        float* mean = pr.mean;
        float* rstd = pr.rstd;
        const float eps = p.eps;
        if (pr.al)
            batched_rows<OP, T, SLOTS, true>(X, Y, P0, P1, mean, rstd, r - first, last - first, d,
                                             eps, lane);
        else
            batched_rows<OP, T, SLOTS, false>(X, Y, P0, P1, mean, rstd, r - first, last - first,
                                              d, eps, lane);
        r = last;
        if (r >= r_end) break;
        ++k;   // problems in the table all have rows > 0
    }
}

template <int OP, typename T, int SLOTS>
struct BatchInst {
    static cudaError_t launch(const BatchParams& p, int grid, cudaStream_t s) {
        return launch_pdl(batched_kernel<OP, T, SLOTS>, (unsigned)grid, kBatchThreads, 0, s, p);
    }
    static const BatchEntry entry;
};

template <int OP, typename T, int SLOTS>
const BatchEntry BatchInst<OP, T, SLOTS>::entry = {(const void*)&batched_kernel<OP, T, SLOTS>,
                                                   kBatchThreads,
                                                   &BatchInst<OP, T, SLOTS>::launch};

template <int OP, typename T>
const BatchEntry* batch_pick(int slots) {
    constexpr int M = 32 / Elem<T>::kVec;   // 8 FP32 or 4 16-bit vectors per lane
    switch (slots) {
        case 1: return &BatchInst<OP, T, 1>::entry;
        case 2: return &BatchInst<OP, T, 2>::entry;
        case 4: return &BatchInst<OP, T, 4>::entry;
        case 8: if constexpr (M >= 8) return &BatchInst<OP, T, 8>::entry; else return nullptr;
        default: return nullptr;
    }
}

}  // namespace rn
