// rn_reg.cuh -- register-held row kernels (warp per row, or a CTA per row).
//
// Shape of the computation, for one row of width d:
//   1. every thread issues all of its loads of the row up front: SLOTS
//      vectors of VEC floats (128-bit ld.global.nc when VEC == 4), plus at
//      most one scalar of the unaligned head or tail; the row is read from
//      HBM exactly once and stays in registers until it is written back
//      (the single-pass, row-in-registers structure of "The load in flight,
//      and the shape Triton uses", section "The layer norm was rewritten in
//      the shape Triton uses");
//   2. LayerNorm: each warp reduces its share with xor shuffles to a count,
//      a sum and the sum of squared deviations about the warp's own mean;
//      when several warps share a row they meet once in shared memory behind
//      one named barrier and every thread merges the per-warp triples with
//      the parallel-axis rule  M2 = sum_w [M2_w + n_w (mean_w - mu)^2].
//      With one warp per row the centred pass runs on the held registers
//      after the mean. Either way there is no E[x^2] - mu^2 cancellation.
//      RMSNorm needs only the sum of squares;
//   3. rstd = rsqrtf(var + eps) and the row is written from the registers
//      with streaming 128-bit stores.
//
// Vector layout of a row: h scalars up to the first 16-byte boundary of the
// row (the "head peel", 0..3), nv aligned vectors, tl scalars of tail (0..3).
// Vector q goes to thread q % TPR, slot q / TPR; the h + tl <= 6 scalars go to
// threads 0..h+tl-1. Rows whose x and y differ in 16-byte phase use VEC = 1.
#pragma once

#include "rn_device.cuh"

namespace rn {

// Resident CTAs each kernel is compiled for, which sets its register cap:
// 64 registers per thread when a thread holds at most 16 floats of the row
// (4 on the scalar path, whose per-element addressing costs more), 80 above
// that (the largest slice, 8 vectors of 4, is 32 floats).
constexpr int reg_min_ctas(int threads, int held, int vec) {
    return threads >= 1024 ? 1 : 65536 / ((held > 16 || (vec == 1 && held > 4) ? 80 : 64) * threads);
}

template <int OP, int VEC, int SLOTS, int TPR, int RPC>
__global__ void __launch_bounds__(TPR * RPC, reg_min_ctas(TPR * RPC, SLOTS * VEC, VEC)) reg_kernel(const Params p) {
    static_assert(TPR % 32 == 0 && TPR * RPC <= 1024, "bad CTA shape");
    constexpr int WPR = TPR / 32;                    // warps per row
    constexpr int NST = (OP == OP_LN) ? 4 : 1;       // floats a warp publishes
    constexpr int NBUF = (WPR > 1) ? 2 : 1;
    __shared__ __align__(16) float xch[NBUF][RPC][WPR][NST];

    const int g = threadIdx.x / TPR;                 // row group within the CTA
    const int t = threadIdx.x - g * TPR;             // thread within the row group
    const int w = t >> 5;
    const int lane = t & 31;
    const int d = (int)p.d;                          // register-held rows are < 2^31 wide
    const float fd = (float)d;

    int it = 0;
    for (int64_t row = (int64_t)blockIdx.x * RPC + g; row < p.rows;
         row += (int64_t)gridDim.x * RPC, ++it) {
        const float* xr = p.x + row * p.d;
        float* yr = p.y + row * p.d;

        int h = 0, tl = 0;
        int nv;
        if constexpr (VEC == 4) {
            h = head_peel(xr, d);
            nv = (d - h) >> 2;
            tl = (int)(d - h - 4 * nv);
        } else {
            nv = d;
        }

        // ---- 1. load the row slice --------------------------------------
        Vec<VEC> v[SLOTS];
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            const int q = t + s * TPR;
            if (q < nv) {
                ld_x(v[s], xr + h + q * VEC);
            } else {
#pragma unroll
                for (int k = 0; k < VEC; ++k) v[s].v[k] = 0.f;
            }
        }
        float e = 0.f;
        int ei = 0;
        bool has_e = false;
        if constexpr (VEC == 4) {
            has_e = t < h + tl;
            if (has_e) {
                ei = (t < h) ? t : h + 4 * nv + (t - h);
                e = ld_x1(xr + ei);
            }
        }

        // ---- 2. statistics ---------------------------------------------
        float mu = 0.f, rs;
        if constexpr (OP == OP_LN) {
            float sum = e;
#pragma unroll
            for (int s = 0; s < SLOTS; ++s)
#pragma unroll
                for (int k = 0; k < VEC; ++k) sum += v[s].v[k];   // unused slots hold 0

            if constexpr (WPR == 1) {
                mu = warp_sum(sum) / fd;
                float m2 = 0.f;
                if (has_e) m2 = (e - mu) * (e - mu);
#pragma unroll
                for (int s = 0; s < SLOTS; ++s) {
                    if (t + s * TPR < nv) {
#pragma unroll
                        for (int k = 0; k < VEC; ++k) {
                            const float c = v[s].v[k] - mu;
                            m2 = fmaf(c, c, m2);
                        }
                    }
                }
                rs = rsqrtf(warp_sum(m2) / fd + p.eps);
            } else {
                const float wsum = warp_sum(sum);
                int nw = (w == 0) ? (h + tl) : 0;          // elements this warp holds
#pragma unroll
                for (int s = 0; s < SLOTS; ++s) {
                    const int rem = nv - s * TPR - 32 * w;
                    nw += VEC * (rem <= 0 ? 0 : (rem >= 32 ? 32 : rem));
                }
                const float wmean = nw > 0 ? wsum / (float)nw : 0.f;
                float m2 = 0.f;
                if (has_e) m2 = (e - wmean) * (e - wmean);
#pragma unroll
                for (int s = 0; s < SLOTS; ++s) {
                    if (t + s * TPR < nv) {
#pragma unroll
                        for (int k = 0; k < VEC; ++k) {
                            const float c = v[s].v[k] - wmean;
                            m2 = fmaf(c, c, m2);
                        }
                    }
                }
                m2 = warp_sum(m2);
                float(*slot)[NST] = xch[it & (NBUF - 1)][g];
                if (lane == 0)
                    *reinterpret_cast<float4*>(slot[w]) = make_float4((float)nw, wsum, wmean, m2);
                named_sync(1 + g, TPR);
                float M2;
                merge_ln_warps<WPR>(slot, lane, fd, mu, M2);
                rs = rsqrtf(M2 / fd + p.eps);
            }
        } else {
            float ss = e * e;
#pragma unroll
            for (int s = 0; s < SLOTS; ++s)
#pragma unroll
                for (int k = 0; k < VEC; ++k) ss = fmaf(v[s].v[k], v[s].v[k], ss);
            if constexpr (WPR == 1) {
                ss = warp_sum(ss);
            } else {
                const float wss = warp_sum(ss);
                float(*slot)[NST] = xch[it & (NBUF - 1)][g];
                if (lane == 0) slot[w][0] = wss;
                named_sync(1 + g, TPR);
                ss = merge_sum_warps<WPR, NST>(slot, lane);
            }
            rs = rsqrtf(ss / fd + p.eps);
        }

        // ---- 3. normalize and store from the held registers --------------
        bool pa = true;   // parameter vectors 16-byte aligned at this row's phase
        if constexpr (VEC == 4) {
            pa = ((((uintptr_t)p.p0 >> 2) + h) & 3) == 0;
            if constexpr (OP == OP_LN) pa = pa && ((((uintptr_t)p.p1 >> 2) + h) & 3) == 0;
        }
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            const int q = t + s * TPR;
            if (q < nv) {
                const int j = h + q * VEC;
                Vec<VEC> a, o;
                ld_p(a, p.p0 + j, pa);
                if constexpr (OP == OP_LN) {
                    Vec<VEC> b;
                    ld_p(b, p.p1 + j, pa);
#pragma unroll
                    for (int k = 0; k < VEC; ++k)
                        o.v[k] = fmaf((v[s].v[k] - mu) * rs, a.v[k], b.v[k]);
                } else {
#pragma unroll
                    for (int k = 0; k < VEC; ++k) o.v[k] = v[s].v[k] * rs * a.v[k];
                }
                st_y(yr + j, o);
            }
        }
        if (has_e) {
            const float a = ld_p1(p.p0 + ei);
            float o;
            if constexpr (OP == OP_LN)
                o = fmaf((e - mu) * rs, a, ld_p1(p.p1 + ei));
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
    }
}

// Launcher and registry entry of one configuration.
template <int OP, int VEC, int SLOTS, int TPR>
struct RegInst {
    static constexpr int RPC = (TPR == 32) ? kWarpRowsPerCta : 1;
    static cudaError_t launch(const Params& p, int grid, cudaStream_t s) {
        reg_kernel<OP, VEC, SLOTS, TPR, RPC><<<grid, TPR * RPC, 0, s>>>(p);
        return cudaGetLastError();
    }
    static const KernelEntry entry;
};

template <int OP, int VEC, int SLOTS, int TPR>
const KernelEntry RegInst<OP, VEC, SLOTS, TPR>::entry = {
    (const void*)&reg_kernel<OP, VEC, SLOTS, TPR, RegInst<OP, VEC, SLOTS, TPR>::RPC>,
    TPR * RegInst<OP, VEC, SLOTS, TPR>::RPC, RegInst<OP, VEC, SLOTS, TPR>::RPC, 0,
    &RegInst<OP, VEC, SLOTS, TPR>::launch};

template <int OP, int VEC, int TPR>
const KernelEntry* reg_pick_slots(int slots) {
    switch (slots) {
        case 1: return &RegInst<OP, VEC, 1, TPR>::entry;
        case 2: return &RegInst<OP, VEC, 2, TPR>::entry;
        case 3: return &RegInst<OP, VEC, 3, TPR>::entry;
        case 4: return &RegInst<OP, VEC, 4, TPR>::entry;
        case 5: return &RegInst<OP, VEC, 5, TPR>::entry;
        case 6: return &RegInst<OP, VEC, 6, TPR>::entry;
        case 7: return &RegInst<OP, VEC, 7, TPR>::entry;
        case 8: return &RegInst<OP, VEC, 8, TPR>::entry;
        default: return nullptr;
    }
}

template <int OP, int VEC>
const KernelEntry* reg_pick(int slots, int tpr) {
    switch (tpr) {
        case 32: return reg_pick_slots<OP, VEC, 32>(slots);
        case 64: return reg_pick_slots<OP, VEC, 64>(slots);
        case 128: return reg_pick_slots<OP, VEC, 128>(slots);
        case 256: return reg_pick_slots<OP, VEC, 256>(slots);
        case 512: return reg_pick_slots<OP, VEC, 512>(slots);
        case 1024: return reg_pick_slots<OP, VEC, 1024>(slots);
        default: return nullptr;
    }
}

}  // namespace rn
