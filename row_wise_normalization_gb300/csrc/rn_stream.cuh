// rn_stream.cuh -- streaming row kernel for any width (x read twice).
//
// One CTA per row (persistent over rows). The first read accumulates the row
// statistics without holding the row: for LayerNorm each thread keeps a
// running (count, mean, M2) and folds in one vector at a time with Chan's
// pairwise update (the vector's own mean and centred square sum merged into
// the running triple), warps merge lane triples through shuffles, and the
// warps meet once in shared memory. Every element is first shifted by the
// row's first element K: a merge adds the product of the partial means'
// rounding error (~u |mean|) and their spread to M2, so working on x - K
// (mean ~ mu - K, of the order of sigma for typical rows) keeps that error
// ~u instead of ~u |mu| / sigma. The second read writes y. No width limit
// and no shared memory beyond the exchange slots; it is the fallback for rows
// the register-held and staged kernels cannot hold.
#pragma once

#include "rn_device.cuh"

namespace rn {

// (n, mean, M2) <- (n, mean, M2) merged with (nb, mb, Mb).
__device__ __forceinline__ void chan_merge(float& n, float& m, float& M, float nb, float mb,
                                           float Mb) {
    const float nn = n + nb;
    if (nn == 0.f) return;
    const float f = nb * __frcp_rn(nn);
    const float dl = mb - m;
    m = fmaf(dl, f, m);
    M = M + Mb + dl * dl * n * f;
    n = nn;
}

// Loads VEC elements of x (plus the residual when RES) at element offset j,
// as FP32.
template <typename T, int VEC, bool RES>
__device__ __forceinline__ void ld_xr(Vec<VEC>& v, const T* xr, const T* rr, int64_t j) {
    ldt_x(v, xr + j);
    if constexpr (RES) {
        Vec<VEC> r;
        ldt_x(r, rr + j);
#pragma unroll
        for (int k = 0; k < VEC; ++k) v.v[k] = v.v[k] + r.v[k];
    }
}

template <typename T, bool RES>
__device__ __forceinline__ float ld_xr1(const T* xr, const T* rr, int64_t j) {
    return RES ? ldt_x1(xr + j) + ldt_x1(rr + j) : ldt_x1(xr + j);
}

template <int OP, typename T, int VEC, int TPB, bool RES>
__global__ void __launch_bounds__(TPB, 1024 / TPB) stream_kernel(const Params p) {
    static_assert(VEC == 1 || VEC == Elem<T>::kVec, "a vector is one 128-bit access");
    static_assert(!RES || sizeof(T) == 4, "the residual form is FP32");
    const T* X = reinterpret_cast<const T*>(p.x);
    const T* R = reinterpret_cast<const T*>(p.r);
    const T* P0 = reinterpret_cast<const T*>(p.p0);
    const T* P1 = reinterpret_cast<const T*>(p.p1);
    T* Y = reinterpret_cast<T*>(p.y);
    T* H = reinterpret_cast<T*>(p.h);
    constexpr int W = TPB / 32;
    constexpr int U = VEC == 1 ? 8 : 16 / VEC;   // vectors a thread loads at once (first read)
    __shared__ __align__(16) float xch[2][W][4];
    const int t = threadIdx.x;
    const int w = t >> 5, lane = t & 31;
    const int64_t d = p.d;
    const float fd = (float)d;

    pdl_launch_dependents();
    if ((int64_t)blockIdx.x >= p.rows) return;
    pdl_wait();   // no global access before this
    int it = 0;
    for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x, ++it) {
        const T* xr = X + row * p.ldx;
        const T* rr = RES ? R + row * p.ldr : nullptr;
        T* yr = Y + row * p.ldy;
        T* hr = RES && p.h ? H + row * p.ldh : nullptr;
        int h = 0, tl = 0;
        int64_t nv;
        if constexpr (VEC > 1) {
            h = head_peel_t(xr, d);
            nv = (d - h) / VEC;
            tl = (int)(d - h - VEC * nv);
        } else {
            nv = d;
        }
        const bool has_e = (VEC > 1) && (t < h + tl);
        const int64_t ei = (t < h) ? (int64_t)t : (int64_t)h + VEC * nv + (t - h);
        float(*slot)[4] = xch[it & 1];

        // FP32 output is formed in the shifted frame, (x - K) - mus, so that
        // its error does not grow with |mean| / sigma
        constexpr bool SHIFT_OUT = sizeof(T) == 4;
        float mu = 0.f, rs, K = 0.f, mus = 0.f;
        if constexpr (OP == OP_LN) {
            K = ld_xr1<T, RES>(xr, rr, 0);   // shift (the same address for every thread)
            float n = 0.f, m = 0.f, M = 0.f;
            // chunks of U vectors a thread (their loads in flight together),
            // one merge per chunk; then the remaining vectors one by one
            int64_t q = t;
            for (; q + (U - 1) * TPB < nv; q += U * TPB) {
                Vec<VEC> v[U];
#pragma unroll
                for (int u = 0; u < U; ++u) ld_xr<T, VEC, RES>(v[u], xr, rr, h + (q + u * TPB) * VEC);
                float s = 0.f;
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int k = 0; k < VEC; ++k) {
                        v[u].v[k] -= K;
                        s += v[u].v[k];
                    }
                const float mc = s * (1.0f / (U * VEC));
                float Mc = 0.f;
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int k = 0; k < VEC; ++k) {
                        const float c = v[u].v[k] - mc;
                        Mc = fmaf(c, c, Mc);
                    }
                chan_merge(n, m, M, (float)(U * VEC), mc, Mc);
            }
            for (; q < nv; q += TPB) {
                Vec<VEC> v;
                ld_xr<T, VEC, RES>(v, xr, rr, h + q * VEC);
#pragma unroll
                for (int k = 0; k < VEC; ++k) v.v[k] -= K;
                float s = 0.f;
#pragma unroll
                for (int k = 0; k < VEC; ++k) s += v.v[k];
                const float mc = s * (1.0f / VEC);
                float Mc = 0.f;
#pragma unroll
                for (int k = 0; k < VEC; ++k) {
                    const float c = v.v[k] - mc;
                    Mc = fmaf(c, c, Mc);
                }
                chan_merge(n, m, M, (float)VEC, mc, Mc);
            }
            if (has_e) chan_merge(n, m, M, 1.f, ld_xr1<T, RES>(xr, rr, ei) - K, 0.f);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float nb = __shfl_xor_sync(0xffffffffu, n, o);
                const float mb = __shfl_xor_sync(0xffffffffu, m, o);
                const float Mb = __shfl_xor_sync(0xffffffffu, M, o);
                chan_merge(n, m, M, nb, mb, Mb);
            }
            if (lane == 0) *reinterpret_cast<float4*>(slot[w]) = make_float4(n, n * m, m, M);
            __syncthreads();
            float M2;
            merge_ln_warps<W>(slot, lane, fd, mus, M2);
            mu = K + mus;
            rs = rsqrtf(M2 / fd + p.eps);
        } else {
            float ss = 0.f;
#pragma unroll 4
            for (int64_t q = t; q < nv; q += TPB) {
                Vec<VEC> v;
                ld_xr<T, VEC, RES>(v, xr, rr, h + q * VEC);
#pragma unroll
                for (int k = 0; k < VEC; ++k) ss = fmaf(v.v[k], v.v[k], ss);
            }
            if (has_e) {
                const float e = ld_xr1<T, RES>(xr, rr, ei);
                ss = fmaf(e, e, ss);
            }
            ss = warp_sum(ss);
            if (lane == 0) slot[w][0] = ss;
            __syncthreads();
            ss = merge_sum_warps<W, 4>(slot, lane);
            rs = rsqrtf(ss / fd + p.eps);
        }

        bool pa = true;
        if constexpr (VEC > 1) {
            pa = aligned16(P0, h);
            if constexpr (OP == OP_LN) pa = pa && aligned16(P1, h);
        }
#pragma unroll 2
        for (int64_t q = t; q < nv; q += TPB) {
            const int64_t j = h + q * VEC;
            Vec<VEC> v, a, o;
            ld_xr<T, VEC, RES>(v, xr, rr, j);
            if (RES && hr) stt_y(hr + j, v);
            ldt_p(a, P0 + j, pa);
            if constexpr (OP == OP_LN) {
                Vec<VEC> b;
                ldt_p(b, P1 + j, pa);
#pragma unroll
                for (int k = 0; k < VEC; ++k)
                    o.v[k] = SHIFT_OUT ? fmaf(((v.v[k] - K) - mus) * rs, a.v[k], b.v[k])
                                       : fmaf((v.v[k] - mu) * rs, a.v[k], b.v[k]);
            } else {
#pragma unroll
                for (int k = 0; k < VEC; ++k) o.v[k] = v.v[k] * rs * a.v[k];
            }
            stt_y(yr + j, o);
        }
        if (has_e) {
            const float e = ld_xr1<T, RES>(xr, rr, ei);
            if (RES && hr) stt_y1(hr + ei, e);
            const float a = ldt_p1(P0 + ei);
            float o;
            if constexpr (OP == OP_LN)
                o = fmaf((SHIFT_OUT ? (e - K) - mus : e - mu) * rs, a, ldt_p1(P1 + ei));
            else
                o = e * rs * a;
            stt_y1(yr + ei, o);
        }
        if constexpr (OP == OP_LN) {
            if (t == 0) {
                if (p.mean) p.mean[row] = mu;
                if (p.rstd) p.rstd[row] = rs;
            }
        }
    }
}

template <int OP, typename T, int VEC, bool RES>
struct StreamInst {
    static cudaError_t launch(const Params& p, int grid, cudaStream_t s) {
        return launch_pdl(stream_kernel<OP, T, VEC, kStreamThreads, RES>, (unsigned)grid,
                          kStreamThreads, 0, s, p);
    }
    static const KernelEntry entry;
};

template <int OP, typename T, int VEC, bool RES>
const KernelEntry StreamInst<OP, T, VEC, RES>::entry = {
    (const void*)&stream_kernel<OP, T, VEC, kStreamThreads, RES>, kStreamThreads, 1, 0,
    &StreamInst<OP, T, VEC, RES>::launch, nullptr};

}  // namespace rn
