// rn_cluster.cuh -- rows split across a thread-block cluster.
//
// A row too wide for one CTA's registers is spread over the CL CTAs of a
// cluster (CL = 2..16, each on its own SM): CTA c holds quads
// [c*Q, (c+1)*Q) of the row's aligned body in registers (Q = ceil(nv/CL);
// SLOTS quads per thread), CTA 0 also takes the <= 6 head/tail scalars. The
// row is read from HBM once and written from the registers, exactly as in the
// CTA-per-row kernel; only the statistics cross SMs. Each warp reduces its
// share to (count, sum, mean, centred M2) about its own mean, and lanes
// 0..CL-1 send that float4 straight into slot (c, warp) of every CTA of the
// cluster with an asynchronous distributed-shared-memory store
// (st.async ... mbarrier::complete_tx) that also counts its 16 bytes on the
// receiving CTA's mbarrier for that slot buffer. A CTA waits on its own
// mbarrier until all CL * WPR partials of the row have landed, then every
// thread merges them with the parallel-axis rule.
//
// No cluster barrier and no memory fence sits on the per-row path: a
// barrier.cluster.arrive.release orders every earlier memory access of the
// thread, the prefetched next row's global loads included, so each row used
// to wait for the next row's loads before its statistics could meet.
//
// Slot buffers and their mbarriers are double-buffered by row parity. Reuse
// needs no release signal: a CTA writes row i + 2's partials into buffer
// (i & 1) of a peer only after it has received every partial of row i + 1,
// and each warp of that peer sends its row i + 1 partial only after it has
// read buffer (i & 1) for row i. Thread 0 of each CTA arms the next phase of
// a buffer (arrive + expect_tx of CL * WPR * 16 bytes) right after its own
// wait on that buffer, before its warp sends the next row's partial.
//
// Waits are bounded (1 s of %globaltimer): a wait that runs out sets
// RN_DEVERR_CLUSTER_TIMEOUT in the device error word it was given and its
// warp stops processing rows; every warp still meets the cluster barrier at
// the end, so that no CTA leaves while a peer could address its shared
// memory.
//
// The partials are formed on x - K, K the row's first element: a merge adds
// the product of a partial mean's rounding error (~u |mean|) and the spread
// of the partial means to M2, which matters when a row is split into partials
// of few elements and |mu| >> sigma; after the shift the partial means are
// of the order of sigma.
//
// Clusters are persistent: cluster k walks rows k, k + nclusters, ... with
// all its CTAs in step (the same trip count), prefetching the next row's
// slice when PF is set.
#pragma once

#include "rn_async.cuh"

namespace rn {

__device__ __forceinline__ unsigned cluster_ctarank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The address that the shared-memory location `local` of this CTA has in
// CTA `rank` of the cluster.
__device__ __forceinline__ unsigned dsmem_map(const void* local, unsigned rank) {
    unsigned la = (unsigned)__cvta_generic_to_shared(local), ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
    return ra;
}

// Asynchronous store of a float4 into CTA `rank`'s shared memory at the
// address `local` has in this CTA, completing 16 bytes of transaction count
// on that CTA's mbarrier at the address `bar` has in this CTA.
__device__ __forceinline__ void dsmem_send4(const void* local, const void* bar, unsigned rank,
                                            float4 v) {
    const unsigned ra = dsmem_map(local, rank), rb = dsmem_map(bar, rank);
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, "
        "[%5];" ::"r"(ra),
        "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(rb)
        : "memory");
}

// Wait (acquire at cluster scope: the data came from other CTAs' st.async)
// for the phase of `bar` with the given parity; gives up after limit_ns.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint32_t bar, uint32_t parity,
                                                          unsigned long long limit_ns) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait_cluster(bar, parity)) {
        if (global_ns() - t0 > limit_ns) return false;
    }
    return true;
}

template <int OP, int SLOTS, int TPB, int CL, bool PF, bool AL>
struct ClusterCfg {
    static constexpr int WPR = TPB / 32;
    static constexpr int NE = CL * WPR;          // partials merged per row
    static constexpr int MINB = PF ? (TPB <= 256 ? 2 : 1) : (TPB >= 1024 ? 1 : (TPB == 512 ? 2 : 768 / TPB));
    // PSM: aligned rows of 256-thread CTAs keep the CTA's slice of gamma/beta
    // (w) in dynamic shared memory, loaded once: every thread its own quads,
    // in planes of TPB float4 per slot (64 KB per CTA for LayerNorm at 8 quads
    // a thread). Unaligned rows move their head peel, and with it the
    // columns a thread owns, from row to row; wider CTAs would need more
    // shared memory than an SM has for two of them.
    static constexpr bool PSM = AL && TPB == 256;
    static constexpr int SMEM = PSM ? (OP == OP_LN ? 2 : 1) * SLOTS * TPB * 16 : 0;
};

template <int OP, int SLOTS, int TPB, int CL, bool PF, bool AL>
__global__ void __launch_bounds__(TPB, (ClusterCfg<OP, SLOTS, TPB, CL, PF, AL>::MINB))
    cluster_kernel(const Params p) {
    using C = ClusterCfg<OP, SLOTS, TPB, CL, PF, AL>;
    constexpr int WPR = C::WPR;
    constexpr int NE = C::NE;
    __shared__ __align__(16) float4 slots[2][NE];
    __shared__ __align__(8) unsigned long long full[2];   // one mbarrier per slot buffer

    const int t = threadIdx.x, w = t >> 5, lane = t & 31;
    const unsigned c = cluster_ctarank();
    const int64_t cluster_id = blockIdx.x / CL;
    const int64_t nclusters = gridDim.x / CL;
    const int d = (int)p.d;
    const float fd = (float)d;
    constexpr uint32_t kRowBytes = NE * 16;                // partials one row brings to a CTA

    pdl_launch_dependents();
    // rows of this cluster: cluster_id, cluster_id + nclusters, ...
    const int64_t nmine =
        cluster_id < p.rows ? (p.rows - 1 - cluster_id) / nclusters + 1 : 0;
    if (t == 0) {
        mbar_init(smem_addr(&full[0]), 1);
        mbar_init(smem_addr(&full[1]), 1);
        // arm the phases of the first two rows
        if (nmine > 0) mbar_arrive_expect_tx(smem_addr(&full[0]), kRowBytes);
        if (nmine > 1) mbar_arrive_expect_tx(smem_addr(&full[1]), kRowBytes);
        mbar_fence_init();
    }
    // every CTA of the cluster is running, with its mbarriers initialised,
    // before anyone sends into a peer
    cluster_sync_all();
    pdl_wait();   // no global access before this

    // the CTA's parameter slice, staged once (PSM); thread t reads back only
    // the entries it wrote, so no barrier is needed
    extern __shared__ __align__(16) float4 cl_par[];
    if constexpr (C::PSM) {
        const int nv = d >> 2;
        const int Q = (nv + CL - 1) / CL;
        const int q0 = (int)c * Q;
        const int nq = nv - q0 < Q ? nv - q0 : Q;
#pragma unroll
        for (int k = 0; k < SLOTS; ++k) {
            const int q = t + k * TPB;
            if (q < nq) {
                cl_par[k * TPB + t] = ld_p4(p.p0 + 4 * (q0 + q));
                if constexpr (OP == OP_LN)
                    cl_par[(SLOTS + k) * TPB + t] = ld_p4(p.p1 + 4 * (q0 + q));
            }
        }
    }

    struct Slice {
        Vec<4> v[SLOTS];
        float e, K;              // head/tail scalar, the row's first element
        int h, nv, tl, q0, nq;   // row layout and this CTA's quads [q0, q0 + nq)
    };
    auto load = [&](Slice& s, int64_t row) {
        const float* xr = p.x + row * p.ldx;
        if constexpr (AL) {
            s.h = 0;
            s.nv = d >> 2;
            s.tl = 0;
        } else {
            s.h = head_peel(xr, d);
            s.nv = (d - s.h) >> 2;
            s.tl = d - s.h - 4 * s.nv;
        }
        const int Q = (s.nv + CL - 1) / CL;
        s.q0 = (int)c * Q;
        s.nq = s.nv - s.q0 < Q ? s.nv - s.q0 : Q;
        if (s.nq < 0) s.nq = 0;
#pragma unroll
        for (int k = 0; k < SLOTS; ++k) {
            const int q = t + k * TPB;
            if (q < s.nq) {
                ld_x(s.v[k], xr + s.h + 4 * (s.q0 + q));
            } else {
                s.v[k].v[0] = s.v[k].v[1] = s.v[k].v[2] = s.v[k].v[3] = 0.f;
            }
        }
        s.e = 0.f;
        if (!AL && c == 0 && t < s.h + s.tl)
            s.e = ld_x1(xr + ((t < s.h) ? t : s.h + 4 * s.nv + (t - s.h)));
        s.K = OP == OP_LN ? ld_x1(xr) : 0.f;   // the same address for every thread
    };

    int64_t row = cluster_id;
    Slice cur;
    if (row < p.rows) load(cur, row);
    for (int64_t it = 0; it < nmine; ++it, row += nclusters) {
        const int64_t nrow = row + nclusters;
        Slice nxt;
        if constexpr (PF) {
            if (nrow < p.rows) load(nxt, nrow);
        }
        // aligned rows: the bulk-copy engine fetches this CTA's slice of the
        // row after the ones held into L2 (one instruction, one thread)
        if constexpr (AL) {
            const int64_t frow = PF ? nrow + nclusters : nrow;
            if (t == 0 && frow < p.rows && cur.nq > 0)
                prefetch_l2_bulk(p.x + frow * p.ldx + 4 * (int64_t)cur.q0,
                                 (uint32_t)cur.nq * 16u);
        }
        const int h = cur.h, nv = cur.nv, tl = cur.tl, q0 = cur.q0, nq = cur.nq;
        const bool has_e = !AL && c == 0 && t < h + tl;
        const int ei = (t < h) ? t : h + 4 * nv + (t - h);

        // ---- per-warp partial statistics --------------------------------
        float4 part;   // (count, sum, mean, M2) or (-, sum of squares, -, -)
        {
            int nw = (!AL && c == 0 && w == 0) ? (h + tl) : 0;
#pragma unroll
            for (int k = 0; k < SLOTS; ++k) {
                const int rem = nq - k * TPB - 32 * w;
                nw += 4 * (rem <= 0 ? 0 : (rem >= 32 ? 32 : rem));
            }
            // element pairs on the packed FP32 pipe; LayerNorm shifts the
            // held quads by K in place (x -> x - K), once
            if constexpr (OP == OP_LN) {
                const float K = cur.K;
                const F2 k2 = f2s(K);
                F2 acc = f2s(0.f);
#pragma unroll
                for (int k = 0; k < SLOTS; ++k) {
                    if (t + k * TPB < nq) {
#pragma unroll
                        for (int j = 0; j < 4; j += 2) {
                            const F2 d = sub2(f2(cur.v[k].v[j], cur.v[k].v[j + 1]), k2);
                            f2_get(d, cur.v[k].v[j], cur.v[k].v[j + 1]);
                            acc = add2(acc, d);
                        }
                    }
                }
                float a0, a1;
                f2_get(acc, a0, a1);
                const float sum = (has_e ? cur.e - K : 0.f) + (a0 + a1);
                const float wsum = warp_sum(sum);
                const float wmean = nw > 0 ? wsum / (float)nw : 0.f;   // of x - K
                const float de = (cur.e - K) - wmean;
                const F2 w2 = f2s(wmean);
                F2 mm = f2s(0.f);
#pragma unroll
                for (int k = 0; k < SLOTS; ++k) {
                    if (t + k * TPB < nq) {
#pragma unroll
                        for (int j = 0; j < 4; j += 2) {
                            const F2 dd = sub2(f2(cur.v[k].v[j], cur.v[k].v[j + 1]), w2);
                            mm = fma2(dd, dd, mm);
                        }
                    }
                }
                float m0, m1;
                f2_get(mm, m0, m1);
                const float m2 = (has_e ? de * de : 0.f) + (m0 + m1);
                part = make_float4((float)nw, wsum, wmean, warp_sum(m2));
            } else {
                F2 sq = f2s(0.f);
#pragma unroll
                for (int k = 0; k < SLOTS; ++k)
#pragma unroll
                    for (int j = 0; j < 4; j += 2) {   // unused slots hold 0
                        const F2 x2 = f2(cur.v[k].v[j], cur.v[k].v[j + 1]);
                        sq = fma2(x2, x2, sq);
                    }
                float s0, s1;
                f2_get(sq, s0, s1);
                part = make_float4(0.f, warp_sum(cur.e * cur.e + (s0 + s1)), 0.f, 0.f);
            }
        }
        // lane r sends this warp's partial into CTA r's slot (c, w) and
        // counts its bytes on CTA r's mbarrier of this buffer
        const int b = (int)(it & 1);
        float4* buf = slots[b];
        if (lane < CL) dsmem_send4(&buf[c * WPR + w], &full[b], (unsigned)lane, part);
        const uint32_t bar = smem_addr(&full[b]);
        const bool ok = mbar_wait_cluster_bounded(bar, (uint32_t)((it >> 1) & 1), kWaitLimitNs);
        // thread 0 arms this buffer's next phase (row it + 2) before its warp
        // sends row it + 1's partial; other CTAs' sends for row it + 2 come
        // after they have received that partial
        if (t == 0 && it + 2 < nmine) mbar_arrive_expect_tx(bar, kRowBytes);
        // a wait that ran out stops the whole warp (the loop holds no CTA
        // barrier, so warps may stop at different rows: each later wait of a
        // warp still running also runs out)
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0 && p.err) atomicOr(p.err, kErrClusterTimeout);
            break;
        }

        // ---- merge the CL * WPR partials (every thread) -----------------
        float mu = 0.f, rs, mus = 0.f;   // mus = mu - K; the output is formed as (x - K) - mus
        {
            float s1 = 0.f;
#pragma unroll
            for (int k = lane; k < NE; k += 32) s1 += buf[k].y;
            s1 = warp_sum(s1);
            if constexpr (OP == OP_LN) {
                mus = s1 / fd;                        // mean of x - K
                float m2 = 0.f;
#pragma unroll
                for (int k = lane; k < NE; k += 32) {
                    const float4 e4 = buf[k];
                    const float dm = e4.z - mus;
                    m2 += fmaf(e4.x * dm, dm, e4.w);
                }
                mu = cur.K + mus;
                rs = rsqrtf(warp_sum(m2) / fd + p.eps);
            } else {
                rs = rsqrtf(s1 / fd + p.eps);
            }
        }

        // ---- normalize and store from the held registers ----------------
        float* yr = p.y + row * p.ldy;
        bool pa = true;
        if constexpr (!AL) {
            pa = ((((uintptr_t)p.p0 >> 2) + h) & 3) == 0;
            if constexpr (OP == OP_LN) pa = pa && ((((uintptr_t)p.p1 >> 2) + h) & 3) == 0;
        }
#pragma unroll
        for (int k = 0; k < SLOTS; ++k) {
            const int q = t + k * TPB;
            if (q < nq) {
                const int j = h + 4 * (q0 + q);
                Vec<4> a, bb, o;
                if constexpr (C::PSM) {
                    const float4 a4 = cl_par[k * TPB + t];
                    a.v[0] = a4.x; a.v[1] = a4.y; a.v[2] = a4.z; a.v[3] = a4.w;
                    if constexpr (OP == OP_LN) {
                        const float4 b4 = cl_par[(SLOTS + k) * TPB + t];
                        bb.v[0] = b4.x; bb.v[1] = b4.y; bb.v[2] = b4.z; bb.v[3] = b4.w;
                    }
                } else {
                    ld_p(a, p.p0 + j, pa);
                    if constexpr (OP == OP_LN) ld_p(bb, p.p1 + j, pa);
                }
                // LayerNorm: the held quads are x - K
                o = out_pairs<OP, (OP == OP_LN)>(cur.v[k], a, bb, mus, rs);
                st_y(yr + j, o);
            }
        }
        if (has_e) {
            const float a = ld_p1(p.p0 + ei);
            float o;
            if constexpr (OP == OP_LN)
                o = fmaf(((cur.e - cur.K) - mus) * rs, a, ld_p1(p.p1 + ei));
            else
                o = cur.e * rs * a;
            st_y1(yr + ei, o);
        }
        if constexpr (OP == OP_LN) {
            if (c == 0 && t == 0) {
                if (p.mean) p.mean[row] = mu;
                if (p.rstd) p.rstd[row] = rs;
            }
        }
        if constexpr (PF) {
            cur = nxt;
        } else {
            if (nrow < p.rows) load(cur, nrow);
        }
    }
    // no CTA leaves while a peer could still address its shared memory
    cluster_sync_all();
}

template <int OP, int SLOTS, int TPB, int CL, bool AL>
struct ClusterInst {
    static constexpr bool PF = TPB <= 256;
    static constexpr int SMEM = ClusterCfg<OP, SLOTS, TPB, CL, PF, AL>::SMEM;
    static cudaError_t launch(const Params& p, int grid, cudaStream_t s) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid, 1, 1);
        cfg.blockDim = dim3(TPB, 1, 1);
        cfg.dynamicSmemBytes = SMEM;
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = CL;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        return cudaLaunchKernelEx(&cfg, cluster_kernel<OP, SLOTS, TPB, CL, PF, AL>, p);
    }
    static cudaError_t prepare(int) {
        cudaError_t e = cudaSuccess;
        if (CL > 8)
            e = cudaFuncSetAttribute(cluster_kernel<OP, SLOTS, TPB, CL, PF, AL>,
                                     cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        // any dynamic shared memory: the default limit covers static and
        // dynamic together (48 KB), which the static part already uses some of
        if (e == cudaSuccess && SMEM > 0)
            e = cudaFuncSetAttribute(cluster_kernel<OP, SLOTS, TPB, CL, PF, AL>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        return e;
    }
    // Clusters that can be resident at once.
    static cudaError_t max_clusters(int* n) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(CL, 1, 1);
        cfg.blockDim = dim3(TPB, 1, 1);
        cfg.dynamicSmemBytes = SMEM;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = CL;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaOccupancyMaxActiveClusters(n, cluster_kernel<OP, SLOTS, TPB, CL, PF, AL>, &cfg);
    }
    static const ClusterEntry entry;
};

template <int OP, int SLOTS, int TPB, int CL, bool AL>
const ClusterEntry ClusterInst<OP, SLOTS, TPB, CL, AL>::entry = {
    CL, TPB, SLOTS, &ClusterInst<OP, SLOTS, TPB, CL, AL>::launch,
    &ClusterInst<OP, SLOTS, TPB, CL, AL>::prepare, &ClusterInst<OP, SLOTS, TPB, CL, AL>::max_clusters};

}  // namespace rn
