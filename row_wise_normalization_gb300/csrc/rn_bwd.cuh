// rn_bwd.cuh -- LayerNorm / RMSNorm backward (FP32).
//
// Row part (dx), one row group per row at a time, row slice in registers as in
// the forward kernels:
//   LayerNorm, from the saved mean and rstd of the forward:
//     xhat = (x - mean) * rstd,  g = dy * gamma,
//     dx = rstd * (g - mean_j(g) - xhat * mean_j(g * xhat));
//   RMSNorm, with r = (mean_j x^2 + eps)^-1/2 recomputed from the held row:
//     g = dy * w,  dx = r * (g - x * r^2 * mean_j(g * x)).
// Both need two row sums, which meet in one exchange (warp xor shuffles, then
// one named barrier when several warps share a row). g is rounded once
// (__fmul_rn, never contracted into a later fma), so the g the sums saw is the
// g that dx subtracts from: for a one-element row g - mean(g) is exactly 0,
// where a contracted product would leave its rounding residue times rstd.
//
// T is the storage type of dy, x, dx and the parameter vector (FP32, BF16 or
// FP16; 16-bit values are widened on load, dx rounded once on store); all
// arithmetic, the saved statistics and the workspace partials are FP32, and
// the parameter gradients are rounded once, into T, by the column reduction.
//
// Parameter part (dgamma/dbeta, dw): a thread owns the same columns for every
// row it processes (whole aligned vectors, or single elements when the
// arrays are not all 16-byte aligned with d % 4 == 0), so it accumulates its
// columns' sums over its rows in registers. A CTA holds 256 / TPR row groups
// (at least one); when its rows are done the groups' sums are added through
// shared memory in group order and the CTA writes one partial row to the
// workspace. A 1024-thread row group (rows wider than 8192) has 64 registers
// a thread, which hold x and dy but not also the parameters and the
// accumulators: there those live in shared memory instead (SMS), each
// thread reading and writing only its own entries. column_reduce_kernel then adds the CTAs' rows in a fixed order
// with Kahan compensation: deterministic for a given grid, no atomics. It is
// launched as a programmatic dependent of the row kernel, so its launch
// overlaps the row kernel's tail and it waits (griddepcontrol.wait) for the
// row kernel's writes before reading.
#pragma once

#include "rn_async.cuh"

namespace rn {

// Registers a thread is budgeted: x, dy, the held parameters and (PG) two
// accumulators per held element, plus indices and addresses; the CTAs per SM
// follow from it (65536 registers, allocated in units of 8 per thread).
constexpr int bwd_min_ctas(int threads, int held, bool pg) {
    const int need = 48 + held * (pg ? 5 : 3);
    const int budget = need < 64 ? 64 : need;
    const int n = 65536 / (((budget + 7) / 8) * 8 * threads);
    return n < 1 ? 1 : (n > 32 ? 32 : n);
}

// FP32 store of one thread's partial sums to the workspace (VEC 1, 4 or 8).
template <int VEC>
__device__ __forceinline__ void st_ws(float* p, const Vec<VEC>& r) {
    if constexpr (VEC == 8) {
        Vec<4> a, b;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            a.v[k] = r.v[k];
            b.v[k] = r.v[4 + k];
        }
        st_y(p, a);
        st_y(p + 4, b);
    } else {
        st_y(p, r);
    }
}

// Whether an instance keeps its per-thread state in shared memory, and how
// many bytes of it: the parameters, and (PG) one or two accumulators, each
// SLOTS x TPR vectors.
constexpr bool bwd_sms(int threads) { return threads == 1024; }
constexpr int bwd_sms_bytes(int op, int vec, int slots, int tpr, bool pg) {
    return bwd_sms(tpr) ? (1 + (pg ? (op == OP_LN ? 2 : 1) : 0)) * slots * vec * tpr * 4 : 0;
}

// A thread's vector `s` of one shared-memory plane set: planes of TPR
// 16-byte chunks (VEC 4 or 8) or floats (VEC 1), so that a warp's accesses to
// one plane are contiguous and free of bank conflicts.
template <int VEC, int TPR>
__device__ __forceinline__ void sms_ld(Vec<VEC>& v, const float* base, int s, int t) {
    if constexpr (VEC == 1) {
        v.v[0] = base[s * TPR + t];
    } else {
#pragma unroll
        for (int c = 0; c < VEC / 4; ++c) {
            const float4 q = reinterpret_cast<const float4*>(base)[(s * (VEC / 4) + c) * TPR + t];
            v.v[4 * c] = q.x;
            v.v[4 * c + 1] = q.y;
            v.v[4 * c + 2] = q.z;
            v.v[4 * c + 3] = q.w;
        }
    }
}
template <int VEC, int TPR>
__device__ __forceinline__ void sms_st(float* base, int s, int t, const Vec<VEC>& v) {
    if constexpr (VEC == 1) {
        base[s * TPR + t] = v.v[0];
    } else {
#pragma unroll
        for (int c = 0; c < VEC / 4; ++c)
            reinterpret_cast<float4*>(base)[(s * (VEC / 4) + c) * TPR + t] =
                make_float4(v.v[4 * c], v.v[4 * c + 1], v.v[4 * c + 2], v.v[4 * c + 3]);
    }
}

// STG (staged): one CTA is one row group (RPC == 1, 256 or 512 threads,
// vector layout) and thread 0 has the bulk-copy engine bring the CTA's rows
// of x and dy into a ring of p.stages (2..kBwdMaxStages) shared-memory
// stages, p.stages - 1 rows ahead of the row being reduced: the bytes in flight no longer depend on the
// registers the accumulators leave. A stage is refilled once every thread
// has passed the next row's exchange barrier (all its reads of the stage are
// done). Each wait is bounded; a CTA whose wait runs out (the vote at that
// barrier) sets a bit in p.err, waits (bounded) for its copies still in
// flight and returns.
template <int OP, typename T, int VEC, int SLOTS, int TPR, int RPC, bool PG, bool STG = false>
__global__ void __launch_bounds__(TPR * RPC, bwd_min_ctas(TPR * RPC, SLOTS * VEC, PG))
    bwd_kernel(const BwdParams p) {
    static_assert(TPR % 32 == 0 && TPR * RPC <= 1024, "bad CTA shape");
    static_assert(VEC == 1 || VEC == Elem<T>::kVec, "a vector is one 128-bit access");
    static_assert(!STG || (RPC == 1 && VEC > 1 && TPR >= 64 && (!bwd_sms(TPR) || OP == OP_RMS)),
                  "staged: one row group per CTA, vector layout, accumulators in registers");
    const T* X = reinterpret_cast<const T*>(p.x);
    const T* DY = reinterpret_cast<const T*>(p.dy);
    const T* P0 = reinterpret_cast<const T*>(p.p0);
    T* DX = reinterpret_cast<T*>(p.dx);
    constexpr int WPR = TPR / 32;
    constexpr int NBUF = WPR > 1 ? 2 : 1;
    __shared__ __align__(16) float xch[NBUF][RPC][WPR][2];

    const int g = threadIdx.x / TPR;
    const int t = threadIdx.x - g * TPR;
    const int w = t >> 5, lane = t & 31;
    const int d = (int)p.d;
    const int nv = d / VEC;               // vectors only when d % VEC == 0 (host checks)
    const float inv_d = 1.0f / (float)d;
    const int64_t group = (int64_t)blockIdx.x * RPC + g;
    const int64_t ngroups = (int64_t)gridDim.x * RPC;

    // staged: the ring (in dynamic shared memory; SMS is off) and the
    // issue of the CTA's k-th row into stage k % nst (thread 0)
    extern __shared__ __align__(16) float bwd_state[];
    __shared__ __align__(8) unsigned long long sbar[STG ? kBwdMaxStages : 1];
    const int nst = STG ? p.stages : 1;
    const int64_t rowbytes = (int64_t)d * (int64_t)sizeof(T);
    const int64_t rpad = (rowbytes + 127) / 128 * 128;
    // (after the parameter plane when the parameters live in shared memory)
    unsigned char* const ring = reinterpret_cast<unsigned char*>(bwd_state) +
                                (STG && bwd_sms(TPR * RPC) ? SLOTS * VEC * TPR * 4 : 0);
    auto issue = [&](int k) {
        const int64_t r = group + (int64_t)k * ngroups;
        if (r >= p.rows) return;
        const int st = k % nst;
        const uint32_t bar = smem_addr(&sbar[st]);
        unsigned char* const base = ring + (size_t)st * 2 * rpad;
        mbar_arrive_expect_tx(bar, (uint32_t)(2 * rowbytes));
        bulk_g2s(smem_addr(base), X + r * p.d, (uint32_t)rowbytes, bar);
        bulk_g2s(smem_addr(base + rpad), DY + r * p.d, (uint32_t)rowbytes, bar);
    };
    if constexpr (STG) {
        if (t == 0) {
            for (int k = 0; k < nst; ++k) mbar_init(smem_addr(&sbar[k]), 1);
            mbar_fence_init();
            for (int k = 0; k < nst; ++k) issue(k);
        }
        __syncthreads();
    }

    // parameters of my columns, held for every row (in registers, or SMS:
    // in shared memory, as are the accumulators)
    // PSM: the parameters in shared memory (1024-thread groups); SMS: the
    // accumulators too (the register form; the staged 1024-thread RMSNorm
    // keeps its single accumulator in registers and gives the rest of the
    // shared memory to its ring)
    constexpr bool PSM = bwd_sms(TPR * RPC);
    constexpr bool SMS = PSM && !STG;
    constexpr int NRP = PSM ? 1 : SLOTS;  // parameter vectors held in registers
    constexpr int NR = SMS ? 1 : SLOTS;   // accumulator vectors held in registers
    float* const s_par = bwd_state;
    float* const s_acc0 = bwd_state + SLOTS * VEC * TPR;
    float* const s_acc1 = s_acc0 + SLOTS * VEC * TPR;
    Vec<VEC> par[NRP];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        const int q = t + s * TPR;
        Vec<VEC> v;
        if (q < nv) {
            ldt_p(v, P0 + q * VEC, true);
        } else {
#pragma unroll
            for (int k = 0; k < VEC; ++k) v.v[k] = 0.f;
        }
        if constexpr (PSM)
            sms_st<VEC, TPR>(s_par, s, t, v);
        else
            par[s] = v;
    }
    Vec<VEC> acc0[PG ? NR : 1], acc1[(PG && OP == OP_LN) ? NR : 1];
    if constexpr (PG) {
        Vec<VEC> z;
#pragma unroll
        for (int k = 0; k < VEC; ++k) z.v[k] = 0.f;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            if constexpr (SMS) {
                sms_st<VEC, TPR>(s_acc0, s, t, z);
                if constexpr (OP == OP_LN) sms_st<VEC, TPR>(s_acc1, s, t, z);
            } else {
                acc0[s] = z;
                if constexpr (OP == OP_LN) acc1[s] = z;
            }
        }
    }

    // staged 16-bit LayerNorm: the saved statistics of the group's next row
    // are loaded one row ahead, so that a row whose stage is ready does not
    // wait for them (BF16 8192 x 8192 94.3 -> 82.5 us; FP32 rows, whose
    // stages take twice as long to land, were 1-2% slower with it)
    constexpr bool SPF = STG && OP == OP_LN && sizeof(T) == 2;
    float mu_next = 0.f, rs_next = 0.f;
    if constexpr (SPF) {
        if (group < p.rows) {
            mu_next = ld_p1(p.mean + group);
            rs_next = ld_p1(p.rstd + group);
        }
    }
    int it = 0;
    for (int64_t row = group; row < p.rows; row += ngroups, ++it) {
        // SMS: re-read the state every row rather than let it be hoisted
        // into registers that the held row needs
        if constexpr (PSM) asm volatile("" ::: "memory");
        const T* xr = X + row * p.d;
        const T* dyr = DY + row * p.d;
        Vec<VEC> xv[SLOTS], dv[SLOTS];
        float mu = 0.f, rs = 0.f;
        bool ok = true;   // staged: this thread's wait for the row completed
        if constexpr (STG) {
            if constexpr (SPF) {
                mu = mu_next;
                rs = rs_next;
                if (row + ngroups < p.rows) {
                    mu_next = ld_p1(p.mean + row + ngroups);
                    rs_next = ld_p1(p.rstd + row + ngroups);
                }
            } else if constexpr (OP == OP_LN) {
                mu = ld_p1(p.mean + row);
                rs = ld_p1(p.rstd + row);
            }
            const int st = it % nst;
            ok = mbar_wait_bounded(smem_addr(&sbar[st]), (uint32_t)((it / nst) & 1));
            const T* sx = reinterpret_cast<const T*>(ring + (size_t)st * 2 * rpad);
            const T* sdy = reinterpret_cast<const T*>(ring + (size_t)st * 2 * rpad + rpad);
#pragma unroll
            for (int s = 0; s < SLOTS; ++s) {
                const int q = t + s * TPR;
                if (ok && q < nv) {
                    lds_vec<T, VEC>(xv[s], sx + q * VEC);
                    lds_vec<T, VEC>(dv[s], sdy + q * VEC);
                } else {
#pragma unroll
                    for (int k = 0; k < VEC; ++k) xv[s].v[k] = dv[s].v[k] = 0.f;
                }
            }
        } else {
#pragma unroll
            for (int s = 0; s < SLOTS; ++s) {
                const int q = t + s * TPR;
                if (q < nv) {
                    ldt_x(xv[s], xr + q * VEC);
                    ldt_x(dv[s], dyr + q * VEC);
                } else {
#pragma unroll
                    for (int k = 0; k < VEC; ++k) xv[s].v[k] = dv[s].v[k] = 0.f;
                }
            }
            // vector layout (every row whole 16-byte chunks): the group's next
            // row is fetched into L2 while this one is reduced and written
            if constexpr (VEC > 1) {
                const int64_t nx = row + ngroups;
                if (t == 0 && nx < p.rows) {
                    prefetch_l2_bulk(X + nx * p.d, (uint32_t)(p.d * (int64_t)sizeof(T)));
                    prefetch_l2_bulk(DY + nx * p.d, (uint32_t)(p.d * (int64_t)sizeof(T)));
                }
            }
            if constexpr (OP == OP_LN) {
                mu = ld_p1(p.mean + row);
                rs = ld_p1(p.rstd + row);
            }
        }
        // two row sums: LN (sum g, sum g*xhat); RMS (sum x^2, sum g*x)
        float s1 = 0.f, s2 = 0.f;
        F2 s1p = f2s(0.f), s2p = f2s(0.f);
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            if (t + s * TPR < nv) {
                Vec<VEC> ps;
                if constexpr (PSM)
                    sms_ld<VEC, TPR>(ps, s_par, s, t);
                else
                    ps = par[s];
                if constexpr (VEC > 1) {
                    // adjacent elements in pairs (packed FP32): the two
                    // halves of s1p/s2p are the even and odd partial sums
#pragma unroll
                    for (int k = 0; k < VEC; k += 2) {
                        const F2 xk = f2(xv[s].v[k], xv[s].v[k + 1]);
                        const F2 gk = mul2(f2(dv[s].v[k], dv[s].v[k + 1]),
                                           f2(ps.v[k], ps.v[k + 1]));
                        if constexpr (OP == OP_LN) {
                            const F2 xh = mul2(sub2(xk, f2s(mu)), f2s(rs));
                            s1p = add2(s1p, gk);
                            s2p = fma2(gk, xh, s2p);
                        } else {
                            s1p = fma2(xk, xk, s1p);
                            s2p = fma2(gk, xk, s2p);
                        }
                    }
                } else {
                    const float gk = __fmul_rn(dv[s].v[0], ps.v[0]);
                    if constexpr (OP == OP_LN) {
                        const float xh = (xv[s].v[0] - mu) * rs;
                        s1 += gk;
                        s2 = fmaf(gk, xh, s2);
                    } else {
                        s1 = fmaf(xv[s].v[0], xv[s].v[0], s1);
                        s2 = fmaf(gk, xv[s].v[0], s2);
                    }
                }
            }
        }
        if constexpr (VEC > 1) {
            float a, b;
            f2_get(s1p, a, b);
            s1 = a + b;
            f2_get(s2p, a, b);
            s2 = a + b;
        }
        s1 = warp_sum(s1);
        s2 = warp_sum(s2);
        if constexpr (WPR > 1) {
            float(*slot)[2] = xch[it & (NBUF - 1)][g];
            if (lane == 0) {
                slot[w][0] = s1;
                slot[w][1] = s2;
            }
            if constexpr (STG) {
                if (!__syncthreads_and(ok)) {
                    // a wait ran out: record it, let this CTA's copies still
                    // in flight (rows it .. it + nst - 2) land, and leave
                    if (t == 0) {
                        if (p.err) atomicOr(p.err, kErrStagedTimeout);
                        for (int k = it; k < it + nst - 1; ++k)
                            if (group + (int64_t)k * ngroups < p.rows)
                                (void)mbar_wait_bounded(smem_addr(&sbar[k % nst]),
                                                        (uint32_t)((k / nst) & 1));
                    }
                    return;
                }
                // every thread is past its reads of the previous row's stage
                if (t == 0 && it >= 1) {
                    fence_proxy_async_smem();
                    issue(it - 1 + nst);
                }
            } else {
                named_sync(1 + g, TPR);
            }
            if constexpr (WPR >= 16) {
                // 16 or 32 partials: a shuffle reduction (every lane ends
                // with the same sums) rather than a serial chain of that
                // many shared-memory loads, which the 64 registers of a
                // 1024-thread CTA could not hold without spilling
                s1 = warp_sum(lane < WPR ? slot[lane][0] : 0.f);
                s2 = warp_sum(lane < WPR ? slot[lane][1] : 0.f);
            } else {
                s1 = 0.f;
                s2 = 0.f;
#pragma unroll
                for (int k = 0; k < WPR; ++k) {
                    s1 += slot[k][0];
                    s2 += slot[k][1];
                }
            }
        }
        float c1, c2;
        if constexpr (OP == OP_LN) {
            c1 = s1 * inv_d;
            c2 = s2 * inv_d;
        } else {
            rs = rsqrtf(s1 * inv_d + p.eps);
            c1 = 0.f;
            c2 = s2 * inv_d * rs * rs;
        }
        T* dxr = DX + row * p.d;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            const int q = t + s * TPR;
            if (q < nv) {
                Vec<VEC> o, ps, a0, a1;
                if constexpr (SMS) {
                    sms_ld<VEC, TPR>(ps, s_par, s, t);
                    if constexpr (PG) {
                        sms_ld<VEC, TPR>(a0, s_acc0, s, t);
                        if constexpr (OP == OP_LN) sms_ld<VEC, TPR>(a1, s_acc1, s, t);
                    }
                } else {
                    if constexpr (PSM)
                        sms_ld<VEC, TPR>(ps, s_par, s, t);
                    else
                        ps = par[s];
                    if constexpr (PG) {
                        a0 = acc0[s];
                        if constexpr (OP == OP_LN) a1 = acc1[s];
                    }
                }
                if constexpr (VEC > 1) {
                    // per element exactly the scalar sequence below, two
                    // elements per packed instruction
#pragma unroll
                    for (int k = 0; k < VEC; k += 2) {
                        const F2 xk = f2(xv[s].v[k], xv[s].v[k + 1]);
                        const F2 dk = f2(dv[s].v[k], dv[s].v[k + 1]);
                        const F2 gk = mul2(dk, f2(ps.v[k], ps.v[k + 1]));
                        F2 ok;
                        if constexpr (OP == OP_LN) {
                            const F2 xh = mul2(sub2(xk, f2s(mu)), f2s(rs));
                            ok = mul2(f2s(rs), fma2(xh, f2s(-c2), sub2(gk, f2s(c1))));
                            if constexpr (PG) {
                                const F2 u0 = add2(f2(a0.v[k], a0.v[k + 1]), dk);
                                const F2 u1 = fma2(dk, xh, f2(a1.v[k], a1.v[k + 1]));
                                f2_get(u0, a0.v[k], a0.v[k + 1]);
                                f2_get(u1, a1.v[k], a1.v[k + 1]);
                            }
                        } else {
                            ok = mul2(f2s(rs), fma2(xk, f2s(-c2), gk));
                            if constexpr (PG) {
                                const F2 u0 = fma2(dk, mul2(xk, f2s(rs)),
                                                   f2(a0.v[k], a0.v[k + 1]));
                                f2_get(u0, a0.v[k], a0.v[k + 1]);
                            }
                        }
                        f2_get(ok, o.v[k], o.v[k + 1]);
                    }
                } else {
                    const float gk = __fmul_rn(dv[s].v[0], ps.v[0]);
                    if constexpr (OP == OP_LN) {
                        const float xh = (xv[s].v[0] - mu) * rs;
                        o.v[0] = rs * (gk - c1 - xh * c2);
                        if constexpr (PG) {
                            a0.v[0] += dv[s].v[0];
                            a1.v[0] = fmaf(dv[s].v[0], xh, a1.v[0]);
                        }
                    } else {
                        o.v[0] = rs * (gk - xv[s].v[0] * c2);
                        if constexpr (PG) a0.v[0] = fmaf(dv[s].v[0], xv[s].v[0] * rs, a0.v[0]);
                    }
                }
                if constexpr (PG) {
                    if constexpr (SMS) {
                        sms_st<VEC, TPR>(s_acc0, s, t, a0);
                        if constexpr (OP == OP_LN) sms_st<VEC, TPR>(s_acc1, s, t, a1);
                    } else {
                        acc0[s] = a0;
                        if constexpr (OP == OP_LN) acc1[s] = a1;
                    }
                }
                stt_y(dxr + q * VEC, o);
            }
        }
    }

    // let the column reduction's CTAs launch; they wait for this grid's writes
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if constexpr (PG) {
        float* wr = p.ws + (int64_t)blockIdx.x * p.ws_width;
        if constexpr (SMS) {
#pragma unroll
            for (int s = 0; s < SLOTS; ++s) {
                const int q = t + s * TPR;
                if (q < nv) {
                    Vec<VEC> a;
                    sms_ld<VEC, TPR>(a, s_acc0, s, t);
                    st_ws(wr + q * VEC, a);
                    if constexpr (OP == OP_LN) {
                        sms_ld<VEC, TPR>(a, s_acc1, s, t);
                        st_ws(wr + d + q * VEC, a);
                    }
                }
            }
        } else if constexpr (RPC == 1) {
#pragma unroll
            for (int s = 0; s < SLOTS; ++s) {
                const int q = t + s * TPR;
                if (q < nv) {
                    st_ws(wr + q * VEC, acc0[s]);
                    if constexpr (OP == OP_LN) st_ws(wr + d + q * VEC, acc1[s]);
                }
            }
        } else {
            // add the CTA's row groups, in group order, one slot at a time
            __shared__ __align__(16) float red[RPC][TPR * VEC];
            constexpr int HALVES = OP == OP_LN ? 2 : 1;
#pragma unroll
            for (int s = 0; s < SLOTS; ++s) {
#pragma unroll
                for (int hf = 0; hf < HALVES; ++hf) {
                    const Vec<VEC>& a = hf ? acc1[s] : acc0[s];
#pragma unroll
                    for (int k = 0; k < VEC; ++k) red[g][t * VEC + k] = a.v[k];
                    __syncthreads();
                    const int q = t + s * TPR;
                    if (g == 0 && q < nv) {
                        Vec<VEC> sum;
#pragma unroll
                        for (int k = 0; k < VEC; ++k) sum.v[k] = red[0][t * VEC + k];
#pragma unroll
                        for (int gg = 1; gg < RPC; ++gg)
#pragma unroll
                            for (int k = 0; k < VEC; ++k) sum.v[k] += red[gg][t * VEC + k];
                        st_ws(wr + hf * d + q * VEC, sum);
                    }
                    __syncthreads();
                }
            }
        }
    }
}

// Sum of the workspace's rows: out0[j] = sum_c ws[c][j] for j < d, out1[j - d]
// for d <= j < width (either output may be NULL), rounded once into TO. A CTA takes 32 columns and
// 32 slices of the rows: lane l of warp w adds rows w, w + 32, ... of column
// l with Kahan compensation (a warp reads 128 contiguous bytes per row), and
// warp 0 adds the 32 slice sums in slice order, again compensated.
constexpr int kReduceCols = 32;
constexpr int kReduceSlices = 32;

template <typename TO>
__global__ void __launch_bounds__(kReduceCols * kReduceSlices)
    column_reduce_kernel(const float* __restrict__ ws, int64_t rows, int64_t width, int64_t d,
                         TO* out0, TO* out1) {
    __shared__ float part[kReduceSlices][kReduceCols + 1];
    // wait until the row kernel's partials are written and visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31, slice = threadIdx.x >> 5;
    const int64_t j = (int64_t)blockIdx.x * kReduceCols + lane;
    float s = 0.f, c = 0.f;
    if (j < width) {
#pragma unroll 4
        for (int64_t r = slice; r < rows; r += kReduceSlices) {
            const float v = __ldcg(ws + r * width + j) - c;
            const float tsum = s + v;
            c = (tsum - s) - v;
            s = tsum;
        }
    }
    part[slice][lane] = s;
    __syncthreads();
    if (slice == 0 && j < width) {
        float u = 0.f, e = 0.f;
#pragma unroll
        for (int k = 0; k < kReduceSlices; ++k) {
            const float v = part[k][lane] - e;
            const float tsum = u + v;
            e = (tsum - u) - v;
            u = tsum;
        }
        if (j < d) {
            if (out0) stt_y1(out0 + j, u);
        } else if (out1) {
            stt_y1(out1 + (j - d), u);
        }
    }
}

}  // namespace rn

namespace rn {

template <int OP, typename T, int VEC, int SLOTS, int TPR, bool PG>
struct BwdInst {
    static constexpr int RPC = TPR < 256 ? 256 / TPR : 1;
    static constexpr int SMEM = bwd_sms_bytes(OP, VEC, SLOTS, TPR * RPC, PG);
    static cudaError_t launch(const BwdParams& p, int grid, cudaStream_t s) {
        bwd_kernel<OP, T, VEC, SLOTS, TPR, RPC, PG><<<grid, TPR * RPC, SMEM, s>>>(p);
        return cudaGetLastError();
    }
    // the limit is per function and process-wide; raising it again is harmless
    static cudaError_t prepare() {
        return cudaFuncSetAttribute(bwd_kernel<OP, T, VEC, SLOTS, TPR, RPC, PG>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    }
    static const BwdEntry entry;
};

template <int OP, typename T, int VEC, int SLOTS, int TPR, bool PG>
const BwdEntry BwdInst<OP, T, VEC, SLOTS, TPR, PG>::entry = {
    (const void*)&bwd_kernel<OP, T, VEC, SLOTS, TPR, BwdInst<OP, T, VEC, SLOTS, TPR, PG>::RPC, PG>,
    TPR * BwdInst<OP, T, VEC, SLOTS, TPR, PG>::RPC, BwdInst<OP, T, VEC, SLOTS, TPR, PG>::RPC,
    BwdInst<OP, T, VEC, SLOTS, TPR, PG>::SMEM, &BwdInst<OP, T, VEC, SLOTS, TPR, PG>::launch,
    // (any dynamic shared memory raises the limit: the default 48 KB counts
    // the static shared memory too)
    BwdInst<OP, T, VEC, SLOTS, TPR, PG>::SMEM > 0 ? &BwdInst<OP, T, VEC, SLOTS, TPR, PG>::prepare
                                                  : nullptr};

// Staged instances: the ring's size follows d and p.stages, so the dynamic
// shared memory is set per launch and its limit raised once to the whole
// budget.
template <int OP, typename T, int SLOTS, int TPR, bool PG>
struct BwdStagedInst {
    static constexpr int VEC = Elem<T>::kVec;
    // the parameter plane of 1024-thread groups, ahead of the ring
    static constexpr int PAR = bwd_sms(TPR) ? SLOTS * VEC * TPR * 4 : 0;
    static cudaError_t launch(const BwdParams& p, int grid, cudaStream_t s) {
        const int smem = PAR + (int)(p.stages * bwd_stage_bytes(p.d, (int)sizeof(T)));
        bwd_kernel<OP, T, VEC, SLOTS, TPR, 1, PG, true><<<grid, TPR, smem, s>>>(p);
        return cudaGetLastError();
    }
    static cudaError_t prepare() {
        return cudaFuncSetAttribute(bwd_kernel<OP, T, VEC, SLOTS, TPR, 1, PG, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kBwdStagedSmemBudget);
    }
    static const BwdEntry entry;
};

template <int OP, typename T, int SLOTS, int TPR, bool PG>
const BwdEntry BwdStagedInst<OP, T, SLOTS, TPR, PG>::entry = {
    (const void*)&bwd_kernel<OP, T, Elem<T>::kVec, SLOTS, TPR, 1, PG, true>, TPR, 1,
    BwdStagedInst<OP, T, SLOTS, TPR, PG>::PAR, &BwdStagedInst<OP, T, SLOTS, TPR, PG>::launch,
    &BwdStagedInst<OP, T, SLOTS, TPR, PG>::prepare, 1};

// The staged shapes the planner reaches: 256 or 512 threads per row and,
// since it takes the fewest threads that hold the row, more than half the
// held vectors per thread (FP32: 3 or 4 quads; 16-bit: 2 vectors of 8).
template <int OP, typename T, bool PG>
const BwdEntry* bwd_staged_pick(int slots, int tpr) {
    if constexpr (sizeof(T) == 4) {
        if (tpr == 64 && slots == 3) return &BwdStagedInst<OP, T, 3, 64, PG>::entry;
        if (tpr == 64 && slots == 4) return &BwdStagedInst<OP, T, 4, 64, PG>::entry;
        if (tpr == 128 && slots == 3) return &BwdStagedInst<OP, T, 3, 128, PG>::entry;
        if (tpr == 128 && slots == 4) return &BwdStagedInst<OP, T, 4, 128, PG>::entry;
        if (tpr == 256 && slots == 3) return &BwdStagedInst<OP, T, 3, 256, PG>::entry;
        if (tpr == 256 && slots == 4) return &BwdStagedInst<OP, T, 4, 256, PG>::entry;
        if (tpr == 512 && slots == 3) return &BwdStagedInst<OP, T, 3, 512, PG>::entry;
        if (tpr == 512 && slots == 4) return &BwdStagedInst<OP, T, 4, 512, PG>::entry;
    } else {
        if (tpr == 64 && slots == 2) return &BwdStagedInst<OP, T, 2, 64, PG>::entry;
        if (tpr == 128 && slots == 2) return &BwdStagedInst<OP, T, 2, 128, PG>::entry;
        if (tpr == 256 && slots == 2) return &BwdStagedInst<OP, T, 2, 256, PG>::entry;
        if (tpr == 512 && slots == 2) return &BwdStagedInst<OP, T, 2, 512, PG>::entry;
        if constexpr (OP == OP_RMS)
            if (tpr == 1024 && slots == 2) return &BwdStagedInst<OP, T, 2, 1024, PG>::entry;
    }
    return nullptr;
}

template <typename T>
const BwdEntry* bwd_staged_pick_type(int op, int slots, int tpr, bool pg) {
    if (op == OP_LN)
        return pg ? bwd_staged_pick<OP_LN, T, true>(slots, tpr)
                  : bwd_staged_pick<OP_LN, T, false>(slots, tpr);
    return pg ? bwd_staged_pick<OP_RMS, T, true>(slots, tpr)
              : bwd_staged_pick<OP_RMS, T, false>(slots, tpr);
}

// Vectors a backward thread holds: up to 16 floats of x and of dy (4 FP32 or
// 2 16-bit vectors), or 8 scalars.
template <int VEC>
constexpr int bwd_max_slots() {
    return VEC == 1 ? 8 : 16 / VEC;
}

// The shapes the planner reaches: it takes the fewest threads that hold the
// row, so rows of 64 or more threads hold more than half of a thread's
// vectors (FP32: 3 or 4 quads; 16-bit: 2 vectors of 8), and scalar rows of
// 64 or more threads are given 8 slots; rows of one warp take any count.
// Nothing else is compiled.
template <int VEC, int S, int TPR>
constexpr bool bwd_reachable() {
    constexpr int M = bwd_max_slots<VEC>();
    if (S > M) return false;
    if (TPR == 32) return true;
    return VEC == 1 ? S == 8 : 2 * S > M;
}

template <int OP, typename T, int VEC, int S, int TPR, bool PG>
const BwdEntry* bwd_inst_entry() {
    if constexpr (bwd_reachable<VEC, S, TPR>())
        return &BwdInst<OP, T, VEC, S, TPR, PG>::entry;
    else
        return nullptr;
}

template <int OP, typename T, int VEC, int TPR, bool PG>
const BwdEntry* bwd_pick_slots(int slots) {
    switch (slots) {
        case 1: return bwd_inst_entry<OP, T, VEC, 1, TPR, PG>();
        case 2: return bwd_inst_entry<OP, T, VEC, 2, TPR, PG>();
        case 3: return bwd_inst_entry<OP, T, VEC, 3, TPR, PG>();
        case 4: return bwd_inst_entry<OP, T, VEC, 4, TPR, PG>();
        case 8: return bwd_inst_entry<OP, T, VEC, 8, TPR, PG>();
        default: return nullptr;
    }
}

template <int OP, typename T, int VEC, bool PG>
const BwdEntry* bwd_pick(int slots, int tpr) {
    switch (tpr) {
        case 32: return bwd_pick_slots<OP, T, VEC, 32, PG>(slots);
        case 64: return bwd_pick_slots<OP, T, VEC, 64, PG>(slots);
        case 128: return bwd_pick_slots<OP, T, VEC, 128, PG>(slots);
        case 256: return bwd_pick_slots<OP, T, VEC, 256, PG>(slots);
        case 512: return bwd_pick_slots<OP, T, VEC, 512, PG>(slots);
        case 1024: return bwd_pick_slots<OP, T, VEC, 1024, PG>(slots);
        default: return nullptr;
    }
}

// Every (op, vector width, parameter-gradient) family of one storage type.
template <typename T>
const BwdEntry* bwd_pick_type(int op, int vec, int slots, int tpr, bool pg) {
    constexpr int V = Elem<T>::kVec;
    if (op == OP_LN) {
        if (vec == V) return pg ? bwd_pick<OP_LN, T, V, true>(slots, tpr) : bwd_pick<OP_LN, T, V, false>(slots, tpr);
        return pg ? bwd_pick<OP_LN, T, 1, true>(slots, tpr) : bwd_pick<OP_LN, T, 1, false>(slots, tpr);
    }
    if (vec == V) return pg ? bwd_pick<OP_RMS, T, V, true>(slots, tpr) : bwd_pick<OP_RMS, T, V, false>(slots, tpr);
    return pg ? bwd_pick<OP_RMS, T, 1, true>(slots, tpr) : bwd_pick<OP_RMS, T, 1, false>(slots, tpr);
}

template <typename TO>
cudaError_t column_reduce_t(const float* ws, int64_t rows, int64_t width, int64_t d, void* out0,
                            void* out1, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((width + kReduceCols - 1) / kReduceCols));
    cfg.blockDim = dim3(kReduceCols * kReduceSlices);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, column_reduce_kernel<TO>, ws, rows, width, d,
                              static_cast<TO*>(out0), static_cast<TO*>(out1));
}

}  // namespace rn
