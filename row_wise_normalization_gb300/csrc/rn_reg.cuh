// rn_reg.cuh -- register-held row kernels (warp per row, or a CTA per row).
//
// Shape of the computation, for one row of width d:
//   1. every thread issues all of its loads of the row up front: SLOTS
//      vectors of VEC floats (128-bit loads when VEC == 4), plus at
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
// FP32 vector rows, and the 16-bit rows (widened to FP32) of one warp or of
// a CTA's LayerNorm, do their element-wise arithmetic on pairs of elements
// with the packed .f32x2 instructions (shift_sum_pairs and the helpers
// beside it), which halves the instructions a row takes.
//
// The grid is persistent (at most the resident CTA count); a row group walks
// rows g, g + step, ... With PF the loads of the next row are issued before
// the current row is reduced and stored, so every thread keeps a row's worth
// of loads in flight while it computes (software pipelining across rows, the
// grid-stride hypothesis of issue #54 taken one step further). With PP the
// parameter vectors are loaded into registers once per thread and reused for
// every row, which requires every row to start at the same 16-byte phase
// (d % 4 == 0; the host checks). Instances that hold neither the parameters
// nor a slice small enough to load them with the row stage them in shared
// memory once per CTA instead (SP, reg_sp_bytes). Nothing is loaded through
// the non-coherent path: the kernel ahead on the stream may still be writing
// when this one starts (programmatic dependent launch).
//
// Vector layout of a row: h scalars up to the first 16-byte boundary of the
// row (the "head peel", 0..3), nv aligned vectors, tl scalars of tail (0..3).
// Vector q goes to thread q % TPR, slot q / TPR; the h + tl <= 6 scalars go to
// threads 0..h+tl-1. Rows whose x and y differ in 16-byte phase use VEC = 1.
#pragma once

#include "rn_async.cuh"

namespace rn {

// Registers a thread of reg_kernel is budgeted: the held row (twice with
// prefetch), the parameters held across rows, and a fixed allowance for
// indices, statistics and addresses.
constexpr int reg_budget(int op, int vec, int slots, bool pf, bool pp, bool res = false) {
    return 48 + slots * vec * (pf ? 2 : 1) * (res ? 2 : 1) + (res && !pf ? slots * vec : 0) +
           (pp ? 8 + slots * vec * (op == 0 ? 2 : 1) : 0) + (vec == 1 ? 3 * slots : 0);
}

// Resident CTAs each kernel is compiled for, which sets its register cap
// (65536 registers per SM, allocated in units of 8 per thread). For the wide
// slices (6+ vectors per thread) the counts are the measured optima on
// GB300 (cold L2, against a same-session device-to-device copy; "wide" is 24+
// floats held per thread, 6+ FP32 or 3+ 16-bit vectors): with
// prefetch about 384 resident threads per SM (the two held rows keep enough
// bytes in flight, and the spare registers let loads issue early), without
// it about 768-1024. 16-bit storage runs its wide slices on rows of 128+
// threads without prefetch (see reg_prefetch) at 1024 resident threads per
// SM, LayerNorm rows of 256 threads at 768. Narrower slices fill the SM as
// far as the budget allows.
constexpr int reg_min_ctas(int threads, int op, int vec, int slots, bool pf, bool pp,
                           bool res = false, bool al = true, bool ps = false) {
    if (ps) {
        // parameters in shared memory (warp-per-row instances): as many CTAs
        // as the held row (two with prefetch) and a fixed allowance let fit,
        // so that without prefetch every row of a call up to that size is in
        // flight at once (LayerNorm FP32 d = 768: 72 registers, 7 CTAs of 128)
        // (FP32 rows of 8 vectors a lane need 8 more: at 80 registers they
        // spilled 4 bytes)
        const int per = ((48 + slots * vec * (pf ? 2 : 1) + (vec == 4 && slots == 8 ? 8 : 0) + 7) /
                         8) * 8;
        const int n = 65536 / (per * threads);
        return n < 1 ? 1 : (n > 16 ? 16 : n);
    }
    if (vec == 8 && slots * vec >= 24 && !pf && threads >= 128) {
        const int target = (op == 0 && threads == 256) ? 768 : 1024;
        return target / threads > 0 ? target / threads : 1;
    }
    if (vec > 1 && slots * vec >= 24 && !res) {
        if (pf) return threads == 64 ? 5 : (threads >= 384 ? 1 : 384 / threads);
        // without prefetch: 768 threads on 256-thread rows; below 256 threads
        // (the one-wave instances) 512, which leaves 128 registers (a wide
        // LayerNorm slice needs about 100) and no spills
        if (threads < 256) return 512 / threads;
        // the one-wave LayerNorm instances of 256 threads and 6-7 vectors
        // (their default instance prefetches): two CTAs, 128 registers and
        // no spill; at three CTAs they spilled 8-12 bytes and ran 12-13%
        // slower back to back (300 x 6144 5.50 -> 4.79 us, 300 x 7168
        // 6.11 -> 5.36 us; equal with the L2 flushed before each launch)
        if (threads == 256 && op == 0 && al && (slots == 6 || slots == 7)) return 2;
        return threads >= 1024 ? 1 : (threads == 512 ? 2 : 768 / threads);
    }
    // the general (unaligned) vector layout also carries the row's head
    // and tail scalars, their parameters and per-row alignment tests
    const int extra = (!al && vec > 1) ? 12 : 0;
    const int per = ((reg_budget(op, vec, slots, pf, pp, res) + extra + 7) / 8) * 8;
    const int n = 65536 / (per * threads);
    return n < 1 ? 1 : (n > 32 ? 32 : n);
}

// One row as a thread holds it. With a residual (RES) the residual slice is
// held apart (vr, er) until the row is processed, so that a prefetched row's
// loads stay in flight; add_residual() then folds it into v and e.
template <int VEC, int SLOTS, bool RES = false>
struct HeldRow {
    Vec<VEC> v[SLOTS];
    Vec<VEC> vr[RES ? SLOTS : 1];
    float e, er;      // the thread's head/tail scalar (0 if none), its residual
    float k, kr;      // the row's first element and its residual (KLOAD only)
    int h, nv, tl;    // head peel, aligned vectors, tail of this row
};

template <int VEC, int SLOTS, bool RES>
__device__ __forceinline__ void add_residual(HeldRow<VEC, SLOTS, RES>& r) {
    if constexpr (RES) {
#pragma unroll
        for (int s = 0; s < SLOTS; ++s)
#pragma unroll
            for (int k = 0; k < VEC; ++k) r.v[s].v[k] = r.v[s].v[k] + r.vr[s].v[k];
        r.e = r.e + r.er;
        r.k = r.k + r.kr;
    }
}

// Loads one row of x (and of the residual rr when RES) at the phase of xr; the
// residual must share x's 16-byte phase (the host checks). T is the storage
// type (FP32: VEC 4 or 1; BF16/FP16: VEC 8 or 1); the row is held as FP32.
// KLOAD: every thread also loads the row's first element (the shift of the
// LayerNorm mean when several warps share the row).
template <typename T, int VEC, int SLOTS, int TPR, bool AL, bool RES = false, bool KLOAD = false>
__device__ __forceinline__ void load_row(HeldRow<VEC, SLOTS, RES>& r, const T* xr,
                                         const T* rr, int d, int t) {
    constexpr int LV = VEC == 8 ? 3 : (VEC == 4 ? 2 : 0);   // log2(VEC)
    if constexpr (AL) {
        r.h = 0;
        r.nv = d >> LV;
        r.tl = 0;
    } else if constexpr (VEC > 1) {
        r.h = head_peel_t(xr, d);
        r.nv = (d - r.h) >> LV;
        r.tl = d - r.h - VEC * r.nv;
    } else {
        r.h = 0;
        r.nv = d;
        r.tl = 0;
    }
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        const int q = t + s * TPR;
        if (q < r.nv) {
            ldt_x(r.v[s], xr + r.h + q * VEC);
            if constexpr (RES) ldt_x(r.vr[s], rr + r.h + q * VEC);
        } else {
#pragma unroll
            for (int k = 0; k < VEC; ++k) r.v[s].v[k] = 0.f;
            if constexpr (RES) {
#pragma unroll
                for (int k = 0; k < VEC; ++k) r.vr[s].v[k] = 0.f;
            }
        }
    }
    r.e = 0.f;
    r.er = 0.f;
    r.k = 0.f;
    r.kr = 0.f;
    if constexpr (KLOAD) {
        r.k = ldt_x1(xr);
        if constexpr (RES) r.kr = ldt_x1(rr);
    }
    if constexpr (VEC > 1 && !AL) {
        if (t < r.h + r.tl) {
            const int ei = (t < r.h) ? t : r.h + VEC * r.nv + (t - r.h);
            r.e = ldt_x1(xr + ei);
            if constexpr (RES) r.er = ldt_x1(rr + ei);
        }
    }
}

// 16-bit LayerNorm rows do more arithmetic per byte than FP32 ones; on rows
// of a CTA their element-wise statistics and output run on adjacent pairs with the packed
// FP32 instructions (each half rounded as the scalar instruction would be;
// the sums become even/odd partial sums).
template <int VEC, int SLOTS, bool RES>
__device__ __forceinline__ float held_sum_pairs(const HeldRow<VEC, SLOTS, RES>& r) {
    F2 a = f2s(0.f);
#pragma unroll
    for (int s = 0; s < SLOTS; ++s)
#pragma unroll
        for (int k = 0; k < VEC; k += 2) a = add2(a, f2(r.v[s].v[k], r.v[s].v[k + 1]));
    float x0, x1;
    f2_get(a, x0, x1);
    return x0 + x1;
}
template <int VEC, int SLOTS, int TPR, bool RES>
__device__ __forceinline__ float held_m2_pairs(const HeldRow<VEC, SLOTS, RES>& r, float c, int t,
                                               int nv) {
    F2 m = f2s(0.f);
    const F2 c2 = f2s(c);
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        if (t + s * TPR < nv) {
#pragma unroll
            for (int k = 0; k < VEC; k += 2) {
                const F2 d = sub2(f2(r.v[s].v[k], r.v[s].v[k + 1]), c2);
                m = fma2(d, d, m);
            }
        }
    }
    float x0, x1;
    f2_get(m, x0, x1);
    return x0 + x1;
}

// FP32 rows held as 128-bit vectors (PK: VEC 4, no residual) run the same
// way, and apply the LayerNorm shift by the row's first element K to the
// held vectors in place, once; with one warp per row the centring by the
// row's shifted mean mu_s too. The output is then one packed multiply and
// one packed fused multiply-add per pair: the same roundings, in the same
// order, as the scalar ((x - K) - mu_s) * rs * gamma + beta, at half the
// instructions.
template <int VEC, int SLOTS, int TPR, bool RES>
__device__ __forceinline__ float shift_sum_pairs(HeldRow<VEC, SLOTS, RES>& r, float K, int t,
                                                 int nv) {
    const F2 k2 = f2s(K);
    F2 a = f2s(0.f);
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        if (t + s * TPR < nv) {
#pragma unroll
            for (int k = 0; k < VEC; k += 2) {
                const F2 d = sub2(f2(r.v[s].v[k], r.v[s].v[k + 1]), k2);
                f2_get(d, r.v[s].v[k], r.v[s].v[k + 1]);
                a = add2(a, d);
            }
        }
    }
    float x0, x1;
    f2_get(a, x0, x1);
    return x0 + x1;
}
template <int VEC, int SLOTS, int TPR, bool RES>
__device__ __forceinline__ float centre_m2_pairs(HeldRow<VEC, SLOTS, RES>& r, float c, int t,
                                                 int nv) {
    const F2 c2 = f2s(c);
    F2 m = f2s(0.f);
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        if (t + s * TPR < nv) {
#pragma unroll
            for (int k = 0; k < VEC; k += 2) {
                const F2 d = sub2(f2(r.v[s].v[k], r.v[s].v[k + 1]), c2);
                f2_get(d, r.v[s].v[k], r.v[s].v[k + 1]);
                m = fma2(d, d, m);
            }
        }
    }
    float x0, x1;
    f2_get(m, x0, x1);
    return x0 + x1;
}
template <int VEC, int SLOTS, bool RES>
__device__ __forceinline__ float held_ss_pairs(const HeldRow<VEC, SLOTS, RES>& r) {
    F2 a = f2s(0.f);
#pragma unroll
    for (int s = 0; s < SLOTS; ++s)
#pragma unroll
        for (int k = 0; k < VEC; k += 2) {   // unused slots hold 0
            const F2 x = f2(r.v[s].v[k], r.v[s].v[k + 1]);
            a = fma2(x, x, a);
        }
    float x0, x1;
    f2_get(a, x0, x1);
    return x0 + x1;
}
// The parameters (gamma/beta or w) of one held row's vectors and its
// head/tail scalar, for thread t of a row group of TPR threads.
template <int OP, typename T, int VEC, int SLOTS, int TPR>
__device__ __forceinline__ void load_row_params(Vec<VEC> (&a)[SLOTS],
                                                Vec<VEC> (&b)[OP == OP_LN ? SLOTS : 1],
                                                float& ae, float& be, const T* P0, const T* P1,
                                                int h, int nv, bool has_e, int ei, bool aligned,
                                                int t) {
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        const int q = t + s * TPR;
        if (q < nv) {
            ldt_p(a[s], P0 + h + q * VEC, aligned);
            if constexpr (OP == OP_LN) ldt_p(b[s], P1 + h + q * VEC, aligned);
        }
    }
    if (has_e) {
        ae = ldt_p1(P0 + ei);
        if constexpr (OP == OP_LN) be = ldt_p1(P1 + ei);
    }
}

// Statistics of a row that one warp holds (lane t): the shift K, the shifted
// mean mu_s, the mean and rs, as the warp-per-row and batched kernels both
// take them, so that the two agree bit for bit. FP32 LayerNorm works in the
// frame shifted by K (see reg_kernel). With PK (vector rows without a
// residual: FP32 and 16-bit storage) the arithmetic runs on packed pairs and
// the held vectors of a LayerNorm row leave centred in place: (x - K) - mu_s
// for FP32, x - mu for 16-bit storage (where mu_s is mu).
template <int OP, typename T, int VEC, int SLOTS, bool RES>
__device__ __forceinline__ void warp_row_stats(HeldRow<VEC, SLOTS, RES>& cur, int t, bool has_e,
                                               float fd, float eps, float& K, float& mu_s,
                                               float& mu, float& rs) {
    constexpr bool SHIFT = OP == OP_LN && sizeof(T) == 4;
    constexpr bool PK = VEC % 2 == 0 && !RES;
    const int h = cur.h, nv = cur.nv;
    if constexpr (OP == OP_LN) {
        float sum;
        if constexpr (SHIFT) {
            // lane 0 holds the row's first element: its head scalar, else its
            // first vector, else (no vectors) its tail scalar
            const float first = (h > 0 || nv == 0) ? cur.e : cur.v[0].v[0];
            K = __shfl_sync(0xffffffffu, first, 0);
            sum = has_e ? cur.e - K : 0.f;
            if constexpr (PK) {
                sum += shift_sum_pairs<VEC, SLOTS, 32, RES>(cur, K, t, nv);
            } else {
#pragma unroll
                for (int s = 0; s < SLOTS; ++s) {
                    if (t + s * 32 < nv) {
#pragma unroll
                        for (int k = 0; k < VEC; ++k) sum += cur.v[s].v[k] - K;
                    }
                }
            }
        } else if constexpr (PK) {
            sum = cur.e + held_sum_pairs(cur);   // unused slots hold 0
        } else {
            sum = cur.e;
#pragma unroll
            for (int s = 0; s < SLOTS; ++s)
#pragma unroll
                for (int k = 0; k < VEC; ++k) sum += cur.v[s].v[k];   // unused slots hold 0
        }
        mu_s = warp_sum(sum) / fd;
        mu = SHIFT ? K + mu_s : mu_s;
        // deviations in the shifted frame too: (x - K) - mu_s
        const float ce = SHIFT ? (cur.e - K) - mu_s : cur.e - mu;
        float m2 = has_e ? ce * ce : 0.f;
        if constexpr (PK) {
            m2 += centre_m2_pairs<VEC, SLOTS, 32, RES>(cur, mu_s, t, nv);
        } else {
#pragma unroll
            for (int s = 0; s < SLOTS; ++s) {
                if (t + s * 32 < nv) {
#pragma unroll
                    for (int k = 0; k < VEC; ++k) {
                        const float c = SHIFT ? (cur.v[s].v[k] - K) - mu_s : cur.v[s].v[k] - mu;
                        m2 = fmaf(c, c, m2);
                    }
                }
            }
        }
        rs = rsqrtf(warp_sum(m2) / fd + eps);
    } else {
        float ss = cur.e * cur.e;
        if constexpr (PK) {
            ss += held_ss_pairs(cur);
        } else {
#pragma unroll
            for (int s = 0; s < SLOTS; ++s)
#pragma unroll
                for (int k = 0; k < VEC; ++k) ss = fmaf(cur.v[s].v[k], cur.v[s].v[k], ss);
        }
        rs = rsqrtf(warp_sum(ss) / fd + eps);
    }
}

// Whether an instance loads each row's parameters together with the row
// (EP), so that their latency overlaps the row's own loads: slices of at
// most 8 floats without held or staged parameters.
template <int OP, int VEC, int SLOTS, bool PP, bool PS>
constexpr bool reg_early_params() {
    return !PP && !PS && SLOTS * VEC <= 8;
}

// Bytes of shared memory an instance stages its parameters in (0: none).
// PS instances always do; otherwise every instance that neither holds its
// parameters in registers (PP) nor loads them with the row (EP), as long as
// the copies of its resident CTAs take at most 136 KB of an SM (128 KB of
// parameters plus the padding of reg_sp_elems). Those instances would otherwise load the parameters
// from global memory after each row's reduction, where the dependent chain
// waits for them. Measured on GB300: LayerNorm 2048 x 4096 13.2 -> 12.5 us
// back to back (3 CTAs of 32 KB); but with 192 KB of an SM staged (LayerNorm
// 256 x 8 vectors, 3 CTAs of 64 KB) 320 -> 386 us at 32768 x 8192, as the
// L1 left beside it no longer held the loads in flight.
// Elements per staged array: the held vectors' span plus room for an
// unaligned row's head and tail scalars (at most 6), a whole number of
// 16-byte units so that the second array stays aligned.
template <int VEC, int SLOTS, int TPR>
constexpr int reg_sp_elems() {
    return SLOTS * TPR * VEC + 2 * VEC;
}

template <int OP, typename T, int VEC, int SLOTS, int TPR, int RPC, bool PF, bool PP, bool AL,
          bool RES, bool PS>
constexpr int reg_sp_bytes() {
    const int bytes = (OP == OP_LN ? 2 : 1) * reg_sp_elems<VEC, SLOTS, TPR>() * (int)sizeof(T);
    if (PS) return bytes;
    if (PP || reg_early_params<OP, VEC, SLOTS, PP, PS>()) return 0;
    const int ctas = reg_min_ctas(TPR * RPC, OP, VEC, SLOTS, PF, PP, RES, AL, PS);
    return ctas * bytes <= 136 * 1024 ? bytes : 0;
}

template <int OP, typename T, int VEC, int SLOTS, int TPR, int RPC, bool PF, bool PP, bool AL,
          bool RES, bool PS = false>
__global__ void __launch_bounds__(TPR * RPC,
                                  reg_min_ctas(TPR * RPC, OP, VEC, SLOTS, PF, PP, RES, AL, PS))
    reg_kernel(const Params p) {
    static_assert(TPR % 32 == 0 && TPR * RPC <= 1024, "bad CTA shape");
    static_assert(!PS || (AL && !PP && !RES && TPR == 32), "shared parameters: aligned warp rows");
    static_assert(VEC == 1 || VEC == Elem<T>::kVec, "a vector is one 128-bit access");
    static_assert(!PP || VEC > 1, "parameters are held only on the vector path");
    static_assert(!AL || VEC > 1, "the aligned layout is a vector layout");
    static_assert(!RES || sizeof(T) == 4, "the residual form is FP32");
    const T* X = reinterpret_cast<const T*>(p.x);
    const T* R = reinterpret_cast<const T*>(p.r);
    const T* P0 = reinterpret_cast<const T*>(p.p0);
    const T* P1 = reinterpret_cast<const T*>(p.p1);
    T* Y = reinterpret_cast<T*>(p.y);
    T* H = reinterpret_cast<T*>(p.h);
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
    // FP32 LayerNorm works in the frame shifted by K, the row's first
    // element: it sums x - K (summands of the order of the row's spread, not
    // of its mean), keeps mu_s = mean - K, and takes every deviation --
    // for the sum of squares and for the output -- as (x - K) - mu_s, so
    // neither rstd nor y loses accuracy as |mean| / sigma grows (with the
    // mean rounded to FP32, every deviation would carry half an ulp of the
    // mean). 16-bit storage carries 8-11 significant bits, far coarser.
    constexpr bool SHIFT = OP == OP_LN && sizeof(T) == 4;
    constexpr bool KLOAD = SHIFT && WPR > 1;
    // (16-bit pairs on CTA-per-row rows only: warp-per-row rows take their
    // statistics from warp_row_stats, which the batched kernel shares)
    constexpr bool PAIRS = OP == OP_LN && sizeof(T) == 2 && VEC == 8 && WPR > 1;
    // FP32 vector rows without a residual: packed pairs, the LayerNorm shift
    // (and, for warp rows, the centring) applied to the held vectors in place
    constexpr bool PK = sizeof(T) == 4 && VEC == 4 && !RES;
    // 16-bit warp rows without a residual: the same through warp_row_stats
    constexpr bool PKW = WPR == 1 && VEC == 8 && !RES;
    const int64_t step = (int64_t)gridDim.x * RPC;
    int64_t row = (int64_t)blockIdx.x * RPC + g;
    pdl_launch_dependents();
    HeldRow<VEC, SLOTS, RES> cur;
    // SP (parameters staged in shared memory, reg_sp_bytes): gamma/beta (w)
    // are copied into dynamic shared memory once, while the rows' loads are
    // in flight, and every row reads them from there -- no registers held
    // for them across rows, and no global load of them after a row's
    // reduction. Where the arrays are 16-byte aligned (always for aligned
    // rows, SPB), thread 0 has the bulk-copy engine make the copy and the
    // first row waits (bounded) for it before its output; thread 0's group
    // always has a row (the grid is at most one CTA per row group), so the
    // CTA outlives the copy. Otherwise every thread copies its share, then
    // the CTA meets once, before any group leaves.
    constexpr bool SP = reg_sp_bytes<OP, T, VEC, SLOTS, TPR, RPC, PF, PP, AL, RES, PS>() > 0;
    constexpr bool SPB = SP && AL;
    extern __shared__ __align__(16) unsigned char reg_dyn_smem[];
    __shared__ __align__(8) unsigned long long sp_bar;
    T* const sp0 = reinterpret_cast<T*>(reg_dyn_smem);
    T* const sp1 = sp0 + reg_sp_elems<VEC, SLOTS, TPR>();
    // bulk: the copy is made by the bulk-copy engine (arrays 16-byte aligned;
    // always for aligned rows); else by the threads behind one barrier
    bool bulk = true;
    if constexpr (SP) {
        if (threadIdx.x == 0) {
            mbar_init(smem_addr(&sp_bar), 1);
            mbar_fence_init();
        }
        __syncthreads();
        pdl_wait();                                  // no global access before this
        constexpr int E16 = 16 / (int)sizeof(T);     // elements in 16 bytes
        if constexpr (!SPB) bulk = aligned16(P0, 0) && (OP != OP_LN || aligned16(P1, 0));
        const bool active = row < p.rows;
        if (!bulk) {
            // the same decision in every thread of the CTA: copy, meet once
            if (active)
                load_row<T, VEC, SLOTS, TPR, AL, RES, KLOAD>(
                    cur, X + row * p.ldx, RES ? R + row * p.ldr : nullptr, d, t);
            for (int j = threadIdx.x; j < d; j += TPR * RPC) {
                sp0[j] = P0[j];
                if constexpr (OP == OP_LN) sp1[j] = P1[j];
            }
            __syncthreads();
            if (!active) return;                     // the whole group leaves together
        } else {
            if (!active) return;                     // the whole group leaves together
            load_row<T, VEC, SLOTS, TPR, AL, RES, KLOAD>(cur, X + row * p.ldx,
                                                         RES ? R + row * p.ldr : nullptr, d, t);
            if (threadIdx.x == 0) {
                // an unaligned row's last d % E16 elements: written by this
                // thread before its arrive, which releases them to the waiters
                const int body = AL ? d : d - d % E16;
                for (int j = body; j < d; ++j) {
                    sp0[j] = P0[j];
                    if constexpr (OP == OP_LN) sp1[j] = P1[j];
                }
                const uint32_t bytes = (uint32_t)body * (uint32_t)sizeof(T);   // 16 | bytes
                const uint32_t bar = smem_addr(&sp_bar);
                mbar_arrive_expect_tx(bar, (OP == OP_LN ? 2u : 1u) * bytes);
                if (bytes > 0) {
                    bulk_g2s(smem_addr(sp0), P0, bytes, bar);
                    if constexpr (OP == OP_LN) bulk_g2s(smem_addr(sp1), P1, bytes, bar);
                }
            }
        }
    } else {
        if (row >= p.rows) return;                   // the whole group leaves together
        pdl_wait();                                  // no global access before this
        load_row<T, VEC, SLOTS, TPR, AL, RES, KLOAD>(cur, X + row * p.ldx,
                                                     RES ? R + row * p.ldr : nullptr, d, t);
    }

    // Parameters held across rows (PP, only with AL): every row is aligned.
    Vec<VEC> pg[PP ? SLOTS : 1], pb[(PP && OP == OP_LN) ? SLOTS : 1];
    float pge = 0.f, pbe = 0.f;
    if constexpr (PP) {
        const bool pa0 = AL || aligned16(P0, cur.h);
        const bool pa1 = AL || OP != OP_LN || aligned16(P1, cur.h);
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            const int q = t + s * TPR;
            if (q < cur.nv) {
                ldt_p(pg[s], P0 + cur.h + q * VEC, pa0);
                if constexpr (OP == OP_LN) ldt_p(pb[s], P1 + cur.h + q * VEC, pa1);
            }
        }
        if (!AL && t < cur.h + cur.tl) {
            const int ei = (t < cur.h) ? t : cur.h + VEC * cur.nv + (t - cur.h);
            pge = ldt_p1(P0 + ei);
            if constexpr (OP == OP_LN) pbe = ldt_p1(P1 + ei);
        }
    }

    // Groups that keep few bytes in flight have the bulk-copy engine fetch,
    // into L2, the row they take next: a group works through its rows one
    // at a time, and the fetch covers the DRAM round trip its next load
    // would otherwise start with. That is the 1024-thread rows (one CTA
    // per SM, no prefetch) and 16-bit LayerNorm rows of 128+ threads
    // without prefetch (half the bytes per held register, more arithmetic
    // per byte). Measured on GB300, cold L2: LayerNorm 1024 x 32768
    // 62.0 -> 51.8 us, BF16 32768 x 8192 208.7 -> 177.0 us, BF16 8192 x 4096
    // 30.9 -> 28.2 us; where more bytes are already in flight it cost 2-7%
    // (FP32 32768 x 8192 326.5 -> 350 us), so it is off there.
    constexpr bool L2PF = AL && !RES && !PF &&
                          (TPR == 1024 || (sizeof(T) == 2 && OP == OP_LN && TPR >= 128));
    int it = 0;
    for (;; ++it) {
        const int64_t nrow = row + step;
        HeldRow<VEC, SLOTS, RES> nxt;
        if constexpr (PF) {
            if (nrow < p.rows)
                load_row<T, VEC, SLOTS, TPR, AL, RES, KLOAD>(nxt, X + nrow * p.ldx,
                                                             RES ? R + nrow * p.ldr : nullptr, d,
                                                             t);
        }
        if constexpr (L2PF) {
            const int64_t frow = PF ? nrow + step : nrow;
            if (t == 0 && frow < p.rows)
                prefetch_l2_bulk(X + frow * p.ldx, (uint32_t)((int64_t)d * sizeof(T)));
        }
        add_residual(cur);
        const int h = cur.h, nv = cur.nv, tl = cur.tl;
        const bool has_e = (VEC > 1) && !AL && (t < h + tl);
        const int ei = (t < h) ? t : h + VEC * nv + (t - h);

        // EP (early parameters): slices of at most 8 floats without held
        // parameters load this row's gamma/beta (w) now, so that the loads
        // overlap the reduction instead of following it -- on the short,
        // launch-bound rows the dependent chain is the whole kernel
        constexpr bool EP = reg_early_params<OP, VEC, SLOTS, PP, PS>();
        constexpr int NPA = EP ? SLOTS : 1;
        Vec<VEC> ea[NPA], eb[OP == OP_LN ? NPA : 1];
        float eae = 0.f, ebe = 0.f;
        bool pa = true;   // parameter vectors 16-byte aligned at this row's phase
        if constexpr (VEC > 1 && !PP && !AL) {
            pa = aligned16(P0, h);
            if constexpr (OP == OP_LN) pa = pa && aligned16(P1, h);
        }
        if constexpr (EP)
            load_row_params<OP, T, VEC, NPA, TPR>(ea, eb, eae, ebe, P0, P1, h, nv, has_e, ei, pa,
                                                  t);

        // ---- statistics ------------------------------------------------
        float mu = 0.f, rs, K = 0.f, mu_s = 0.f;   // mu_s = mu - K (SHIFT)
        if constexpr (WPR == 1) {
            warp_row_stats<OP, T, VEC, SLOTS, RES>(cur, t, has_e, fd, p.eps, K, mu_s, mu, rs);
        } else if constexpr (OP == OP_LN) {
            float sum;
            if constexpr (SHIFT) {
                K = cur.k;
                sum = has_e ? cur.e - K : 0.f;
                if constexpr (PK) {
                    sum += shift_sum_pairs<VEC, SLOTS, TPR, RES>(cur, K, t, nv);   // x -> x - K
                } else {
#pragma unroll
                    for (int s = 0; s < SLOTS; ++s) {
                        if (t + s * TPR < nv) {
#pragma unroll
                            for (int k = 0; k < VEC; ++k) sum += cur.v[s].v[k] - K;
                        }
                    }
                }
            } else {
                if constexpr (PAIRS) {
                    sum = cur.e + held_sum_pairs(cur);   // unused slots hold 0
                } else {
                    sum = cur.e;
#pragma unroll
                    for (int s = 0; s < SLOTS; ++s)
#pragma unroll
                        for (int k = 0; k < VEC; ++k) sum += cur.v[s].v[k];   // unused slots hold 0
                }
            }

            {
                const float wsum = warp_sum(sum);
                int nw = (w == 0) ? (h + tl) : 0;          // elements this warp holds
#pragma unroll
                for (int s = 0; s < SLOTS; ++s) {
                    const int rem = nv - s * TPR - 32 * w;
                    nw += VEC * (rem <= 0 ? 0 : (rem >= 32 ? 32 : rem));
                }
                const float wmean_s = nw > 0 ? wsum / (float)nw : 0.f;   // shifted by K
                // deviations from the warp mean, taken in the shifted frame
                const float ce = SHIFT ? (cur.e - K) - wmean_s : cur.e - wmean_s;
                float m2 = has_e ? ce * ce : 0.f;
                if constexpr (PAIRS || PK) {   // PK: the held vectors are x - K
                    m2 += held_m2_pairs<VEC, SLOTS, TPR, RES>(cur, wmean_s, t, nv);
                } else {
#pragma unroll
                    for (int s = 0; s < SLOTS; ++s) {
                        if (t + s * TPR < nv) {
#pragma unroll
                            for (int k = 0; k < VEC; ++k) {
                                const float c = SHIFT ? (cur.v[s].v[k] - K) - wmean_s
                                                      : cur.v[s].v[k] - wmean_s;
                                m2 = fmaf(c, c, m2);
                            }
                        }
                    }
                }
                m2 = warp_sum(m2);
                float(*slot)[NST] = xch[it & (NBUF - 1)][g];
                // the merge works on the shifted sums and means
                if (lane == 0)
                    *reinterpret_cast<float4*>(slot[w]) = make_float4((float)nw, wsum, wmean_s, m2);
                named_sync(1 + g, TPR);
                float M2;
                merge_ln_warps<WPR>(slot, lane, fd, mu_s, M2);
                mu = SHIFT ? K + mu_s : mu_s;
                rs = rsqrtf(M2 / fd + p.eps);
            }
        } else {
            float ss = cur.e * cur.e;
            if constexpr (PK) {
                ss += held_ss_pairs(cur);
            } else {
#pragma unroll
                for (int s = 0; s < SLOTS; ++s)
#pragma unroll
                    for (int k = 0; k < VEC; ++k) ss = fmaf(cur.v[s].v[k], cur.v[s].v[k], ss);
            }
            const float wss = warp_sum(ss);
            float(*slot)[NST] = xch[it & (NBUF - 1)][g];
            if (lane == 0) slot[w][0] = wss;
            named_sync(1 + g, TPR);
            ss = merge_sum_warps<WPR, NST>(slot, lane);
            rs = rsqrtf(ss / fd + p.eps);
        }

        // ---- normalize and store from the held registers ----------------
        if constexpr (SP) {
            if (it == 0 && bulk && !mbar_wait_bounded(smem_addr(&sp_bar), 0) && p.err)
                atomicOr(p.err, kErrParamsTimeout);   // the outputs are then not valid
        }
        T* yr = Y + row * p.ldy;
        T* hr = RES && p.h ? H + row * p.ldh : nullptr;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            const int q = t + s * TPR;
            if (q < nv) {
                const int j = h + q * VEC;
                Vec<VEC> a, b, o;
                if constexpr (PP) {
                    a = pg[s];
                    if constexpr (OP == OP_LN) b = pb[s];
                } else if constexpr (SP) {
                    // 16-byte aligned in shared memory when the row's head
                    // peel is whole vectors (always, for aligned rows)
                    const bool sa = AL || h % VEC == 0;
                    lds_vec_at<T, VEC>(a, sp0 + j, sa);
                    if constexpr (OP == OP_LN) lds_vec_at<T, VEC>(b, sp1 + j, sa);
                } else if constexpr (EP) {
                    a = ea[s];
                    if constexpr (OP == OP_LN) b = eb[s];
                } else {
                    ldt_p(a, P0 + j, pa);
                    if constexpr (OP == OP_LN) ldt_p(b, P1 + j, pa);
                }
                if constexpr (PK || PKW) {
                    // LayerNorm: warp rows hold their centred values, FP32
                    // CTA rows x - K
                    o = out_pairs<OP, (OP == OP_LN && WPR > 1), VEC>(cur.v[s], a, b, mu_s, rs);
                } else if constexpr (PAIRS) {
#pragma unroll
                    for (int k = 0; k < VEC; k += 2) {
                        const F2 xo = mul2(sub2(f2(cur.v[s].v[k], cur.v[s].v[k + 1]), f2s(mu)),
                                           f2s(rs));
                        f2_get(fma2(xo, f2(a.v[k], a.v[k + 1]), f2(b.v[k], b.v[k + 1])), o.v[k],
                               o.v[k + 1]);
                    }
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
                if constexpr (RES) {
                    if (hr) stt_y(hr + j, cur.v[s]);
                }
            }
        }
        if (RES && has_e && hr) stt_y1(hr + ei, cur.e);
        if (has_e) {
            const float a =
                PP ? pge : (EP ? eae : (SP ? lds_f(sp0 + ei) : ldt_p1(P0 + ei)));
            float o;
            if constexpr (OP == OP_LN)
                o = fmaf((SHIFT ? (cur.e - K) - mu_s : cur.e - mu) * rs, a,
                         PP ? pbe : (EP ? ebe : (SP ? lds_f(sp1 + ei) : ldt_p1(P1 + ei))));
            else
                o = cur.e * rs * a;
            stt_y1(yr + ei, o);
        }
        if constexpr (OP == OP_LN) {
            if (t == 0) {
                if (p.mean) p.mean[row] = mu;
                if (p.rstd) p.rstd[row] = rs;
            }
        }

        if (nrow >= p.rows) break;
        row = nrow;
        if constexpr (PF)
            cur = nxt;
        else
            load_row<T, VEC, SLOTS, TPR, AL, RES, KLOAD>(cur, X + row * p.ldx,
                                                         RES ? R + row * p.ldr : nullptr, d, t);
    }
}

// ---------------------------------------------------------------------------
// Configurations and their registry entries (the choice of PF and PP per
// configuration is in rn_params.h, shared with the host-side planner).
// ---------------------------------------------------------------------------
// AL (all aligned): x, y and the parameter vectors are 16-byte aligned and
// d % 4 == 0, so every row is whole 128-bit vectors -- no head/tail scalars
// and no per-row alignment tests (the common case: allocators align to 256
// bytes). PP is only compiled with AL.
// NOPF: the same configuration compiled without prefetch at the no-prefetch
// occupancy, for calls whose rows all fit in one wave of it (nothing to
// overlap a prefetch with); only where the default instance prefetches.
// PS: the one-wave warp-per-row instances with the parameters staged in
// shared memory (reg_sp_bytes stages them in others too).
template <int OP, typename T, int VEC, int SLOTS, int TPR, bool PP, bool AL, bool RES,
          bool NOPF = false, bool PS = false>
struct RegInst {
    static constexpr int RPC = reg_rows_per_cta(OP, VEC, SLOTS, TPR, RES, AL);
    static constexpr bool PF = NOPF ? false : reg_prefetch(VEC, SLOTS, TPR, RES);
    static constexpr int SMEM = reg_sp_bytes<OP, T, VEC, SLOTS, TPR, RPC, PF, PP, AL, RES, PS>();
    static cudaError_t launch(const Params& p, int grid, cudaStream_t s) {
        return launch_pdl(reg_kernel<OP, T, VEC, SLOTS, TPR, RPC, PF, PP, AL, RES, PS>,
                          (unsigned)grid, TPR * RPC, SMEM, s, p);
    }
    // the limit is per function and process-wide; raising it again is harmless
    static cudaError_t prepare(int) {
        return cudaFuncSetAttribute(reg_kernel<OP, T, VEC, SLOTS, TPR, RPC, PF, PP, AL, RES, PS>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    }
    static const KernelEntry entry;
};

template <int OP, typename T, int VEC, int SLOTS, int TPR, bool PP, bool AL, bool RES, bool NOPF,
          bool PS>
const KernelEntry RegInst<OP, T, VEC, SLOTS, TPR, PP, AL, RES, NOPF, PS>::entry = {
    (const void*)&reg_kernel<OP, T, VEC, SLOTS, TPR,
                             RegInst<OP, T, VEC, SLOTS, TPR, PP, AL, RES, NOPF, PS>::RPC,
                             RegInst<OP, T, VEC, SLOTS, TPR, PP, AL, RES, NOPF, PS>::PF, PP, AL,
                             RES, PS>,
    TPR * RegInst<OP, T, VEC, SLOTS, TPR, PP, AL, RES, NOPF, PS>::RPC,
    RegInst<OP, T, VEC, SLOTS, TPR, PP, AL, RES, NOPF, PS>::RPC,
    RegInst<OP, T, VEC, SLOTS, TPR, PP, AL, RES, NOPF, PS>::SMEM,
    &RegInst<OP, T, VEC, SLOTS, TPR, PP, AL, RES, NOPF, PS>::launch,
    // (any dynamic shared memory raises the limit: the default 48 KB counts
    // the static shared memory too)
    RegInst<OP, T, VEC, SLOTS, TPR, PP, AL, RES, NOPF, PS>::SMEM > 0
        ? &RegInst<OP, T, VEC, SLOTS, TPR, PP, AL, RES, NOPF, PS>::prepare
        : nullptr};

// The warp-per-row instances with their parameters in shared memory: every
// slot count a row of up to 32 * 8 FP32 (32 * 4 16-bit) vectors needs, with
// (NOPF false) or without prefetch.
template <int OP, typename T, int VEC, int S, bool NOPF>
const KernelEntry* reg_ps_entry() {
    // with prefetch only the rows that would otherwise hold their parameters
    // in registers take it
    if constexpr (S <= 32 / VEC && (NOPF || reg_may_hold_params(VEC, S, 32)))
        return &RegInst<OP, T, VEC, S, 32, false, true, false, NOPF, true>::entry;
    else
        return nullptr;
}

template <int OP, typename T, int VEC, bool NOPF = true>
const KernelEntry* reg_pick_ps(int slots) {
    switch (slots) {
        case 1: return reg_ps_entry<OP, T, VEC, 1, NOPF>();
        case 2: return reg_ps_entry<OP, T, VEC, 2, NOPF>();
        case 3: return reg_ps_entry<OP, T, VEC, 3, NOPF>();
        case 4: return reg_ps_entry<OP, T, VEC, 4, NOPF>();
        case 5: return reg_ps_entry<OP, T, VEC, 5, NOPF>();
        case 6: return reg_ps_entry<OP, T, VEC, 6, NOPF>();
        case 7: return reg_ps_entry<OP, T, VEC, 7, NOPF>();
        case 8: return reg_ps_entry<OP, T, VEC, 8, NOPF>();
        default: return nullptr;
    }
}

// Slots per thread a family is compiled for: up to 8 FP32 vectors (32 floats),
// 4 16-bit vectors (32 floats) or 8 scalars; held parameters allow 24 floats,
// on the rows where the planner holds them (reg_may_hold_params).
template <typename T, int VEC, bool PP, int TPR>
constexpr int reg_max_slots() {
    if constexpr (PP) {
        int m = 0;
        for (int s = 1; s <= 24 / VEC; ++s)
            if (reg_may_hold_params(VEC, s, TPR)) m = s;
        return m;
    } else {
        return VEC == 1 ? 8 : 32 / VEC;
    }
}

// Configurations the planner can select. The CTA-per-row shape takes the
// fewest threads that hold the row, so a row of 128 or more threads holds
// more than half of a thread's slots (a row that fits in half of them takes
// half the threads); rows of 32 or 64 threads take any slot count (the warp
// range, and the CTA variant forced on narrow rows). Residual rows of 1024
// threads are refused by the planner (x and the residual do not fit the 64
// registers a thread of a 1024-thread CTA has). Nothing else is compiled.
template <int VEC, int S, int TPR, bool RES>
constexpr bool reg_reachable() {
    constexpr int maxs = VEC == 1 ? kMaxSlots : 32 / VEC;
    return !(RES && TPR == 1024) && (TPR <= 64 || 2 * S > maxs);
}

template <int OP, typename T, int VEC, int S, int TPR, bool PP, bool AL, bool RES, bool NOPF>
const KernelEntry* reg_inst_entry() {
    if constexpr (!reg_reachable<VEC, S, TPR, RES>())
        return nullptr;
    else if constexpr (AL && !PP && reg_may_hold_params(VEC, S, TPR))
        return nullptr;   // aligned rows of this shape hold their parameters (the PP sibling)
    else if constexpr (NOPF && !reg_prefetch(VEC, S, TPR, RES))
        return nullptr;   // the default instance already runs without prefetch
    else
        return &RegInst<OP, T, VEC, S, TPR, PP, AL, RES, NOPF>::entry;
}

template <int OP, typename T, int VEC, int TPR, bool PP, bool AL, bool RES, bool NOPF = false>
const KernelEntry* reg_pick_slots(int slots) {
    constexpr int M = reg_max_slots<T, VEC, PP, TPR>();
    if (slots < 1 || slots > M) return nullptr;
    switch (slots) {
        case 1: return reg_inst_entry<OP, T, VEC, 1, TPR, PP, AL, RES, NOPF>();
        case 2: if constexpr (M >= 2) return reg_inst_entry<OP, T, VEC, 2, TPR, PP, AL, RES, NOPF>(); else return nullptr;
        case 3: if constexpr (M >= 3) return reg_inst_entry<OP, T, VEC, 3, TPR, PP, AL, RES, NOPF>(); else return nullptr;
        case 4: if constexpr (M >= 4) return reg_inst_entry<OP, T, VEC, 4, TPR, PP, AL, RES, NOPF>(); else return nullptr;
        case 5: if constexpr (M >= 5) return reg_inst_entry<OP, T, VEC, 5, TPR, PP, AL, RES, NOPF>(); else return nullptr;
        case 6: if constexpr (M >= 6) return reg_inst_entry<OP, T, VEC, 6, TPR, PP, AL, RES, NOPF>(); else return nullptr;
        case 7: if constexpr (M >= 7) return reg_inst_entry<OP, T, VEC, 7, TPR, PP, AL, RES, NOPF>(); else return nullptr;
        case 8: if constexpr (M >= 8) return reg_inst_entry<OP, T, VEC, 8, TPR, PP, AL, RES, NOPF>(); else return nullptr;
        default: return nullptr;
    }
}

// (slots, tpr) -> entry for one (VEC, PP, AL) family; PP families exist for
// rows of at most 128 threads and 6 vectors per thread.
template <int OP, typename T, int VEC, bool PP, bool AL, bool RES = false, bool NOPF = false>
const KernelEntry* reg_pick(int slots, int tpr) {
    switch (tpr) {
        case 32: return reg_pick_slots<OP, T, VEC, 32, PP, AL, RES, NOPF>(slots);
        case 64: return reg_pick_slots<OP, T, VEC, 64, PP, AL, RES, NOPF>(slots);
        case 128: return reg_pick_slots<OP, T, VEC, 128, PP, AL, RES, NOPF>(slots);
        case 256: if constexpr (!PP) return reg_pick_slots<OP, T, VEC, 256, PP, AL, RES, NOPF>(slots); else return nullptr;
        case 512: if constexpr (!PP) return reg_pick_slots<OP, T, VEC, 512, PP, AL, RES, NOPF>(slots); else return nullptr;
        case 1024: if constexpr (!PP) return reg_pick_slots<OP, T, VEC, 1024, PP, AL, RES, NOPF>(slots); else return nullptr;
        default: return nullptr;
    }
}

}  // namespace rn
