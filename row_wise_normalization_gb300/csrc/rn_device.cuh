// rn_device.cuh -- device helpers shared by the row-normalization kernels:
// cache-hinted global loads and stores, warp and named-barrier primitives.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "rn_params.h"

namespace rn {

// ---------------------------------------------------------------------------
// Global memory access.
//
// x is streamed: read exactly once, so it bypasses L1 (no_allocate) and asks
// L2 to fetch whole 256-byte blocks. gamma/beta/w are re-read by every row, so
// they are cached in L1. y is written once and never re-read by the kernel, so
// it is stored with the streaming (.cs) hint.
// No load takes the non-coherent (.nc) path, which needs its data read-only
// for the whole life of the kernel: under programmatic dependent launch
// (below) a kernel's life starts while the kernel ahead of it may still be
// writing what this one reads. With .nc loads of x, ping-pong chains of calls
// on GB300 (each call reading the buffer the previous call wrote) read stale
// values in about 0.4 % of 2400 chains of the warp-per-row LayerNorm; with
// coherent loads, none in 8000.
// ---------------------------------------------------------------------------
// Programmatic dependent launch. The forward kernels are launched with
// programmatic stream serialization (launch_pdl in rn_params.h): the GPU may
// schedule such a kernel while the kernel ahead of it on the stream is still
// running, so its launch and CTA set-up overlap that kernel's tail. Each
// forward kernel therefore (1) lets the kernel behind it be scheduled as soon
// as all of its own CTAs are resident (every CTA signals at its start; a
// persistent grid is one wave, so no CTA of it waits for a slot the next
// kernel took), and (2) touches no global memory before pdl_wait() returns,
// which is when the kernel ahead has completed and its writes are visible.
// Without a kernel ahead (first launch, a copy or an event before it) the
// wait returns at once. That includes L2 prefetches: with one bulk L2
// prefetch of each row issued before the wait, a chain of calls on GB300 in
// which every call overwrote the buffer the previous call read, and read the
// one it wrote, returned stale values for about 1 % of the elements.
// Prefetches after the wait are safe.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Asks the bulk-copy engine to bring `bytes` (a multiple of 16) from a
// 16-byte-aligned global address into L2, without waiting for them.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ float4 ld_x4(const float* p) {
    float4 v;
    asm volatile("ld.global.L1::no_allocate.L2::256B.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float ld_x1(const float* p) {
    float v;
    asm volatile("ld.global.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float4 ld_p4(const float* p) {
    float4 v;
    asm volatile("ld.global.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float ld_p1(const float* p) {
    float v;
    asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_y4(float* p, float a, float b, float c, float d) {
    asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

__device__ __forceinline__ void st_y1(float* p, float a) {
    asm volatile("st.global.cs.f32 [%0], %1;" ::"l"(p), "f"(a) : "memory");
}

// Vector of VEC consecutive floats (VEC = 4: one 128-bit access; VEC = 1: scalar).
template <int VEC>
struct Vec {
    float v[VEC];
};

template <int VEC>
__device__ __forceinline__ void ld_x(Vec<VEC>& r, const float* p) {
    if constexpr (VEC == 4) {
        float4 t = ld_x4(p);
        r.v[0] = t.x; r.v[1] = t.y; r.v[2] = t.z; r.v[3] = t.w;
    } else {
        r.v[0] = ld_x1(p);
    }
}

// Parameter vector at column j. `aligned` says whether p + j is 16-byte aligned.
template <int VEC>
__device__ __forceinline__ void ld_p(Vec<VEC>& r, const float* p, bool aligned) {
    if constexpr (VEC == 4) {
        if (aligned) {
            float4 t = ld_p4(p);
            r.v[0] = t.x; r.v[1] = t.y; r.v[2] = t.z; r.v[3] = t.w;
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) r.v[k] = ld_p1(p + k);
        }
    } else {
        r.v[0] = ld_p1(p);
    }
}

template <int VEC>
__device__ __forceinline__ void st_y(float* p, const Vec<VEC>& r) {
    if constexpr (VEC == 4) {
        st_y4(p, r.v[0], r.v[1], r.v[2], r.v[3]);
    } else {
        st_y1(p, r.v[0]);
    }
}

// ---------------------------------------------------------------------------
// 16-bit storage (BF16, FP16): rows are read and written in the storage type
// and held as FP32. A 128-bit access moves 8 elements. BF16 -> FP32 is exact
// (the BF16 bits are the high half of the FP32 word); FP32 -> BF16/FP16 rounds
// to nearest even through CUDA's conversion intrinsics.
// ---------------------------------------------------------------------------
template <typename T>
struct Elem {
    static constexpr int kVec = 16 / (int)sizeof(T);   // elements per 128-bit vector
};

__device__ __forceinline__ void unpack2(uint32_t u, float& lo, float& hi, __nv_bfloat16*) {
    lo = __uint_as_float(u << 16);
    hi = __uint_as_float(u & 0xffff0000u);
}
__device__ __forceinline__ void unpack2(uint32_t u, float& lo, float& hi, __half*) {
    const __half2 h2 = *reinterpret_cast<const __half2*>(&u);
    const float2 f = __half22float2(h2);
    lo = f.x;
    hi = f.y;
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi, __nv_bfloat16*) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&b);
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi, __half*) {
    const __half2 b = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&b);
}
__device__ __forceinline__ float half_to_f(uint16_t u, __nv_bfloat16*) {
    return __uint_as_float((uint32_t)u << 16);
}
__device__ __forceinline__ float half_to_f(uint16_t u, __half*) {
    return __half2float(__ushort_as_half(u));
}
__device__ __forceinline__ uint16_t f_to_half(float f, __nv_bfloat16*) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ uint16_t f_to_half(float f, __half*) {
    return __half_as_ushort(__float2half_rn(f));
}

// Streamed 128-bit load of 8 16-bit elements as FP32.
template <typename T>
__device__ __forceinline__ void ld_x8(float* o, const T* p) {
    uint32_t a, b, c, d;
    asm volatile("ld.global.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "l"(p));
    unpack2(a, o[0], o[1], (T*)nullptr);
    unpack2(b, o[2], o[3], (T*)nullptr);
    unpack2(c, o[4], o[5], (T*)nullptr);
    unpack2(d, o[6], o[7], (T*)nullptr);
}
template <typename T>
__device__ __forceinline__ void ld_p8(float* o, const T* p) {
    uint32_t a, b, c, d;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "l"(p));
    unpack2(a, o[0], o[1], (T*)nullptr);
    unpack2(b, o[2], o[3], (T*)nullptr);
    unpack2(c, o[4], o[5], (T*)nullptr);
    unpack2(d, o[6], o[7], (T*)nullptr);
}
template <typename T>
__device__ __forceinline__ float ld_h1(const T* p, bool stream) {
    uint16_t u;
    if (stream)
        asm volatile("ld.global.L1::no_allocate.u16 %0, [%1];" : "=h"(u) : "l"(p));
    else
        asm volatile("ld.global.u16 %0, [%1];" : "=h"(u) : "l"(p));
    return half_to_f(u, (T*)nullptr);
}
template <typename T>
__device__ __forceinline__ void st_y8(T* p, const float* v) {
    const uint32_t a = pack2(v[0], v[1], (T*)nullptr), b = pack2(v[2], v[3], (T*)nullptr),
                   c = pack2(v[4], v[5], (T*)nullptr), d = pack2(v[6], v[7], (T*)nullptr);
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}
template <typename T>
__device__ __forceinline__ void st_h1(T* p, float v) {
    const uint16_t u = f_to_half(v, (T*)nullptr);
    asm volatile("st.global.cs.u16 [%0], %1;" ::"l"(p), "h"(u) : "memory");
}

// Typed accesses: T = float (VEC 4 or 1) or a 16-bit type (VEC 8 or 1).
template <typename T, int VEC>
__device__ __forceinline__ void ldt_x(Vec<VEC>& r, const T* p) {
    if constexpr (sizeof(T) == 4) {
        ld_x(r, reinterpret_cast<const float*>(p));
    } else if constexpr (VEC == 8) {
        ld_x8(r.v, p);
    } else {
        r.v[0] = ld_h1(p, true);
    }
}
template <typename T>
__device__ __forceinline__ float ldt_x1(const T* p) {
    if constexpr (sizeof(T) == 4)
        return ld_x1(reinterpret_cast<const float*>(p));
    else
        return ld_h1(p, true);
}
template <typename T>
__device__ __forceinline__ float ldt_p1(const T* p) {
    if constexpr (sizeof(T) == 4)
        return ld_p1(reinterpret_cast<const float*>(p));
    else
        return ld_h1(p, false);
}
template <typename T, int VEC>
__device__ __forceinline__ void ldt_p(Vec<VEC>& r, const T* p, bool aligned) {
    if constexpr (sizeof(T) == 4) {
        ld_p(r, reinterpret_cast<const float*>(p), aligned);
    } else if constexpr (VEC == 8) {
        if (aligned) {
            ld_p8(r.v, p);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) r.v[k] = ld_h1(p + k, false);
        }
    } else {
        r.v[0] = ld_h1(p, false);
    }
}
template <typename T, int VEC>
__device__ __forceinline__ void stt_y(T* p, const Vec<VEC>& r) {
    if constexpr (sizeof(T) == 4) {
        st_y(reinterpret_cast<float*>(p), r);
    } else if constexpr (VEC == 8) {
        st_y8(p, r.v);
    } else {
        st_h1(p, r.v[0]);
    }
}
template <typename T>
__device__ __forceinline__ void stt_y1(T* p, float v) {
    if constexpr (sizeof(T) == 4)
        st_y1(reinterpret_cast<float*>(p), v);
    else
        st_h1(p, v);
}

// Elements of T to the next 16-byte boundary of p (0 .. kVec-1), clamped to d.
template <typename T>
__device__ __forceinline__ int head_peel_t(const T* p, int64_t d) {
    constexpr int LS = sizeof(T) == 4 ? 2 : 1;   // log2(sizeof(T))
    int h = (int)(((0u - (unsigned)(uintptr_t)p) & 15u) >> LS);
    return h > d ? (int)d : h;
}

// True when p + j (elements of T) is 16-byte aligned.
template <typename T>
__device__ __forceinline__ bool aligned16(const T* p, int j) {
    constexpr int LS = sizeof(T) == 4 ? 2 : 1;   // log2(sizeof(T))
    constexpr unsigned M = 16 / sizeof(T) - 1;
    return ((((unsigned)(uintptr_t)p >> LS) + (unsigned)j) & M) == 0;
}

// ---------------------------------------------------------------------------
// Two FP32 values in one 64-bit register. Blackwell's packed FP32 pipe does
// add/sub/mul/fma on both halves in one instruction (.f32x2), each half
// rounded exactly as the scalar instruction rounds it (.rn; no contraction
// of an explicitly rounded mul or add into an fma), so element-wise work on
// adjacent pairs takes half the instructions for identical results.
// ---------------------------------------------------------------------------
struct F2 {
    unsigned long long r;
};
__device__ __forceinline__ F2 f2(float a, float b) {
    F2 o;
    asm("mov.b64 %0, {%1, %2};" : "=l"(o.r) : "f"(a), "f"(b));
    return o;
}
__device__ __forceinline__ F2 f2s(float a) { return f2(a, a); }
__device__ __forceinline__ void f2_get(F2 v, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v.r));
}
__device__ __forceinline__ F2 add2(F2 a, F2 b) {
    F2 o;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(o.r) : "l"(a.r), "l"(b.r));
    return o;
}
__device__ __forceinline__ F2 sub2(F2 a, F2 b) {
    F2 o;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(o.r) : "l"(a.r), "l"(b.r));
    return o;
}
__device__ __forceinline__ F2 mul2(F2 a, F2 b) {
    F2 o;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(o.r) : "l"(a.r), "l"(b.r));
    return o;
}
// a * b + c, one rounding per half
__device__ __forceinline__ F2 fma2(F2 a, F2 b, F2 c) {
    F2 o;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(o.r) : "l"(a.r), "l"(b.r), "l"(c.r));
    return o;
}

// One output vector from held values x (FP32, or 16-bit storage widened):
// LayerNorm (x - m) * rs * a + b (SUB) or x * rs * a + b, RMSNorm x * rs * a.
template <int OP, bool SUB, int VEC = 4>
__device__ __forceinline__ Vec<VEC> out_pairs(const Vec<VEC>& x, const Vec<VEC>& a,
                                              const Vec<VEC>& b, float m, float rs) {
    static_assert(VEC % 2 == 0, "pairs");
    Vec<VEC> o;
    const F2 r2 = f2s(rs), m2 = f2s(m);
#pragma unroll
    for (int k = 0; k < VEC; k += 2) {
        F2 c = f2(x.v[k], x.v[k + 1]);
        if constexpr (SUB) c = sub2(c, m2);
        if constexpr (OP == OP_LN)
            f2_get(fma2(mul2(c, r2), f2(a.v[k], a.v[k + 1]), f2(b.v[k], b.v[k + 1])), o.v[k],
                   o.v[k + 1]);
        else
            f2_get(mul2(mul2(c, r2), f2(a.v[k], a.v[k + 1])), o.v[k], o.v[k + 1]);
    }
    return o;
}

// Reductions.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Barrier over `nthreads` threads (a multiple of 32) using hardware barrier
// `id` (1..15; 0 is __syncthreads). Every thread of the named group arrives.
__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Cross-warp merge of per-warp LayerNorm partials published as float4
// (count, sum, mean, M2) in slot[0..NW): returns the row mean
// mu = sum_w sum_w / fd and M2 = sum_w [M2_w + n_w (mean_w - mu)^2] (the
// parallel-axis rule). Few warps: every thread walks the slots; many warps:
// lane k takes slot k and the warp reduces with shuffles.
template <int NW>
__device__ __forceinline__ void merge_ln_warps(const float (*slot)[4], int lane, float fd,
                                               float& mu, float& M2) {
    if constexpr (NW <= 8) {
        float tot = 0.f;
#pragma unroll
        for (int k = 0; k < NW; ++k) tot += slot[k][1];
        mu = tot / fd;
        float m2 = 0.f;
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const float4 q4 = *reinterpret_cast<const float4*>(slot[k]);
            const float dm = q4.z - mu;
            m2 += fmaf(q4.x * dm, dm, q4.w);
        }
        M2 = m2;
    } else {
        float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (lane < NW) q4 = *reinterpret_cast<const float4*>(slot[lane]);
        mu = warp_sum(q4.y) / fd;
        const float dm = q4.z - mu;
        M2 = warp_sum(lane < NW ? fmaf(q4.x * dm, dm, q4.w) : 0.f);
    }
}

// Sum of one float per warp published in slot[0..NW)[0].
template <int NW, int STRIDE>
__device__ __forceinline__ float merge_sum_warps(const float (*slot)[STRIDE], int lane) {
    if constexpr (NW <= 8) {
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NW; ++k) s += slot[k][0];
        return s;
    } else {
        return warp_sum(lane < NW ? slot[lane][0] : 0.f);
    }
}

// Elements to the next 16-byte boundary of p (0..3), clamped to d.
__device__ __forceinline__ int head_peel(const float* p, int64_t d) {
    int h = (int)((0u - (unsigned)((uintptr_t)p >> 2)) & 3u);
    return h > d ? (int)d : h;
}

// 16 raw bytes of a parameter vector (L1 allocated), and a
// 16-byte store to shared memory: the parameters staged per CTA.
template <typename T>
__device__ __forceinline__ uint4 ld_p_raw16(const T* p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
template <typename T>
__device__ __forceinline__ void st_shared_v4(T* p, uint4 v) {
    *reinterpret_cast<uint4*>(p) = v;
}

// One 128-bit vector of T (4 FP32 or 8 16-bit elements) from shared memory,
// widened to FP32. A plain load: the compiler keeps it after the preceding
// mbarrier wait (an asm statement that clobbers memory).
template <typename T, int VEC>
__device__ __forceinline__ void lds_vec(Vec<VEC>& r, const T* p) {
    static_assert(VEC * sizeof(T) == 16, "one 128-bit vector");
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    if constexpr (sizeof(T) == 4) {
        r.v[0] = __uint_as_float(u.x);
        r.v[1] = __uint_as_float(u.y);
        r.v[2] = __uint_as_float(u.z);
        r.v[3] = __uint_as_float(u.w);
    } else {
        unpack2(u.x, r.v[0], r.v[1], (T*)nullptr);
        unpack2(u.y, r.v[2], r.v[3], (T*)nullptr);
        unpack2(u.z, r.v[4], r.v[5], (T*)nullptr);
        unpack2(u.w, r.v[6], r.v[7], (T*)nullptr);
    }
}

// One element of a staged parameter array as FP32.
template <typename T>
__device__ __forceinline__ float lds_f(const T* p) {
    if constexpr (sizeof(T) == 4)
        return *reinterpret_cast<const float*>(p);
    else
        return half_to_f(*reinterpret_cast<const uint16_t*>(p), (T*)nullptr);
}

// VEC consecutive staged parameters from p, which is 16-byte aligned when
// `al` (one 128-bit load), else element by element.
template <typename T, int VEC>
__device__ __forceinline__ void lds_vec_at(Vec<VEC>& r, const T* p, bool al) {
    if constexpr (VEC * sizeof(T) == 16) {
        if (al) {
            lds_vec<T, VEC>(r, p);
            return;
        }
    }
#pragma unroll
    for (int k = 0; k < VEC; ++k) r.v[k] = lds_f(p + k);
}

}  // namespace rn
