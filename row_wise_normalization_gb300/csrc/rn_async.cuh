// rn_async.cuh -- mbarriers, bounded waits and 1-D bulk copies (the
// bulk-copy/TMA engine's untiled form), shared by the kernels that stage rows
// in shared memory. A wait gives up after a time limit instead of spinning
// forever; the caller then records the failure in the device error word it
// was given and returns.
#pragma once

#include "rn_device.cuh"

namespace rn {

constexpr unsigned kErrStagedTimeout = 1u;
constexpr unsigned kErrClusterTimeout = 2u;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // 1 s

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// 1-D bulk copy global -> this CTA's shared memory, completing `bytes` on bar.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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

}  // namespace rn
