// rownorm_api.cu -- the C ABI declared in include/rownorm.h: argument
// validation, width/alignment dispatch and the launch of one kernel per call.
#include <climits>
#include <cmath>
#include <cstdint>
#include <algorithm>
#include <cstring>
#include <iterator>
#include <utility>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "rownorm.h"
#include "rn_params.h"

namespace rn {
#define RN_DECL_FAMILY(OPN)                                      \
    const KernelEntry* reg_entry_##OPN##_v4(int, int);           \
    const KernelEntry* reg_entry_##OPN##_v4_al(int, int);        \
    const KernelEntry* reg_entry_##OPN##_v4_pp(int, int);        \
    const KernelEntry* reg_entry_##OPN##_v1(int, int);           \
    const KernelEntry* reg_entry_##OPN##_v4_res(int, int);       \
    const KernelEntry* reg_entry_##OPN##_v4_al_res(int, int);    \
    const KernelEntry* reg_entry_##OPN##_v4_pp_res(int, int);    \
    const KernelEntry* reg_entry_##OPN##_v1_res(int, int);
RN_DECL_FAMILY(ln)
RN_DECL_FAMILY(rms)
#undef RN_DECL_FAMILY
const KernelEntry* reg_entry_ps_f32(int, int);
const KernelEntry* reg_entry_pfps_f32(int, int);
const KernelEntry* reg_entry_ps_bf16(int, int);
const KernelEntry* reg_entry_ps_f16(int, int);
const KernelEntry* reg_entry_ln_v4_al_nopf(int, int);
const KernelEntry* reg_entry_rms_v4_al_nopf(int, int);
const KernelEntry* reg_entry_ln_v4_pp_nopf(int, int);
const KernelEntry* reg_entry_rms_v4_pp_nopf(int, int);
#define RN_DECL_FAMILY16(OPN, TN)                                 \
    const KernelEntry* reg_entry_##OPN##_##TN##_v8(int, int);     \
    const KernelEntry* reg_entry_##OPN##_##TN##_v8_al(int, int);  \
    const KernelEntry* reg_entry_##OPN##_##TN##_v8_pp(int, int);  \
    const KernelEntry* reg_entry_##OPN##_##TN##_v1(int, int);
RN_DECL_FAMILY16(ln, bf16)
RN_DECL_FAMILY16(rms, bf16)
RN_DECL_FAMILY16(ln, f16)
RN_DECL_FAMILY16(rms, f16)
#undef RN_DECL_FAMILY16

const KernelEntry* reg_entry(int op, int dtype, int vec, int slots, int tpr, bool pp, bool al,
                             bool res) {
    const bool ln = op == OP_LN;
    if (dtype != DT_F32) {
        if (res) return nullptr;
#define RN_PICK16(TN)                                                                         \
    if (vec != 8) return ln ? reg_entry_ln_##TN##_v1(slots, tpr) : reg_entry_rms_##TN##_v1(slots, tpr); \
    if (pp) return ln ? reg_entry_ln_##TN##_v8_pp(slots, tpr) : reg_entry_rms_##TN##_v8_pp(slots, tpr); \
    if (al) return ln ? reg_entry_ln_##TN##_v8_al(slots, tpr) : reg_entry_rms_##TN##_v8_al(slots, tpr); \
    return ln ? reg_entry_ln_##TN##_v8(slots, tpr) : reg_entry_rms_##TN##_v8(slots, tpr);
        if (dtype == DT_BF16) {
            RN_PICK16(bf16)
        }
        RN_PICK16(f16)
#undef RN_PICK16
    }
    if (res) {
        if (vec != 4) return ln ? reg_entry_ln_v1_res(slots, tpr) : reg_entry_rms_v1_res(slots, tpr);
        if (pp) return ln ? reg_entry_ln_v4_pp_res(slots, tpr) : reg_entry_rms_v4_pp_res(slots, tpr);
        if (al) return ln ? reg_entry_ln_v4_al_res(slots, tpr) : reg_entry_rms_v4_al_res(slots, tpr);
        return ln ? reg_entry_ln_v4_res(slots, tpr) : reg_entry_rms_v4_res(slots, tpr);
    }
    if (vec != 4) return ln ? reg_entry_ln_v1(slots, tpr) : reg_entry_rms_v1(slots, tpr);
    if (pp) return ln ? reg_entry_ln_v4_pp(slots, tpr) : reg_entry_rms_v4_pp(slots, tpr);
    if (al) return ln ? reg_entry_ln_v4_al(slots, tpr) : reg_entry_rms_v4_al(slots, tpr);
    return ln ? reg_entry_ln_v4(slots, tpr) : reg_entry_rms_v4(slots, tpr);
}
}  // namespace rn

namespace {

using namespace rn;

__global__ void empty_kernel() {}

thread_local int g_last_cuda_error = 0;

constexpr int64_t kMaxElems = (int64_t)1 << 61;

// One call, as the entry points received it.
struct Request {
    int op;                 // OP_LN or OP_RMS
    int dtype;              // DT_F32, DT_BF16 or DT_F16 (x, y, parameters, residual)
    bool res;               // residual variant
    const float* x;
    const float* r;         // residual (res only)
    const float* p0;        // gamma or w
    const float* p1;        // beta (LN) or NULL
    float* y;
    float* h;               // x + r written back (res only; may be NULL)
    float* mean;            // may be NULL
    float* rstd;            // may be NULL
    int64_t rows;
    int64_t d;
    float eps;
    // row strides in elements; 0 means contiguous (d). The strided entry
    // points reject strides below d before they get here.
    int64_t ldx = 0, ldy = 0;
};

int64_t ldx_of(const Request& q) { return q.ldx > 0 ? q.ldx : q.d; }
int64_t ldy_of(const Request& q) { return q.ldy > 0 ? q.ldy : q.d; }

// Elements from the first to the last element of a [rows][d] array with row
// stride ld (0 if rows == 0).
int64_t span(int64_t rows, int64_t d, int64_t ld) { return rows > 0 ? (rows - 1) * ld + d : 0; }

// Vectors (of `vec` elements) a row of width d needs held, excluding the
// scalars of an unaligned head and tail (fewer than 2 * vec).
int64_t row_units(int64_t d, int vec) { return d / vec; }

int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// Vectors a register-held thread may hold: 8 FP32 or 4 16-bit vectors (32
// floats either way), or 8 scalars.
int max_slots(int vec) { return vec == 1 ? kMaxSlots : 32 / vec; }

// Register-held CTA-per-row configuration: the fewest threads (>= 64, a power
// of two) that hold the row in at most `maxs` vectors each.
bool block_shape(int64_t units, int maxs, int* tpr, int* slots) {
    for (int t = 64; t <= 1024; t *= 2) {
        if (units <= (int64_t)t * maxs) {
            *tpr = t;
            *slots = units == 0 ? 1 : ceil_div(units, t);
            return true;
        }
    }
    return false;
}

// Cluster split: 256 threads per CTA and 4/6/8 quads per thread over the
// fewest CTAs (2..16); then 512 and 1024 threads with 16 CTAs of 8 quads.
bool cluster_shape(int64_t units, int* threads, int* cl, int* slots) {
    for (int c = 2; c <= kMaxCluster; c *= 2)
        for (int s : {4, 6, 8})
            if (units <= (int64_t)c * 256 * s) {
                *threads = 256;
                *cl = c;
                *slots = s;
                return true;
            }
    for (int t : {512, 1024})
        if (units <= (int64_t)kMaxCluster * t * 8) {
            *threads = t;
            *cl = kMaxCluster;
            *slots = 8;
            return true;
        }
    return false;
}

// Shared-memory staging: row buffers of the aligned body, as many as fit (at
// most kMaxStages). Returns false if one row does not fit.
bool staged_shape(int64_t d, int* stages, int* smem) {
    const int64_t sb = ((d / 4) * 16 + 127) / 128 * 128;
    if (sb > kStagedSmemBudget) return false;
    int n = sb == 0 ? kMaxStages : (int)(kStagedSmemBudget / sb);
    if (n > kMaxStages) n = kMaxStages;
    *stages = n;
    *smem = (int)(n * sb);
    return true;
}

uintptr_t addr(const void* p) { return (uintptr_t)p; }

int plan_impl(const Request& q, int variant, rn_plan* pl) {
    const int64_t d = q.d;
    if (d <= 0) return RN_ERR_SIZE;
    std::memset(pl, 0, sizeof(*pl));
    // 16-byte vectors need every streamed array (x, y, and with a residual r
    // and h) in the same 16-byte phase, so that one head peel aligns them all;
    // otherwise every access is scalar.
    // With row strides, rows keep that common phase when the strides agree
    // modulo a vector (residual rows are contiguous: their stride is d).
    uintptr_t phase = addr(q.x) ^ addr(q.y);
    if (q.res) {
        phase |= addr(q.x) ^ addr(q.r);
        if (q.h) phase |= addr(q.x) ^ addr(q.h);
    }
    const bool f32 = q.dtype == DT_F32;
    const int64_t vv = 16 / dtype_size(q.dtype);
    const int64_t ldx = ldx_of(q), ldy = ldy_of(q);
    const bool strides_agree =
        (ldx - ldy) % vv == 0 && (!q.res || (ldx - d) % vv == 0);
    const int vec = ((phase & 15u) == 0 && strides_agree) ? (int)vv : 1;
    const int64_t units = row_units(d, vec);
    const int maxs = max_slots(vec);
    pl->vec = vec;
    // Every row whole aligned vectors, parameters included.
    uintptr_t bases = addr(q.x) | addr(q.p0) | (q.op == OP_LN ? addr(q.p1) : 0);
    if (q.res) bases |= addr(q.r) | addr(q.h);
    const bool al = vec > 1 && d % vec == 0 && (bases & 15u) == 0 && ldx % vec == 0 &&
                    ldy % vec == 0;

    int v = variant;
    if (v == RN_VARIANT_AUTO) {
        int st, sm, ct, cc, cs;
        // Measured on GB300: one CTA per row holds up to 32768 floats and
        // beats splitting the row over a cluster there; beyond, the cluster
        // keeps the single HBM read that the staged and streaming kernels
        // give up or pay for in shared-memory passes.
        // With a residual, 1024-thread rows would hold x and the residual in
        // 64 registers and spill; those rows stream instead.
        // Aligned FP32 LayerNorm rows too wide for 512 threads go to the
        // cluster (now that its statistics meet without a cluster barrier and
        // its parameters stay in shared memory) rather than to one
        // 1024-thread CTA: measured on GB300, A/B in two runs, LayerNorm
        // 4096 x 20000 123 -> 109 us and 512 x 32768 34.2 -> 28.9 us (cold),
        // 1024 x 24576 35.9 -> 34.1 us (back to back), about even at
        // 2048 x 24576; RMSNorm 1024 x 20000 stays faster on one CTA
        // (27.6 against 29.6 us back to back).
        if (units <= 32 * maxs)
            v = RN_VARIANT_WARP;
        else if (q.op == OP_LN && f32 && !q.res && al && units > 512 * maxs &&
                 units <= 1024 * maxs && cluster_shape(units, &ct, &cc, &cs))
            v = RN_VARIANT_CLUSTER;
        else if (units <= (q.res ? 512 : 1024) * maxs)
            v = RN_VARIANT_BLOCK;
        else if (f32 && !q.res && vec == 4 && cluster_shape(units, &ct, &cc, &cs))
            v = RN_VARIANT_CLUSTER;
        else if (f32 && !q.res && vec == 4 && staged_shape(d, &st, &sm))
            v = RN_VARIANT_STAGED;
        else
            v = RN_VARIANT_STREAM;
    }
    pl->cluster = 1;
    switch (v) {
        case RN_VARIANT_WARP:
            if (units > 32 * maxs) return RN_ERR_VARIANT;
            pl->slots = units == 0 ? 1 : ceil_div(units, 32);
            pl->threads_per_row = 32;
            pl->rows_per_cta = kWarpRowsPerCta;
            pl->threads_per_cta = 32 * kWarpRowsPerCta;
            pl->prefetch = reg_prefetch(vec, pl->slots, 32, q.res);
            pl->aligned = al;
            pl->params_held = al && reg_may_hold_params(vec, pl->slots, 32);
            break;
        case RN_VARIANT_BLOCK: {
            int tpr, slots;
            if (!block_shape(units, maxs, &tpr, &slots)) return RN_ERR_VARIANT;
            // a residual row of 1024 threads would hold x and the residual in
            // the 64 registers such a thread has, and spill: not compiled
            if (q.res && tpr == 1024) return RN_ERR_VARIANT;
            pl->slots = slots;
            pl->threads_per_row = tpr;
            pl->rows_per_cta = reg_rows_per_cta(q.op, vec, slots, tpr, q.res, al);
            pl->threads_per_cta = tpr * pl->rows_per_cta;
            pl->prefetch = reg_prefetch(vec, slots, tpr, q.res);
            pl->aligned = al;
            pl->params_held = al && reg_may_hold_params(vec, slots, tpr);
            break;
        }
        case RN_VARIANT_STAGED: {
            int st, sm;
            if (!f32 || q.res || vec != 4 || !staged_shape(d, &st, &sm)) return RN_ERR_VARIANT;
            pl->slots = st;            // row buffers in the ring
            pl->threads_per_row = kStagedThreads;
            pl->rows_per_cta = 1;
            pl->threads_per_cta = kStagedThreads;
            pl->smem_bytes = sm;
            break;
        }
        case RN_VARIANT_CLUSTER: {
            int ct, cc, cs;
            if (!f32 || q.res || vec != 4 || !cluster_shape(units, &ct, &cc, &cs))
                return RN_ERR_VARIANT;
            pl->slots = cs;
            pl->threads_per_row = ct * cc;
            pl->rows_per_cta = 1;
            pl->threads_per_cta = ct;
            pl->cluster = cc;
            pl->aligned = al;
            break;
        }
        case RN_VARIANT_STREAM:
            pl->slots = 0;
            pl->threads_per_row = kStreamThreads;
            pl->rows_per_cta = 1;
            pl->threads_per_cta = kStreamThreads;
            break;
        default:
            return RN_ERR_VARIANT;
    }
    pl->variant = v;
    return RN_OK;
}

bool overlaps(const void* a, int64_t na, const void* b, int64_t nb) {
    if (!a || !b || na <= 0 || nb <= 0) return false;
    const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
    return pa < pb + (uintptr_t)nb && pb < pa + (uintptr_t)na;
}

bool misaligned(const void* p, int es) { return p && ((uintptr_t)p & (uintptr_t)(es - 1)); }

int validate(const Request& q) {
    if (q.dtype != DT_F32 && q.dtype != DT_BF16 && q.dtype != DT_F16) return RN_ERR_DTYPE;
    if (q.res && q.dtype != DT_F32) return RN_ERR_DTYPE;
    if (q.rows < 0 || q.d <= 0) return RN_ERR_SIZE;
    const int64_t ldx = ldx_of(q), ldy = ldy_of(q);
    if (ldx < q.d || ldy < q.d) return RN_ERR_SIZE;
    const int64_t ldmax = ldx > ldy ? ldx : ldy;
    if (q.rows > 0 && (q.rows - 1) > (kMaxElems - q.d) / ldmax) return RN_ERR_SIZE;
    if (!std::isfinite(q.eps) || q.eps < 0.f) return RN_ERR_EPS;
    if (q.rows == 0) return RN_OK;
    if (!q.x || !q.y || !q.p0 || (q.op == OP_LN && !q.p1) || (q.res && !q.r)) return RN_ERR_NULL;
    const int es = dtype_size(q.dtype);
    const void* data[] = {q.x, q.r, q.p0, q.p1, q.y, q.h};
    for (const void* p : data)
        if (misaligned(p, es)) return RN_ERR_ALIGN;
    if (misaligned(q.mean, 4) || misaligned(q.rstd, 4)) return RN_ERR_ALIGN;
    // spans from the first to the last element (strided rows: the gaps count)
    const int64_t nx = span(q.rows, q.d, ldx) * es, ny = span(q.rows, q.d, ldy) * es;
    const int64_t nd = q.rows * q.d * es, np = q.d * es, ns = q.rows * 4;
    // outputs against inputs and against each other
    const void* outs[4] = {q.y, q.h, q.mean, q.rstd};
    const int64_t nouts[4] = {ny, nd, ns, ns};
    const void* ins[4] = {q.x, q.r, q.p0, q.p1};
    const int64_t nins[4] = {nx, nd, np, np};
    for (int i = 0; i < 4; ++i) {
        for (int j = 0; j < 4; ++j)
            if (overlaps(outs[i], nouts[i], ins[j], nins[j])) return RN_ERR_ALIAS;
        for (int j = i + 1; j < 4; ++j)
            if (overlaps(outs[i], nouts[i], outs[j], nouts[j])) return RN_ERR_ALIAS;
    }
    return RN_OK;
}

// The current CUDA context's identifier, 0 if none is current (or the query
// failed). The per-thread caches below are keyed on it rather than on the
// device number: the function attributes that `prepare` raises belong to a
// context, and a context created anew for a device (after a device reset)
// needs them raised again.
unsigned long long ctx_now() {
    unsigned long long id = 0;
    return current_context_id(&id) == cudaSuccess ? id : 0;
}

// CTAs of `e` with `smem` bytes of dynamic shared memory that fit on the
// current device at once (0 on error). Raises the kernel's dynamic shared
// memory limit first when it needs more than the default.
int resident_ctas(const KernelEntry* e, int smem, cudaError_t* err) {
    if (smem == 0) smem = e->smem_bytes;   // instances that stage their parameters
    struct Cache {
        const void* fn;
        unsigned long long ctx;
        int smem;
        int n;
    };
    static thread_local Cache cache[32];
    static thread_local int cache_next = 0;
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return 0;
    const unsigned long long ctx = ctx_now();
    for (auto& c : cache)
        if (c.fn == e->fn && ctx != 0 && c.ctx == ctx && c.smem == smem && c.n > 0) return c.n;
    if (e->prepare) {
        *err = e->prepare(smem);
        if (*err != cudaSuccess) return 0;
    }
    int sms = 0, per_sm = 0;
    *err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (*err != cudaSuccess) return 0;
    *err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, e->fn, e->threads, smem);
    if (*err != cudaSuccess) return 0;
    if (per_sm < 1) {
        *err = cudaErrorInvalidConfiguration;
        return 0;
    }
    const int n = per_sm * sms;
    cache[cache_next] = {e->fn, ctx_now(), smem, n};
    cache_next = (cache_next + 1) % 32;
    return n;
}

// Clusters of `ce` that fit on the current device at once (0 on error).
int resident_clusters(const ClusterEntry* ce, cudaError_t* err) {
    struct Cache {
        const ClusterEntry* e;
        unsigned long long ctx;
        int n;
    };
    static thread_local Cache cache[16];
    static thread_local int cache_next = 0;
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return 0;
    const unsigned long long ctx = ctx_now();
    for (auto& c : cache)
        if (c.e == ce && ctx != 0 && c.ctx == ctx && c.n > 0) return c.n;
    *err = ce->prepare(0);
    if (*err != cudaSuccess) return 0;
    int n = 0;
    *err = ce->max_clusters(&n);
    if (*err != cudaSuccess) return 0;
    if (n < 1) {
        *err = cudaErrorInvalidConfiguration;
        return 0;
    }
    cache[cache_next] = {ce, ctx_now(), n};
    cache_next = (cache_next + 1) % 16;
    return n;
}

int fail_cuda(cudaError_t err) {
    g_last_cuda_error = (int)err;
    return RN_ERR_CUDA;
}

// Whether p is host memory the GPU reaches over the host link: pinned or
// registered (cudaMemoryTypeHost), or pageable memory read through the host
// page tables (cudaMemoryTypeUnregistered). The query succeeds for every
// address, allocated or not, unless the runtime itself is failing (no
// device, or a sticky error from an earlier fault); that counts as device
// memory, and the launch that follows reports the error.
bool host_resident(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost || a.type == cudaMemoryTypeUnregistered;
}

// Bytes of host-resident rows a call keeps in flight. With every row in
// flight in one wave, every read of a call is issued before its first write
// and the host link carries one direction at a time; a persistent grid that
// walks the rows (the next one prefetched where the plan says so) keeps both
// directions busy, and more requests in flight than the link needs only
// queue on it. Measured on GB300, pinned x and y, calls back to back, one
// wave against grids holding about 0.3 / 0.6 / 1.2 / 2.4 MB: LayerNorm FP32
// 4096 x 768 121 -> 80.6 (0.9 MB) / 81.8 (1.8) / 86.5 (3.6) us, 1024 x
// 4096 147 -> 104 (1.2) / 108 (2.4) / 117 (4.9) us, 1024 x 8192 262 ->
// 214 (0.7) / 206 (1.25) / 210 (2.5) us; BF16 4096 x 1024 78.1 -> 65.3
// (0.6) / 58.4 (1.2) / 63.0 (2.4) us, 4096 x 4096 239 -> 288 (0.3) / 206
// (0.6) / 208 (1.2) us; and FP32 65536 x 128 241 -> 300 us with only
// 0.3 MB in flight.
constexpr int64_t kLinkBytesInFlight = 1280 * 1024;

int run(const Request& q, int variant, void* stream) {
    if (variant < 0 || variant >= RN_VARIANT_COUNT) return RN_ERR_VARIANT;
    int st = validate(q);
    if (st != RN_OK) return st;
    if (q.rows == 0) return RN_OK;
    // The bulk-copy engine is given device memory only: the parameter
    // vectors, which the register-held kernels stage in shared memory by bulk
    // copies, must be in device memory, and rows in host memory do not take
    // the staged kernel (whose ring is filled by bulk copies; the streaming
    // kernel reads them with ordinary loads instead).
    if (host_resident(q.p0) || (q.op == OP_LN && host_resident(q.p1))) return RN_ERR_HOSTMEM;
    rn_plan pl;
    st = plan_impl(q, variant, &pl);
    if (st != RN_OK) return st;
    const bool x_host = host_resident(q.x);
    if (pl.variant == RN_VARIANT_STAGED && x_host) {
        if (variant != RN_VARIANT_AUTO) return RN_ERR_VARIANT;
        st = plan_impl(q, RN_VARIANT_STREAM, &pl);
        if (st != RN_OK) return st;
    }

    Params prm;
    prm.x = q.x;
    prm.y = q.y;
    prm.r = q.res ? q.r : nullptr;
    prm.h = q.res ? q.h : nullptr;
    prm.p0 = q.p0;
    prm.p1 = q.p1;
    prm.mean = q.mean;
    prm.rstd = q.rstd;
    prm.rows = q.rows;
    prm.d = q.d;
    prm.ldx = ldx_of(q);
    prm.ldy = ldy_of(q);
    prm.ldr = q.d;
    prm.ldh = q.d;
    prm.eps = q.eps;
    const cudaStream_t s = (cudaStream_t)stream;
    // where the kernels' bounded waits (cluster exchange, staged parameters)
    // report a timeout
    {
        const cudaError_t e0 = device_error_address(&prm.err);
        if (e0 != cudaSuccess) return fail_cuda(e0);
    }

    if (pl.variant == RN_VARIANT_CLUSTER) {
        const ClusterEntry* ce =
            cluster_entry(q.op, pl.slots, pl.threads_per_cta, pl.cluster, pl.aligned != 0);
        if (!ce) return RN_ERR_VARIANT;
        cudaError_t err = cudaSuccess;
        const int nclusters = resident_clusters(ce, &err);
        if (err != cudaSuccess) return fail_cuda(err);
        const int64_t want = q.rows < nclusters ? q.rows : nclusters;
        err = ce->launch(prm, (int)want * ce->cl, s);
        return err == cudaSuccess ? RN_OK : fail_cuda(err);
    }

    const KernelEntry* e = nullptr;
    if (pl.variant == RN_VARIANT_STREAM)
        e = stream_entry(q.op, q.dtype, pl.vec, q.res);
    else if (pl.variant == RN_VARIANT_STAGED)
        e = staged_entry(q.op, pl.slots);
    else
        e = reg_entry(q.op, q.dtype, pl.vec, pl.slots, pl.threads_per_row, pl.params_held != 0,
                      pl.aligned != 0, q.res);
    if (!e) return RN_ERR_VARIANT;

    cudaError_t err = cudaSuccess;
    int resident = resident_ctas(e, pl.smem_bytes, &err);
    if (err != cudaSuccess) return fail_cuda(err);
    const int64_t want = (q.rows + e->rows_per_cta - 1) / e->rows_per_cta;
    // Rows read from or written to host memory: the planned instance (it
    // prefetches the next row where the plan says so) on a persistent grid
    // that holds about kLinkBytesInFlight of rows, rather than the one-wave
    // instances below, so that each call's reads and writes share the link.
    const auto launch = [&](const KernelEntry* ke, int grid) {
        const cudaError_t e2 = ke->launch(prm, grid, s);
        return e2 == cudaSuccess ? RN_OK : fail_cuda(e2);
    };
    if ((pl.variant == RN_VARIANT_WARP || pl.variant == RN_VARIANT_BLOCK) &&
        (x_host || host_resident(q.y))) {
        const int64_t row_bytes = q.d * dtype_size(q.dtype) * (q.res ? 2 : 1);
        const int64_t cta_bytes = row_bytes * e->rows_per_cta * (pl.prefetch ? 2 : 1);
        int64_t cap = (kLinkBytesInFlight + cta_bytes - 1) / cta_bytes;
        if (cap > resident) cap = resident;
        return launch(e, (int)(want < cap ? want : cap));
    }
    // Aligned FP32 rows that prefetch: when every row fits in one wave of
    // the no-prefetch instance (more CTAs resident, no next row to overlap
    // with), run that instead. Measured on GB300: LayerNorm 1024 x 2048
    // 9.8 -> 8.4 us, 512 x 4096 10.2 -> 9.2 us (cold L2).
    if ((pl.variant == RN_VARIANT_WARP || pl.variant == RN_VARIANT_BLOCK) && pl.prefetch &&
        pl.aligned && q.dtype == DT_F32 && !q.res) {
        const bool ln = q.op == OP_LN;
        const KernelEntry* e1 =
            pl.params_held
                ? (ln ? reg_entry_ln_v4_pp_nopf(pl.slots, pl.threads_per_row)
                      : reg_entry_rms_v4_pp_nopf(pl.slots, pl.threads_per_row))
                : (ln ? reg_entry_ln_v4_al_nopf(pl.slots, pl.threads_per_row)
                      : reg_entry_rms_v4_al_nopf(pl.slots, pl.threads_per_row));
        if (e1 && want > resident) {
            const int r1 = resident_ctas(e1, 0, &err);
            if (err != cudaSuccess) return fail_cuda(err);
            if (want <= r1) {
                e = e1;
                resident = r1;
            }
        }
    }
    // Aligned warp-per-row rows without a residual that would give some warps
    // of the prefetching grid three rows or more (only the next row is
    // prefetched): when every row of the call fits in one wave of the
    // instance that stages the parameters in shared memory (no registers held
    // for them, so more CTAs resident), run that one, with every row in
    // flight at once. Measured on GB300, calls back to back over batches
    // larger than L2: LayerNorm 4096 x 768 6.41 -> 5.95 us, RMSNorm
    // 5.63 -> 5.43 us; where every warp has at most two rows (3000 x 1024:
    // 5.54 -> 6.14 us), or all rows already fit one wave of the instance
    // without prefetch (2048 x 768: 3.79 -> 4.75 us), the registers win.
    if (pl.variant == RN_VARIANT_WARP && pl.aligned && !q.res && want > 2 * (int64_t)resident &&
        e->rows_per_cta == kWarpRowsPerCta) {
        const KernelEntry* ep = q.dtype == DT_F32    ? reg_entry_ps_f32(q.op, pl.slots)
                                : q.dtype == DT_BF16 ? reg_entry_ps_bf16(q.op, pl.slots)
                                                     : reg_entry_ps_f16(q.op, pl.slots);
        if (ep) {
            const int rp = resident_ctas(ep, 0, &err);
            if (err != cudaSuccess) return fail_cuda(err);
            if (want <= rp) {
                e = ep;
                resident = rp;
            } else if (q.dtype == DT_F32 && q.op == OP_LN && pl.params_held && pl.slots >= 5) {
                // more rows than one wave of it: FP32 LayerNorm rows of 5-6
                // quads a lane, whose gamma and beta would take 40-48
                // registers, prefetch with the parameters in shared memory
                // instead (5 CTAs of 128 per SM at d = 768 rather than 3),
                // for up to 8 waves of rows. Measured on GB300, A/B in two
                // runs, back to back: 8192 x 768 10.11 -> 9.58 us, 5000 x
                // 768 7.05 -> 6.86 us, 16384 x 768 17.64 -> 17.45 us; but
                // 65536 x 768 63.9 -> 64.9 us, 12000 x 256 (2 quads)
                // 5.98 -> 6.21 us, RMSNorm 8192 x 768 9.37 -> 9.52 us.
                const KernelEntry* ef = reg_entry_pfps_f32(q.op, pl.slots);
                if (ef) {
                    const int rf = resident_ctas(ef, 0, &err);
                    if (err != cudaSuccess) return fail_cuda(err);
                    if (want <= 8 * (int64_t)rf) {
                        e = ef;
                        resident = rf;
                    }
                }
            }
        }
    }
    return launch(e, (int)(want < resident ? want : resident));
}

Request ln_request(const float* x, const float* res, const float* gamma, const float* beta,
                   float* h, float* y, float* mean, float* rstd, int64_t rows, int64_t d,
                   float eps, bool residual, int dtype = DT_F32) {
    return Request{OP_LN, dtype, residual, x, res, gamma, beta, y, h, mean, rstd, rows, d, eps};
}

Request rms_request(const float* x, const float* res, const float* w, float* h, float* y,
                    int64_t rows, int64_t d, float eps, bool residual, int dtype = DT_F32) {
    return Request{OP_RMS, dtype, residual, x, res, w, nullptr, y, h, nullptr, nullptr, rows, d,
                   eps};
}

// ---------------------------------------------------------------------------
// Batched small problems.
// ---------------------------------------------------------------------------
int batch_resident(const BatchEntry* e, cudaError_t* err) {
    struct Cache {
        const BatchEntry* e;
        int dev;
        int n;
    };
    static thread_local Cache cache[8];
    static thread_local int cache_next = 0;
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return 0;
    for (auto& c : cache)
        if (c.e == e && c.dev == dev && c.n > 0) return c.n;
    int sms = 0, per = 0;
    *err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (*err != cudaSuccess) return 0;
    *err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, e->fn, e->threads, 0);
    if (*err != cudaSuccess) return 0;
    if (per < 1) {
        *err = cudaErrorInvalidConfiguration;
        return 0;
    }
    cache[cache_next] = {e, dev, per * sms};
    cache_next = (cache_next + 1) % 8;
    return per * sms;
}

Request problem_request(int op, int dtype, const rn_problem& pr, float eps) {
    Request q = op == OP_LN
                    ? ln_request((const float*)pr.x, nullptr, (const float*)pr.p0,
                                 (const float*)pr.p1, nullptr, (float*)pr.y, pr.mean_out,
                                 pr.rstd_out, pr.rows, pr.d, eps, false, dtype)
                    : rms_request((const float*)pr.x, nullptr, (const float*)pr.p0, nullptr,
                                  (float*)pr.y, pr.rows, pr.d, eps, false, dtype);
    return q;
}

// Byte ranges a problem reads and writes.
void problem_ranges(int op, int dtype, const rn_problem& pr, const void* in[3], int64_t nin[3],
                    const void* out[3], int64_t nout[3]) {
    const int64_t es = dtype_size(dtype), n = pr.rows * pr.d * es;
    in[0] = pr.x;
    nin[0] = n;
    in[1] = pr.p0;
    nin[1] = pr.d * es;
    in[2] = op == OP_LN ? pr.p1 : nullptr;
    nin[2] = pr.d * es;
    out[0] = pr.y;
    nout[0] = n;
    out[1] = op == OP_LN ? pr.mean_out : nullptr;
    nout[1] = pr.rows * 4;
    out[2] = op == OP_LN ? pr.rstd_out : nullptr;
    nout[2] = pr.rows * 4;
}

int run_batched(int op, int dtype, const rn_problem* prs, int count, float eps, void* stream) {
    if (count < 0) return RN_ERR_SIZE;
    if (count == 0) return RN_OK;
    if (!prs) return RN_ERR_NULL;
    if (dtype != DT_F32 && dtype != DT_BF16 && dtype != DT_F16) return RN_ERR_DTYPE;
    if (!std::isfinite(eps) || eps < 0.f) return RN_ERR_EPS;
    // every problem on its own, then no problem writing what another touches
    for (int i = 0; i < count; ++i) {
        const int st = validate(problem_request(op, dtype, prs[i], eps));
        if (st != RN_OK) return st;
    }
    {
        // Outputs may overlap nothing: no other output, no input (inputs may
        // share memory among themselves, e.g. one gamma for all problems).
        // Sort the outputs; adjacent ones must be disjoint; then each input
        // can only meet the last output starting below its end.
        std::vector<std::pair<uintptr_t, uintptr_t>> outs, ins;   // [begin, end)
        outs.reserve(3 * (size_t)count);
        ins.reserve(3 * (size_t)count);
        for (int i = 0; i < count; ++i) {
            if (prs[i].rows == 0) continue;
            const void *pi[3], *po[3];
            int64_t ni[3], no[3];
            problem_ranges(op, dtype, prs[i], pi, ni, po, no);
            for (int a = 0; a < 3; ++a) {
                if (po[a] && no[a] > 0) outs.emplace_back(addr(po[a]), addr(po[a]) + no[a]);
                if (pi[a] && ni[a] > 0) ins.emplace_back(addr(pi[a]), addr(pi[a]) + ni[a]);
            }
        }
        std::sort(outs.begin(), outs.end());
        for (size_t i = 1; i < outs.size(); ++i)
            if (outs[i].first < outs[i - 1].second) return RN_ERR_ALIAS;
        for (const auto& in : ins) {
            auto it = std::lower_bound(outs.begin(), outs.end(),
                                       std::make_pair(in.second, (uintptr_t)0));
            if (it != outs.begin() && std::prev(it)->second > in.first) return RN_ERR_ALIAS;
        }
    }
    {
        // the parameter vectors must be in device memory, as for one call
        // (problems that take their own launch stage them by bulk copies):
        // each distinct vector is asked once, before anything is launched
        std::vector<const void*> ps;
        ps.reserve(2 * (size_t)count);
        for (int i = 0; i < count; ++i) {
            if (prs[i].rows == 0) continue;
            ps.push_back(prs[i].p0);
            if (op == OP_LN) ps.push_back(prs[i].p1);
        }
        std::sort(ps.begin(), ps.end());
        ps.erase(std::unique(ps.begin(), ps.end()), ps.end());
        for (const void* pp : ps)
            if (host_resident(pp)) return RN_ERR_HOSTMEM;
    }
    const cudaStream_t s = (cudaStream_t)stream;
    cudaError_t err = cudaSuccess;
    const int vec = 16 / dtype_size(dtype);
    BatchParams bp;
    bp.n = 0;
    bp.eps = eps;
    bp.start[0] = 0;
    int64_t widest = 0;   // vectors per row of the table's widest problem
    auto flush = [&]() -> int {
        if (bp.n == 0) return RN_OK;
        // the fewest vectors per lane (1, 2, 4, 8) that hold the widest row
        int slots = 1;
        while ((int64_t)slots * 32 < widest) slots *= 2;
        const BatchEntry* e = batched_entry(op, dtype, slots);
        if (!e) return RN_ERR_VARIANT;
        const int resident = batch_resident(e, &err);
        if (err != cudaSuccess) return fail_cuda(err);
        widest = 0;
        const int64_t rows = bp.start[bp.n];
        const int64_t rows_per_cta = e->threads / 32;
        const int64_t want = (rows + rows_per_cta - 1) / rows_per_cta;
        err = e->launch(bp, (int)(want < resident ? want : resident), s);
        bp.n = 0;
        return err == cudaSuccess ? RN_OK : fail_cuda(err);
    };
    for (int i = 0; i < count; ++i) {
        const rn_problem& pr = prs[i];
        if (pr.rows == 0) continue;
        const bool same_phase = ((addr(pr.x) ^ addr(pr.y)) & 15u) == 0;
        if (pr.d > kBatchMaxD || !same_phase) {
            // wide rows, or x and y in different 16-byte phases: own launch
            const int st = run(problem_request(op, dtype, pr, eps), RN_VARIANT_AUTO, stream);
            if (st != RN_OK) return st;
            continue;
        }
        BatchProblem& b = bp.pr[bp.n];
        b.x = pr.x;
        b.p0 = pr.p0;
        b.p1 = op == OP_LN ? pr.p1 : nullptr;
        b.y = pr.y;
        b.mean = op == OP_LN ? pr.mean_out : nullptr;
        b.rstd = op == OP_LN ? pr.rstd_out : nullptr;
        b.rows = pr.rows;
        b.d = (int)pr.d;
        b.al = pr.d % vec == 0 &&
               ((addr(pr.x) | addr(pr.y) | addr(pr.p0) | (op == OP_LN ? addr(pr.p1) : 0)) &
                15u) == 0;
        if (pr.d / vec > widest) widest = pr.d / vec;
        bp.start[bp.n + 1] = bp.start[bp.n] + pr.rows;
        ++bp.n;
        if (bp.n == kBatchMax) {
            const int st = flush();
            if (st != RN_OK) return st;
            bp.start[0] = 0;
        }
    }
    return flush();
}

// ---------------------------------------------------------------------------
// Backward.
// ---------------------------------------------------------------------------
struct BwdRequest {
    int op;
    const float* dy;
    const float* x;
    const float* p0;     // gamma or w
    const float* mean;   // LN
    const float* rstd;   // LN
    float* dx;
    float* dp0;          // dgamma or dw (may be NULL)
    float* dp1;          // dbeta (LN; may be NULL)
    int64_t rows;
    int64_t d;
    float eps;           // RMS
    void* ws;
    size_t ws_bytes;
    int dtype = DT_F32;  // storage of dy, x, dx and the parameters and their gradients
    bool rows_on_host = false;   // x or dy in host memory: no bulk-copy ring
};

struct BwdPlan {
    const BwdEntry* e;
    int stages;          // staged instances: ring depth (0 otherwise)
    int vec, slots, tpr, grid;
    int64_t width;       // floats per workspace row
    int64_t groups;      // workspace rows written (one per CTA)
};

// The current device's SM count and shared memory per SM, cached per thread.
bool device_shape(int* dev, int* sms, int* smem_sm, cudaError_t* err) {
    struct Cache {
        int dev = -1, sms = 0, smem = 0;
    };
    static thread_local Cache cache[8];
    if ((*err = cudaGetDevice(dev)) != cudaSuccess) return false;
    Cache& c = cache[*dev & 7];
    if (c.dev != *dev) {
        if ((*err = cudaDeviceGetAttribute(&c.sms, cudaDevAttrMultiProcessorCount, *dev)) !=
                cudaSuccess ||
            (*err = cudaDeviceGetAttribute(&c.smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                           *dev)) != cudaSuccess)
            return false;
        c.dev = *dev;
    }
    *sms = c.sms;
    *smem_sm = c.smem;
    return true;
}

// Resident CTAs per SM of a backward kernel with `smem` bytes of dynamic
// shared memory on device `dev` (raising its shared-memory limit first),
// cached per thread so that a call does not repeat the occupancy query.
int bwd_ctas_per_sm(const BwdEntry* e, int smem, int dev, cudaError_t* err) {
    struct Cache {
        const void* fn;
        unsigned long long ctx;
        int smem, n;
    };
    static thread_local Cache cache[32];
    static thread_local int cache_next = 0;
    (void)dev;   // the occupancy query runs on the current device
    const unsigned long long ctx = ctx_now();
    for (auto& c : cache)
        if (c.fn == e->fn && ctx != 0 && c.ctx == ctx && c.smem == smem && c.n > 0) return c.n;
    if (e->prepare && (*err = e->prepare()) != cudaSuccess) return -1;
    int per = 0;
    if ((*err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, e->fn, e->threads, smem)) !=
        cudaSuccess)
        return -1;
    cache[cache_next] = {e->fn, ctx_now(), smem, per};
    cache_next = (cache_next + 1) % 32;
    return per;
}

// Rows per CTA below which 64-128-thread backward rows stay on registers.
constexpr int kBwdStagedMinRows = 8;

int bwd_plan(const BwdRequest& q, bool pg, bool size_only, BwdPlan* bp, cudaError_t* err) {
    *err = cudaSuccess;
    const int vv = 16 / dtype_size(q.dtype);   // elements of one 128-bit vector
    const bool al = q.d % vv == 0 &&
                    ((addr(q.dy) | addr(q.x) | addr(q.p0) | addr(q.dx) | addr(q.ws)) & 15u) == 0;
    const int vec = al ? vv : 1;
    const int maxs = vec == 1 ? 8 : kBwdHeld / vec;
    const int64_t units = q.d / vec;
    int tpr = 0, slots = 0;
    for (int t = 32; t <= 1024; t *= 2)
        if (units <= (int64_t)t * maxs) {
            tpr = t;
            break;
        }
    if (!tpr) return RN_ERR_SIZE;
    const int need = (int)((units + tpr - 1) / tpr);
    slots = need <= 4 ? need : 8;
    // Rows of 256 or 512 threads on the vector layout run the staged form
    // when its ring fits: the bulk-copy engine keeps up to kBwdRingStages - 1
    // rows of x and dy in flight per CTA beyond what the registers hold. Rows
    // of 64 or 128 threads do so only with 16-bit storage and when every CTA
    // walks at least 8 rows: the staged form gives each such row its own
    // CTA, so it writes several times more partial rows for the column
    // reduction, which FP32 rows (already near the bandwidth on registers)
    // and short calls do not win back. Measured on GB300, cold L2: BF16
    // LayerNorm 16384 x 2048 64.9 -> 49.7 us, 32768 x 1024 57.6 -> 51.6 us;
    // FP32 32768 x 1024 72.2 -> 74.0 us and BF16 4096 x 768 16.8 -> 19.2 us
    // had it run staged.
    const BwdEntry* e = nullptr;
    int smem = 0, stages = 0;
    int dev = 0, sms = 0, smem_sm = 0;
    if (!device_shape(&dev, &sms, &smem_sm, err)) return RN_ERR_CUDA;
    if (vec > 1 && tpr >= 64 && (tpr >= 256 || q.dtype != DT_F32) &&
        (tpr <= 512 || (q.op == OP_RMS && q.dtype != DT_F32)) && !q.rows_on_host) {
        const BwdEntry* se = bwd_staged_entry(q.op, q.dtype, slots, tpr, pg);
        if (se) {
            // as many stages (up to kBwdRingStages) as the SM's shared memory
            // gives each of the CTAs its registers allow
            const int regs_ctas = bwd_ctas_per_sm(se, 0, dev, err);
            if (regs_ctas < 0) return RN_ERR_CUDA;
            const int64_t sb = bwd_stage_bytes(q.d, dtype_size(q.dtype));
            int64_t per_cta = smem_sm / (regs_ctas > 0 ? regs_ctas : 1) - 2048;
            if (per_cta > kBwdStagedSmemBudget) per_cta = kBwdStagedSmemBudget;
            int64_t n = (per_cta - se->smem_bytes) / sb;   // after a parameter plane
            if (n > kBwdRingStages) n = kBwdRingStages;
            bool take = n >= 2;
            if (take && tpr < 256) {
                const int per_s = bwd_ctas_per_sm(se, (int)(n * sb), dev, err);
                if (per_s < 0) return RN_ERR_CUDA;
                take = q.rows >= (int64_t)kBwdStagedMinRows * per_s * sms;
            }
            if (take) {
                e = se;
                stages = (int)n;
                smem = se->smem_bytes + (int)(n * sb);
            }
        }
    }
    if (!e) {
        e = bwd_entry(q.op, q.dtype, vec, slots, tpr, pg);
        if (!e) return RN_ERR_VARIANT;
        smem = e->smem_bytes;
    }
    // resident CTAs
    const int per = bwd_ctas_per_sm(e, smem, dev, err);
    if (per < 0) return RN_ERR_CUDA;
    int64_t grid = (int64_t)(per > 0 ? per : 1) * sms;
    const int64_t rows_ctas = (q.rows + e->rows_per_cta - 1) / e->rows_per_cta;
    if (rows_ctas < grid) grid = rows_ctas;
    if (pg) {
        // every CTA writes one partial row of the parameter sums: give each
        // row group several rows, but keep at least one CTA per SM busy
        const int64_t per_cta = (int64_t)e->rows_per_cta * kBwdMinRowsPerGroup;
        int64_t want = (q.rows + per_cta - 1) / per_cta;
        const int64_t floor_ = rows_ctas < sms ? rows_ctas : sms;
        if (want < floor_) want = floor_;
        if (want < grid) grid = want;
    }
    if (grid < 1) grid = 1;
    const int64_t width = q.op == OP_LN ? 2 * q.d : q.d;
    if (pg && !size_only) {
        const int64_t cap = (int64_t)(q.ws_bytes / ((size_t)width * 4));
        if (cap < 1) return RN_ERR_SIZE;   // workspace smaller than one CTA's partial row
        if (cap < grid) grid = cap;
    }
    bp->e = e;
    bp->stages = stages;
    bp->vec = vec;
    bp->slots = slots;
    bp->tpr = tpr;
    bp->grid = (int)grid;
    bp->width = width;
    bp->groups = grid;
    return RN_OK;
}

int bwd_validate(const BwdRequest& q, bool pg) {
    if (q.dtype != DT_F32 && q.dtype != DT_BF16 && q.dtype != DT_F16) return RN_ERR_DTYPE;
    if (q.rows < 0 || q.d <= 0) return RN_ERR_SIZE;
    if (q.rows > 0 && q.d > kMaxElems / q.rows) return RN_ERR_SIZE;
    if (q.op == OP_RMS && (!std::isfinite(q.eps) || q.eps < 0.f)) return RN_ERR_EPS;
    if (q.rows == 0) return RN_OK;
    if (!q.dy || !q.x || !q.p0 || !q.dx) return RN_ERR_NULL;
    if (q.op == OP_LN && (!q.mean || !q.rstd)) return RN_ERR_NULL;
    if (pg && !q.ws) return RN_ERR_NULL;
    const int es = dtype_size(q.dtype);
    const void* data[] = {q.dy, q.x, q.p0, q.dx, q.dp0, q.dp1};
    for (const void* p : data)
        if (misaligned(p, es)) return RN_ERR_ALIGN;
    if (misaligned(q.mean, 4) || misaligned(q.rstd, 4)) return RN_ERR_ALIGN;
    if (pg && (addr(q.ws) & 15u)) return RN_ERR_ALIGN;
    const int64_t nx = q.rows * q.d * es, np = q.d * es, ns = q.rows * 4;
    const int64_t nws = pg ? (int64_t)q.ws_bytes : 0;
    const void* outs[4] = {q.dx, q.dp0, q.dp1, pg ? q.ws : nullptr};
    const int64_t nouts[4] = {nx, np, np, nws};
    const void* ins[5] = {q.dy, q.x, q.p0, q.mean, q.rstd};
    const int64_t nins[5] = {nx, nx, np, ns, ns};
    for (int i = 0; i < 4; ++i) {
        for (int j = 0; j < 5; ++j)
            if (overlaps(outs[i], nouts[i], ins[j], nins[j])) return RN_ERR_ALIAS;
        for (int j = i + 1; j < 4; ++j)
            if (overlaps(outs[i], nouts[i], outs[j], nouts[j])) return RN_ERR_ALIAS;
    }
    return RN_OK;
}

int run_bwd(const BwdRequest& q, void* stream) {
    const bool pg = q.dp0 || q.dp1;
    int st = bwd_validate(q, pg);
    if (st != RN_OK) return st;
    if (q.rows == 0) {
        // an empty batch still defines the parameter gradients: zero
        const cudaStream_t s = (cudaStream_t)stream;
        cudaError_t err = cudaSuccess;
        const size_t np = (size_t)q.d * dtype_size(q.dtype);   // zero is all-zero bits in every type
        if (q.dp0) err = cudaMemsetAsync(q.dp0, 0, np, s);
        if (err == cudaSuccess && q.dp1) err = cudaMemsetAsync(q.dp1, 0, np, s);
        return err == cudaSuccess ? RN_OK : fail_cuda(err);
    }
    BwdPlan bp;
    cudaError_t err;
    // the bulk-copy engine fills the staged ring from device memory only
    BwdRequest qh = q;
    qh.rows_on_host = host_resident(q.x) || host_resident(q.dy);
    st = bwd_plan(qh, pg, false, &bp, &err);
    if (st == RN_ERR_CUDA) return fail_cuda(err);
    if (st != RN_OK) return st;
    BwdParams prm;
    prm.dy = q.dy;
    prm.x = q.x;
    prm.p0 = q.p0;
    prm.mean = q.mean;
    prm.rstd = q.rstd;
    prm.dx = q.dx;
    prm.ws = pg ? (float*)q.ws : nullptr;
    prm.rows = q.rows;
    prm.d = q.d;
    prm.ws_width = bp.width;
    prm.eps = q.eps;
    prm.err = nullptr;
    prm.stages = bp.stages;
    if (bp.e->staged && (err = device_error_address(&prm.err)) != cudaSuccess)
        return fail_cuda(err);
    const cudaStream_t s = (cudaStream_t)stream;
    err = bp.e->launch(prm, bp.grid, s);
    if (err != cudaSuccess) return fail_cuda(err);
    if (pg) {
        // LN workspace rows: [0, d) dbeta partials, [d, 2d) dgamma partials
        void* out0 = q.op == OP_LN ? q.dp1 : q.dp0;
        void* out1 = q.op == OP_LN ? q.dp0 : nullptr;
        err = column_reduce(q.dtype, (const float*)q.ws, bp.groups, bp.width, q.d, out0, out1, s);
        if (err != cudaSuccess) return fail_cuda(err);
    }
    return RN_OK;
}

int bwd_workspace(int op, int64_t rows, int64_t d, size_t* bytes) {
    if (!bytes) return RN_ERR_NULL;
    if (rows < 0 || d <= 0) return RN_ERR_SIZE;
    *bytes = 0;
    if (rows == 0) return RN_OK;
    // every storage type, vector or scalar layout, may run a different grid:
    // size for the largest (one workspace row of FP32 partials per CTA)
    int64_t groups = 0, width = 0;
    int first = RN_ERR_SIZE;
    for (int dt : {DT_F32, DT_BF16, DT_F16}) {
        for (uintptr_t xa : {(uintptr_t)0, (uintptr_t)4}) {   // 4: an unaligned address
            BwdRequest q{};
            q.op = op;
            q.rows = rows;
            q.d = d;
            q.dtype = dt;
            q.x = (const float*)xa;
            BwdPlan bp;
            cudaError_t err;
            const int st = bwd_plan(q, true, true, &bp, &err);
            if (st == RN_ERR_CUDA) return fail_cuda(err);
            if (dt == DT_F32 && xa == 0) first = st;
            if (st != RN_OK) continue;
            if (bp.groups > groups) groups = bp.groups;
            width = bp.width;
        }
    }
    if (first != RN_OK) return first;   // the FP32 vector layout decides what is valid
    *bytes = (size_t)(groups * width * 4);
    return RN_OK;
}

}  // namespace

namespace rn {
int record_cuda_error(cudaError_t err) { return fail_cuda(err); }

int ln_bwd_check_args(const float* dy, const float* x, const float* gamma, const float* mean,
                      const float* rstd, float* dx, float* dgamma, float* dbeta, int64_t rows,
                      int64_t d) {
    BwdRequest q{};
    q.op = OP_LN;
    q.dy = dy;
    q.x = x;
    q.p0 = gamma;
    q.mean = mean;
    q.rstd = rstd;
    q.dx = dx;
    q.dp0 = dgamma;
    q.dp1 = dbeta;
    q.rows = rows;
    q.d = d;
    return bwd_validate(q, false);   // every check except those of the workspace
}

namespace ctxq {
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
struct CtxFns {
    CtxGetCurrentFn current = nullptr;
    CtxGetIdFn id = nullptr;
    cudaError_t err = cudaSuccess;
};
// The two driver calls, found once through the runtime (no link to the
// driver library is needed).
const CtxFns& ctx_fns() {
    static const CtxFns fns = [] {
        CtxFns f;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        f.err = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                                 &q);
        if (f.err != cudaSuccess) return f;
        if (q != cudaDriverEntryPointSuccess || !p) {
            f.err = cudaErrorNotSupported;
            return f;
        }
        f.current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        f.err = cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q);
        if (f.err != cudaSuccess) return f;
        if (q != cudaDriverEntryPointSuccess || !p) {
            f.err = cudaErrorNotSupported;
            return f;
        }
        f.id = reinterpret_cast<CtxGetIdFn>(p);
        return f;
    }();
    return fns;
}
}  // namespace ctxq

cudaError_t current_context_id(unsigned long long* id) {
    const ctxq::CtxFns& f = ctxq::ctx_fns();
    if (!f.current || !f.id) return f.err != cudaSuccess ? f.err : cudaErrorNotSupported;
    CUcontext c = nullptr;
    if (f.current(&c) != CUDA_SUCCESS) return cudaErrorUnknown;
    *id = 0;
    if (c && f.id(c, id) != CUDA_SUCCESS) return cudaErrorUnknown;
    return cudaSuccess;
}
}  // namespace rn

extern "C" {

int ln_bwd_workspace_size(int64_t rows, int64_t d, size_t* bytes) {
    return bwd_workspace(OP_LN, rows, d, bytes);
}

int rms_bwd_workspace_size(int64_t rows, int64_t d, size_t* bytes) {
    return bwd_workspace(OP_RMS, rows, d, bytes);
}

int ln_bwd(const float* dy, const float* x, const float* gamma, const float* mean,
           const float* rstd, float* dx, float* dgamma, float* dbeta, int64_t rows, int64_t d,
           void* workspace, size_t workspace_bytes, void* stream) {
    BwdRequest q{OP_LN, dy, x, gamma, mean, rstd, dx, dgamma, dbeta, rows, d, 0.f,
                 workspace, workspace_bytes};
    return run_bwd(q, stream);
}

int rms_bwd(const float* dy, const float* x, const float* w, float* dx, float* dw, int64_t rows,
            int64_t d, float eps, void* workspace, size_t workspace_bytes, void* stream) {
    BwdRequest q{OP_RMS, dy, x, w, nullptr, nullptr, dx, dw, nullptr, rows, d, eps,
                 workspace, workspace_bytes};
    return run_bwd(q, stream);
}

int ln_bwd_typed(int dtype, const void* dy, const void* x, const void* gamma, const float* mean,
                 const float* rstd, void* dx, void* dgamma, void* dbeta, int64_t rows, int64_t d,
                 void* workspace, size_t workspace_bytes, void* stream) {
    BwdRequest q{OP_LN, (const float*)dy, (const float*)x, (const float*)gamma, mean, rstd,
                 (float*)dx, (float*)dgamma, (float*)dbeta, rows, d, 0.f, workspace,
                 workspace_bytes};
    q.dtype = dtype;
    return run_bwd(q, stream);
}

int rms_bwd_typed(int dtype, const void* dy, const void* x, const void* w, void* dx, void* dw,
                  int64_t rows, int64_t d, float eps, void* workspace, size_t workspace_bytes,
                  void* stream) {
    BwdRequest q{OP_RMS, (const float*)dy, (const float*)x, (const float*)w, nullptr, nullptr,
                 (float*)dx, (float*)dw, nullptr, rows, d, eps, workspace, workspace_bytes};
    q.dtype = dtype;
    return run_bwd(q, stream);
}

int ln_fwd(const float* x, const float* gamma, const float* beta, float* y, float* mean_out,
           float* rstd_out, int64_t rows, int64_t d, float eps, void* stream) {
    return run(ln_request(x, nullptr, gamma, beta, nullptr, y, mean_out, rstd_out, rows, d, eps,
                          false),
               RN_VARIANT_AUTO, stream);
}

int rms_fwd(const float* x, const float* w, float* y, int64_t rows, int64_t d, float eps,
            void* stream) {
    return run(rms_request(x, nullptr, w, nullptr, y, rows, d, eps, false), RN_VARIANT_AUTO,
               stream);
}

int ln_fwd_variant(int variant, const float* x, const float* gamma, const float* beta, float* y,
                   float* mean_out, float* rstd_out, int64_t rows, int64_t d, float eps,
                   void* stream) {
    return run(ln_request(x, nullptr, gamma, beta, nullptr, y, mean_out, rstd_out, rows, d, eps,
                          false),
               variant, stream);
}

int rms_fwd_variant(int variant, const float* x, const float* w, float* y, int64_t rows,
                    int64_t d, float eps, void* stream) {
    return run(rms_request(x, nullptr, w, nullptr, y, rows, d, eps, false), variant, stream);
}

int ln_fwd_residual(const float* x, const float* res, const float* gamma, const float* beta,
                    float* h_out, float* y, float* mean_out, float* rstd_out, int64_t rows,
                    int64_t d, float eps, void* stream) {
    return run(ln_request(x, res, gamma, beta, h_out, y, mean_out, rstd_out, rows, d, eps, true),
               RN_VARIANT_AUTO, stream);
}

int rms_fwd_residual(const float* x, const float* res, const float* w, float* h_out, float* y,
                     int64_t rows, int64_t d, float eps, void* stream) {
    return run(rms_request(x, res, w, h_out, y, rows, d, eps, true), RN_VARIANT_AUTO, stream);
}

int ln_fwd_residual_variant(int variant, const float* x, const float* res, const float* gamma,
                            const float* beta, float* h_out, float* y, float* mean_out,
                            float* rstd_out, int64_t rows, int64_t d, float eps, void* stream) {
    return run(ln_request(x, res, gamma, beta, h_out, y, mean_out, rstd_out, rows, d, eps, true),
               variant, stream);
}

int rms_fwd_residual_variant(int variant, const float* x, const float* res, const float* w,
                             float* h_out, float* y, int64_t rows, int64_t d, float eps,
                             void* stream) {
    return run(rms_request(x, res, w, h_out, y, rows, d, eps, true), variant, stream);
}

int ln_fwd_typed(int dtype, int variant, const void* x, const void* gamma, const void* beta,
                 void* y, float* mean_out, float* rstd_out, int64_t rows, int64_t d, float eps,
                 void* stream) {
    return run(ln_request((const float*)x, nullptr, (const float*)gamma, (const float*)beta,
                          nullptr, (float*)y, mean_out, rstd_out, rows, d, eps, false, dtype),
               variant, stream);
}

int rms_fwd_typed(int dtype, int variant, const void* x, const void* w, void* y, int64_t rows,
                  int64_t d, float eps, void* stream) {
    return run(rms_request((const float*)x, nullptr, (const float*)w, nullptr, (float*)y, rows, d,
                           eps, false, dtype),
               variant, stream);
}

int ln_fwd_strided(int dtype, int variant, const void* x, int64_t ldx, const void* gamma,
                   const void* beta, void* y, int64_t ldy, float* mean_out, float* rstd_out,
                   int64_t rows, int64_t d, float eps, void* stream) {
    if (ldx < d || ldy < d || ldx <= 0) return RN_ERR_SIZE;
    Request q = ln_request((const float*)x, nullptr, (const float*)gamma, (const float*)beta,
                           nullptr, (float*)y, mean_out, rstd_out, rows, d, eps, false, dtype);
    q.ldx = ldx;
    q.ldy = ldy;
    return run(q, variant, stream);
}

int rms_fwd_strided(int dtype, int variant, const void* x, int64_t ldx, const void* w, void* y,
                    int64_t ldy, int64_t rows, int64_t d, float eps, void* stream) {
    if (ldx < d || ldy < d || ldx <= 0) return RN_ERR_SIZE;
    Request q = rms_request((const float*)x, nullptr, (const float*)w, nullptr, (float*)y, rows, d,
                           eps, false, dtype);
    q.ldx = ldx;
    q.ldy = ldy;
    return run(q, variant, stream);
}

int ln_fwd_batched(int dtype, const rn_problem* problems, int count, float eps, void* stream) {
    return run_batched(OP_LN, dtype, problems, count, eps, stream);
}

int rms_fwd_batched(int dtype, const rn_problem* problems, int count, float eps, void* stream) {
    return run_batched(OP_RMS, dtype, problems, count, eps, stream);
}

static int plan_any(int dtype, int op, int variant, int64_t d, const void* x, const void* res,
                    const void* h, const void* y, const void* p0, const void* p1, rn_plan* plan,
                    int64_t ldx = 0, int64_t ldy = 0) {
    if (!plan) return RN_ERR_NULL;
    if (op != RN_OP_LN && op != RN_OP_RMS) return RN_ERR_VARIANT;
    if (variant < 0 || variant >= RN_VARIANT_COUNT) return RN_ERR_VARIANT;
    if (dtype != RN_DTYPE_F32 && dtype != RN_DTYPE_BF16 && dtype != RN_DTYPE_F16)
        return RN_ERR_DTYPE;
    if (res && dtype != RN_DTYPE_F32) return RN_ERR_DTYPE;
    Request q{op == RN_OP_LN ? OP_LN : OP_RMS,
              dtype,
              res != nullptr,
              (const float*)x,
              (const float*)res,
              (const float*)p0,
              (const float*)p1,
              (float*)y,
              (float*)h,
              nullptr,
              nullptr,
              1,
              d,
              0.f};
    if (ldx != 0 || ldy != 0) {
        if (ldx < d || ldy < d) return RN_ERR_SIZE;
        q.ldx = ldx;
        q.ldy = ldy;
    }
    return plan_impl(q, variant, plan);
}

int rn_plan_for_residual(int op, int variant, int64_t d, const void* x, const void* res,
                         const void* h, const void* y, const void* p0, const void* p1,
                         rn_plan* plan) {
    return plan_any(RN_DTYPE_F32, op, variant, d, x, res, h, y, p0, p1, plan);
}

int rn_plan_for_typed(int dtype, int op, int variant, int64_t d, const void* x, const void* y,
                      const void* p0, const void* p1, rn_plan* plan) {
    return plan_any(dtype, op, variant, d, x, nullptr, nullptr, y, p0, p1, plan);
}

int rn_plan_for_strided(int dtype, int op, int variant, int64_t d, const void* x, int64_t ldx,
                        const void* y, int64_t ldy, const void* p0, const void* p1,
                        rn_plan* plan) {
    if (ldx <= 0 || ldy <= 0) return RN_ERR_SIZE;
    return plan_any(dtype, op, variant, d, x, nullptr, nullptr, y, p0, p1, plan, ldx, ldy);
}

int rn_plan_for(int op, int variant, int64_t d, const void* x, const void* y, const void* p0,
                const void* p1, rn_plan* plan) {
    return rn_plan_for_residual(op, variant, d, x, nullptr, nullptr, y, p0, p1, plan);
}

const char* rn_status_str(int status) {
    switch (status) {
        case RN_OK: return "ok";
        case RN_ERR_NULL: return "a required pointer is NULL";
        case RN_ERR_SIZE:
            return "invalid size (rows < 0, d <= 0, rows*d too large or a row stride below d)";
        case RN_ERR_EPS: return "eps must be finite and >= 0";
        case RN_ERR_ALIAS: return "an output overlaps an input or another output";
        case RN_ERR_CUDA: return "CUDA runtime error (see rn_last_cuda_error)";
        case RN_ERR_ALIGN: return "a pointer is not 4-byte aligned";
        case RN_ERR_VARIANT: return "the requested kernel variant cannot run this request";
        case RN_ERR_DTYPE: return "unsupported storage type for this entry point";
        case RN_ERR_HOSTMEM:
            return "the parameter vectors (gamma, beta, w) of a forward call must be in device "
                   "memory";
        case RN_ERR_SCRATCH:
            return "the request needs more than the static scratch holds (ln_bwd_noalloc: "
                   "d <= 4096)";
        default: return "unknown status";
    }
}

int rn_last_cuda_error(void) { return g_last_cuda_error; }

int rn_device_error(unsigned int* flags, int clear) {
    if (!flags) return RN_ERR_NULL;
    const cudaError_t err = device_error_word(flags, clear != 0);
    return err == cudaSuccess ? RN_OK : fail_cuda(err);
}

int rn_selftest_bounded_wait(unsigned int timeout_us, void* stream) {
    if (timeout_us < 1 || timeout_us > 1000000) return RN_ERR_SIZE;
    const cudaError_t e = bounded_wait_selftest(1000ull * timeout_us, (cudaStream_t)stream);
    return e == cudaSuccess ? RN_OK : fail_cuda(e);
}

int rn_pageable_host_access(int* pageable) {
    if (!pageable) return RN_ERR_NULL;
    int dev = 0, v = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess)
        err = cudaDeviceGetAttribute(&v, cudaDevAttrPageableMemoryAccess, dev);
    if (err != cudaSuccess) return fail_cuda(err);
    *pageable = v ? 1 : 0;
    return RN_OK;
}

int rn_launch_empty(int64_t grid, int threads, void* stream) {
    if (grid < 1 || grid >= ((int64_t)1 << 31) || threads < 1 || threads > 1024)
        return RN_ERR_SIZE;
    empty_kernel<<<(unsigned)grid, threads, 0, (cudaStream_t)stream>>>();
    const cudaError_t err = cudaGetLastError();
    return err == cudaSuccess ? RN_OK : fail_cuda(err);
}

const char* rn_variant_name(int variant) {
    switch (variant) {
        case RN_VARIANT_AUTO: return "auto";
        case RN_VARIANT_WARP: return "warp";
        case RN_VARIANT_BLOCK: return "block";
        case RN_VARIANT_STAGED: return "staged";
        case RN_VARIANT_STREAM: return "stream";
        case RN_VARIANT_CLUSTER: return "cluster";
        default: return "unknown";
    }
}

}  // extern "C"
