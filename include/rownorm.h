/*
 * rownorm.h -- C ABI of the GB300 (sm_103a) row-wise normalization library.
 *
 * Two operations over the rows of a row-major matrix x[rows][d] (FP32, or
 * BF16 / FP16 storage with FP32 arithmetic in the *_typed, *_strided and
 * *_batched entry points), with their backward passes (FP32):
 *
 *   LayerNorm:  mu_i      = (1/d) sum_j x_ij
 *               sigma_i^2 = (1/d) sum_j (x_ij - mu_i)^2
 *     (the statistics equation of "Rewriting the layer norm and matmul
 *     kernels", section "A reduction has to meet somewhere"), then
 *               rstd_i = (sigma_i^2 + eps)^(-1/2)
 *               y_ij   = (x_ij - mu_i) * rstd_i * gamma_j + beta_j
 *     (the standard affine output; eps inside the root as in the RMSNorm
 *     equation below).
 *
 *   RMSNorm:    y_rc = x_rc * w_c * ((1/D) sum_j x_rj^2 + eps)^(-1/2)
 *     ("RMSNorm on an RTX 5070: why more reduction threads did not win every
 *     shape", section "The operator and the change", displayed equation).
 *
 * Conventions shared by every entry point:
 *
 *   Memory      Every array pointer is an address the current GPU can
 *               dereference: device memory (cudaMalloc), or host memory the
 *               GPU can address -- pinned host memory (cudaHostAlloc /
 *               cudaHostRegister; with unified addressing its host pointer
 *               is valid on the device) and, on systems whose GPU reads host
 *               page tables (GB300 over NVLink-C2C), ordinary pageable host
 *               memory. Host-resident x is then read and host-resident y
 *               written by the kernel itself over the host link, with no
 *               staging copies; the forward entry points ask the runtime
 *               where x and y live (cudaPointerGetAttributes, no
 *               synchronization) and walk host-resident rows on a smaller,
 *               persistent grid, so that reads and writes share the link.
 *               The exception: the parameter vectors of the forward calls,
 *               single and batched (gamma, beta, w), which the kernels copy
 *               into shared memory with the bulk-copy engine, must be
 *               device memory, else RN_ERR_HOSTMEM before anything is
 *               launched (the backward takes them anywhere, as above).
 *               The caller owns every buffer (the
 *               backward's workspace included); no entry point allocates
 *               or synchronizes, except the diagnostics that say so. Rows
 *               are contiguous with row stride d (in elements), except in
 *               the *_strided entry points. Every pointer must be aligned
 *               to its element (4 bytes for FP32, 2 for 16-bit storage); no
 *               other alignment is required (16-byte aligned rows take the
 *               vector path, others a scalar head/tail or the scalar path).
 *   Stream      `stream` is a cudaStream_t passed as void*; NULL means the
 *               legacy default stream. Work is enqueued asynchronously; the
 *               results are valid once the stream has reached that point.
 *               The forward kernels are launched with programmatic stream
 *               serialization (programmatic dependent launch): the GPU may
 *               start one while the kernel ahead of it on the stream is
 *               still running, and it reads and writes nothing before that
 *               kernel has completed, so stream order holds as for any
 *               launch. Work the caller enqueues afterwards sees the
 *               results as usual; only a kernel of the caller's that is
 *               itself launched with programmatic serialization right after
 *               one of these calls must wait (cudaGridDependencySynchronize)
 *               before it reads the outputs, as for any programmatic launch.
 *   Sizes       rows == 0 is a no-op returning RN_OK (pointers may then be
 *               NULL). rows < 0, d <= 0, or rows*d beyond 2^61 elements
 *               returns RN_ERR_SIZE.
 *   eps         Must be finite and >= 0, else RN_ERR_EPS. eps == 0 is
 *               allowed (an all-zero row then gives Inf/NaN, as it should).
 *   Aliasing    No output may overlap any input or another output
 *               (RN_ERR_ALIAS): a row's outputs are written while other
 *               rows' inputs are still being read, and gamma/beta (w) are
 *               copied once per CTA. In-place normalization is not
 *               supported. The inputs may be the outputs of the call just
 *               before on the same stream: every load is coherent and
 *               comes after the wait for that call.
 *   Errors      Validation happens on the host before anything is enqueued;
 *               on any non-RN_OK status nothing was launched, except
 *               RN_ERR_CUDA, which reports a launch error from the CUDA
 *               runtime (the cudaError_t is kept per thread and returned by
 *               rn_last_cuda_error()).
 *   Threads     Every entry point may be called from several host threads.
 */
#ifndef ROWNORM_H
#define ROWNORM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rn_status {
    RN_OK = 0,
    RN_ERR_NULL = 1,    /* a required pointer is NULL while rows > 0          */
    RN_ERR_SIZE = 2,    /* rows < 0, d <= 0, rows * d too large, stride < d    */
    RN_ERR_EPS = 3,     /* eps < 0, NaN or infinite                            */
    RN_ERR_ALIAS = 4,   /* an output overlaps an input or another output      */
    RN_ERR_CUDA = 5,    /* the CUDA runtime reported an error on launch       */
    RN_ERR_ALIGN = 6,   /* a pointer is not 4-byte aligned                     */
    RN_ERR_VARIANT = 7, /* a forced variant cannot run this shape / alignment  */
    RN_ERR_DTYPE = 8,   /* unknown storage type, or one the entry point lacks  */
    RN_ERR_SCRATCH = 9, /* the request needs more than a static scratch holds  */
    RN_ERR_HOSTMEM = 10 /* a forward call's parameter vectors in host memory   */
} rn_status;

/* Storage types of x, y and the parameter vectors (statistics are FP32). */
enum {
    RN_DTYPE_F32 = 0,
    RN_DTYPE_BF16 = 1,   /* bfloat16: 8 exponent bits, 7 stored mantissa bits */
    RN_DTYPE_F16 = 2     /* IEEE binary16                                      */
};

/*
 * LayerNorm forward.
 *   x        [rows][d]  input, read once from HBM
 *   gamma    [d]        scale
 *   beta     [d]        shift
 *   y        [rows][d]  output
 *   mean_out [rows]     per-row mean mu_i (FP32); may be NULL (not written)
 *   rstd_out [rows]     per-row (sigma_i^2 + eps)^(-1/2), the factor that
 *                       scaled the row (FP32); may be NULL (not written)
 * Statistics are accumulated in FP32 from the values held on chip: the row
 * mean first, then the centred sum of squares about it (no E[x^2] - mu^2
 * cancellation). One kernel launch per call.
 */
int ln_fwd(const float *x, const float *gamma, const float *beta,
           float *y, float *mean_out, float *rstd_out,
           int64_t rows, int64_t d, float eps, void *stream);

/*
 * RMSNorm forward.
 *   x [rows][d] input, w [d] weight, y [rows][d] output.
 * One kernel launch per call.
 */
int rms_fwd(const float *x, const float *w, float *y,
            int64_t rows, int64_t d, float eps, void *stream);

/*
 * Residual add fused with the normalization: h = x + res (an FP32 add, the
 * updated residual stream of a pre-norm transformer block), then LayerNorm
 * or RMSNorm of h, in one pass over the row.
 *   x, res   [rows][d]  inputs (res must not alias any output)
 *   h_out    [rows][d]  h = x + res; may be NULL (not written)
 *   y, mean_out, rstd_out, gamma, beta, w: as in ln_fwd / rms_fwd, of h.
 * The pages name this fusion as absent from their kernels ("RMSNorm on an
 * RTX 5070 ...", section "The operator and the change"). One kernel launch;
 * AUTO uses the register-held kernels on rows of up to 512 threads (d up to
 * 16384 floats with 16-byte aligned rows, 4096 with scalar accesses) and
 * the streaming kernel beyond. A forced RN_VARIANT_BLOCK on a wider row
 * (1024 threads), and the staged and cluster variants, have no residual
 * form: RN_ERR_VARIANT.
 */
int ln_fwd_residual(const float *x, const float *res, const float *gamma, const float *beta,
                    float *h_out, float *y, float *mean_out, float *rstd_out,
                    int64_t rows, int64_t d, float eps, void *stream);

int rms_fwd_residual(const float *x, const float *res, const float *w, float *h_out,
                     float *y, int64_t rows, int64_t d, float eps, void *stream);

/*
 * LayerNorm / RMSNorm with 16-bit (or FP32) storage and FP32 arithmetic.
 *   dtype     RN_DTYPE_F32, RN_DTYPE_BF16 or RN_DTYPE_F16: the element type of
 *             x, y, gamma, beta and w (all the same type)
 *   variant   RN_VARIANT_AUTO or a forced variant (see below)
 *   mean_out, rstd_out: FP32 [rows], may be NULL
 * Values are widened to FP32 on load, every statistic is accumulated in FP32
 * exactly as in ln_fwd / rms_fwd, and y is rounded to the storage type once,
 * to nearest even. Pointers must be aligned to the element size (2 bytes for
 * 16-bit types). With 16-bit storage, AUTO uses the warp / CTA-per-row
 * kernels up to d = 32768 and the streaming kernel beyond; the staged and
 * cluster variants are FP32 only (RN_ERR_VARIANT). RN_DTYPE_F32 here is the
 * same computation as ln_fwd / rms_fwd.
 */
int ln_fwd_typed(int dtype, int variant, const void *x, const void *gamma, const void *beta,
                 void *y, float *mean_out, float *rstd_out, int64_t rows, int64_t d, float eps,
                 void *stream);

int rms_fwd_typed(int dtype, int variant, const void *x, const void *w, void *y, int64_t rows,
                  int64_t d, float eps, void *stream);

/*
 * Strided rows: as ln_fwd_typed / rms_fwd_typed, with row i of x at
 * x + i*ldx and row i of y at y + i*ldy (strides in elements, each >= d;
 * the d elements of a row stay contiguous). This normalises a column block
 * of a wider matrix (e.g. one head's slice of a fused projection output) or
 * rows with a padded pitch, in place of a copy to a contiguous buffer. The
 * elements between rows are neither read nor written. Strides below d
 * return RN_ERR_SIZE. Aliasing is checked on spans (first to last element),
 * so an output interleaved with an input in the same rows is rejected
 * (RN_ERR_ALIAS). The 128-bit path needs x and y in the same 16-byte phase
 * on every row: equal base phases and ldx - ldy a multiple of the vector
 * (4 FP32 or 8 16-bit elements); otherwise every access is scalar. The
 * pages test contiguous rows only ("RMSNorm on an RTX 5070 ...", section
 * "The operator and the change", names arbitrary strides as untested).
 */
int ln_fwd_strided(int dtype, int variant, const void *x, int64_t ldx, const void *gamma,
                   const void *beta, void *y, int64_t ldy, float *mean_out, float *rstd_out,
                   int64_t rows, int64_t d, float eps, void *stream);

int rms_fwd_strided(int dtype, int variant, const void *x, int64_t ldx, const void *w, void *y,
                    int64_t ldy, int64_t rows, int64_t d, float eps, void *stream);

/*
 * Many small problems in one launch. A tensor of a few hundred KB is
 * normalised in a few microseconds of DRAM time but pays a whole kernel
 * launch; a step that normalises many of them is launch-bound (the RMSNorm
 * page times its kernels inside CUDA graphs of 64 launches for this reason:
 * "RMSNorm on an RTX 5070 ...", section "What the timer included"). These
 * entry points take `count` independent problems, each as ln_fwd_typed /
 * rms_fwd_typed would (contiguous rows, one storage type `dtype` and one eps
 * for all), and run every problem of width d <= 1024 whose x and y share a
 * 16-byte phase in one launch per 128 such problems; the others get launches
 * of their own (the same kernels ln_fwd_typed would pick), on the same
 * stream. `problems` is host memory, read during the call only. Each
 * problem is validated as its single call would be, and no problem may
 * write what another reads or writes (RN_ERR_ALIAS); nothing runs unless all
 * pass. Results are those of the single calls, bit for bit, for problems of
 * width <= 1024.
 */
typedef struct rn_problem {
    const void *x;      /* [rows][d] */
    const void *p0;     /* gamma (LN) or w (RMS), [d] */
    const void *p1;     /* beta (LN), [d]; ignored by RMS */
    void *y;            /* [rows][d] */
    float *mean_out;    /* LN: [rows] FP32, may be NULL; ignored by RMS */
    float *rstd_out;    /* LN: [rows] FP32, may be NULL; ignored by RMS */
    int64_t rows;
    int64_t d;
} rn_problem;

int ln_fwd_batched(int dtype, const rn_problem *problems, int count, float eps, void *stream);

int rms_fwd_batched(int dtype, const rn_problem *problems, int count, float eps, void *stream);

/*
 * Backward (FP32). The pages list backward passes as untested; these are the
 * derivatives of the forward definitions above.
 *
 * LayerNorm, from the forward's saved mean and rstd:
 *   xhat = (x - mean) * rstd, g = dy * gamma,
 *   dx     = rstd * (g - mean_j g - xhat * mean_j(g * xhat))   [rows][d]
 *   dgamma = sum_i dy * xhat,  dbeta = sum_i dy                 [d]
 * RMSNorm, with r = (mean_j x^2 + eps)^-1/2 recomputed from x:
 *   dx = r * (g - x * r^2 * mean_j(g * x)), g = dy * w;  dw = sum_i dy * x * r.
 *
 * dgamma / dbeta / dw may be NULL (not computed; with all NULL no workspace
 * is needed). Parameter gradients are summed over rows deterministically: each
 * row group accumulates its rows' column sums in registers, each CTA adds its
 * groups in order and writes one row of partial sums to `workspace` (device
 * memory, 16-byte aligned, caller-owned, contents on entry ignored), and a
 * second kernel adds those rows in a fixed order with Kahan compensation.
 * *_bwd_workspace_size gives the bytes for the full grid on the current
 * device; a smaller workspace (at least one partial row: 2*d*4 bytes for LN,
 * d*4 for RMS) runs fewer CTAs, and one below that returns RN_ERR_SIZE.
 * Results are bitwise repeatable for a given device and workspace size.
 * Calls on one stream may share a workspace; calls that may run at the same
 * time on the GPU need workspaces of their own. Rows wide enough for 256 or
 * 512 threads (and 16-bit rows of 64-128 threads in long calls) are brought
 * into shared memory by bulk copies; their waits are bounded as the staged
 * forward's are (RN_DEVERR_STAGED_TIMEOUT in rn_device_error). The calls
 * launch only on `stream`, so after one ordinary call of a configuration
 * they can be captured into a CUDA graph. Widths up to 16384
 * (aligned arrays, d % 4 == 0) or 8192 (otherwise); wider rows return
 * RN_ERR_SIZE. Two kernel launches when parameter gradients are wanted, one
 * otherwise; rows == 0 zeroes the requested parameter gradients.
 */
int ln_bwd_workspace_size(int64_t rows, int64_t d, size_t *bytes);

int ln_bwd(const float *dy, const float *x, const float *gamma, const float *mean,
           const float *rstd, float *dx, float *dgamma, float *dbeta, int64_t rows, int64_t d,
           void *workspace, size_t workspace_bytes, void *stream);

int rms_bwd_workspace_size(int64_t rows, int64_t d, size_t *bytes);

int rms_bwd(const float *dy, const float *x, const float *w, float *dx, float *dw, int64_t rows,
            int64_t d, float eps, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward with 16-bit (or FP32) storage: as ln_bwd / rms_bwd, with dy, x,
 * dx, gamma (w) and dgamma / dbeta (dw) all of type `dtype` (RN_DTYPE_F32,
 * RN_DTYPE_BF16 or RN_DTYPE_F16; pointers aligned to the element size);
 * mean and rstd stay FP32. Values are widened to FP32 on load, all
 * arithmetic and the workspace partials are FP32, and dx and the parameter
 * gradients are rounded once to the storage type, to nearest even. The
 * *_bwd_workspace_size figure covers every storage type. Widths up to 16384
 * (all of dy, x, dx, gamma and the workspace 16-byte aligned and d a multiple
 * of the 16-byte vector: 4 FP32 or 8 16-bit elements) or 8192 (otherwise).
 * Unknown dtype: RN_ERR_DTYPE.
 */
int ln_bwd_typed(int dtype, const void *dy, const void *x, const void *gamma, const float *mean,
                 const float *rstd, void *dx, void *dgamma, void *dbeta, int64_t rows, int64_t d,
                 void *workspace, size_t workspace_bytes, void *stream);

int rms_bwd_typed(int dtype, const void *dy, const void *x, const void *w, void *dx, void *dw,
                  int64_t rows, int64_t d, float eps, void *workspace, size_t workspace_bytes,
                  void *stream);

/*
 * LayerNorm backward without any allocation. The paper has no counterpart to
 * this entry point; it serves callers that cannot allocate device memory
 * where they run the backward: a process whose caching allocator already
 * holds nearly all of HBM, a loop that cannot afford cudaFree's device-wide
 * synchronisation, or C code with no allocator. Arguments, layouts, results
 * and errors are those of ln_bwd, without the workspace: the parameter-
 * gradient partials go to one static device array of RN_NOALLOC_SCRATCH_BYTES
 * (8 MiB), which every GPU that loads the library holds until exit. At
 * d <= 4096 the array holds at least 256 partial rows, so the grid matches
 * ln_bwd's with a workspace of that size, and the results are the same bits.
 * The first call on a device that needs the array looks it up
 * (cudaGetSymbolAddress, with that device current) and keeps the address for
 * the device's CUDA context; make that call before any stream capture on the
 * device. A new context for the device (after cudaDeviceReset) is looked up
 * again on its first call. Nothing here calls cudaMalloc, cudaFree or
 * another allocating routine. All calls share the array and nothing in it
 * has to start at zero; calls that can overlap on the GPU (two streams, two
 * threads) race on it. The arguments are checked as ln_bwd checks them
 * first; then a call that needs the partials (rows > 0 and dgamma or dbeta
 * not NULL) with d > RN_NOALLOC_MAX_D (4096) returns RN_ERR_SCRATCH and
 * launches nothing. Without parameter gradients no partials are needed and
 * every width ln_bwd takes runs.
 */
#define RN_NOALLOC_SCRATCH_BYTES (8u << 20)
#define RN_NOALLOC_MAX_D 4096

int ln_bwd_noalloc(const float *dy, const float *x, const float *gamma, const float *mean,
                   const float *rstd, float *dx, float *dgamma, float *dbeta, int64_t rows,
                   int64_t d, void *stream);

/* Static, NUL-terminated description of a status code (never NULL). */
const char *rn_status_str(int status);

/* The cudaError_t behind the last RN_ERR_CUDA returned on this thread
 * (0 if none). */
int rn_last_cuda_error(void);

/* ---------------------------------------------------------------------------
 * Kernel variants. ln_fwd / rms_fwd pick one from d and pointer alignment;
 * the *_variant entry points force one (testing and tuning) and return
 * RN_ERR_VARIANT if it cannot run the request.
 *
 *   RN_VARIANT_WARP     one warp per row, row held in registers (narrow d)
 *   RN_VARIANT_BLOCK    a multi-warp CTA per row, row held in registers
 *   RN_VARIANT_STAGED   row copied to shared memory by the bulk-copy (TMA)
 *                       engine, then reduced and written from there
 *   RN_VARIANT_STREAM   any width: statistics in one streaming read, the
 *                       output in a second (x is read twice)
 *   RN_VARIANT_CLUSTER  a row split over a thread-block cluster of 2..16
 *                       CTAs (one per SM), each holding its slice in
 *                       registers; the statistics meet through distributed
 *                       shared memory (rows up to 524288 elements)
 * ------------------------------------------------------------------------ */
enum {
    RN_VARIANT_AUTO = 0,
    RN_VARIANT_WARP = 1,
    RN_VARIANT_BLOCK = 2,
    RN_VARIANT_STAGED = 3,
    RN_VARIANT_STREAM = 4,
    RN_VARIANT_CLUSTER = 5,
    RN_VARIANT_COUNT = 6
};

/* Which kernel configuration a call would launch (host-only; no CUDA call). */
typedef struct rn_plan {
    int variant;          /* RN_VARIANT_* actually chosen                      */
    int vec;              /* elements per vector access: 4 or 1                */
    int slots;            /* vectors held per thread (register and cluster
                             variants); row buffers in the ring (staged)       */
    int threads_per_row;  /* threads cooperating on one row                    */
    int rows_per_cta;     /* rows a CTA works on at once                       */
    int threads_per_cta;
    int smem_bytes;       /* dynamic shared memory per CTA                     */
    int prefetch;         /* 1: the next row's loads overlap this row's work   */
    int params_held;      /* 1: gamma/beta (w) held in registers across rows   */
    int aligned;          /* 1: x, y, params 16-byte aligned and d % 4 == 0    */
    int cluster;          /* CTAs per cluster (cluster variant), else 1        */
} rn_plan;

enum { RN_OP_LN = 0, RN_OP_RMS = 1 };

/* Fill *plan for op RN_OP_LN / RN_OP_RMS, the requested variant (or AUTO),
 * width d and the pointers' alignment (x, y, and the parameter vectors p0 =
 * gamma or w, p1 = beta or NULL). Returns RN_OK, RN_ERR_SIZE or
 * RN_ERR_VARIANT. Performs no CUDA call. */
int rn_plan_for(int op, int variant, int64_t d, const void *x, const void *y,
                const void *p0, const void *p1, rn_plan *plan);

/* The plan of a strided call (ln_fwd_strided / rms_fwd_strided). */
int rn_plan_for_strided(int dtype, int op, int variant, int64_t d, const void *x, int64_t ldx,
                        const void *y, int64_t ldy, const void *p0, const void *p1,
                        rn_plan *plan);

/* rn_plan_for for a storage type (host-only). */
int rn_plan_for_typed(int dtype, int op, int variant, int64_t d, const void *x, const void *y,
                      const void *p0, const void *p1, rn_plan *plan);

/* Short static name of a variant ("warp", "block", ...). */
const char *rn_variant_name(int variant);

int ln_fwd_variant(int variant, const float *x, const float *gamma, const float *beta,
                   float *y, float *mean_out, float *rstd_out,
                   int64_t rows, int64_t d, float eps, void *stream);

int rms_fwd_variant(int variant, const float *x, const float *w, float *y,
                    int64_t rows, int64_t d, float eps, void *stream);

int ln_fwd_residual_variant(int variant, const float *x, const float *res,
                            const float *gamma, const float *beta, float *h_out, float *y,
                            float *mean_out, float *rstd_out, int64_t rows, int64_t d,
                            float eps, void *stream);

int rms_fwd_residual_variant(int variant, const float *x, const float *res, const float *w,
                             float *h_out, float *y, int64_t rows, int64_t d, float eps,
                             void *stream);

/* rn_plan_for for the residual entry points (res and h as they will be
 * passed; h may be NULL). Host-only. */
int rn_plan_for_residual(int op, int variant, int64_t d, const void *x, const void *res,
                         const void *h, const void *y, const void *p0, const void *p1,
                         rn_plan *plan);

/* Device error word of the current device: bit 0 (RN_DEVERR_STAGED_TIMEOUT)
 * is set if a staged kernel's (forward or backward) wait for a bulk copy ran
 * out, bit 1 (RN_DEVERR_CLUSTER_TIMEOUT) if a cluster kernel's wait for its
 * peer CTAs' partial statistics did, bit 2 (RN_DEVERR_PARAMS_TIMEOUT) if a
 * register-held kernel's wait for the bulk copy of gamma/beta (w) into
 * shared memory did (about one second each; the kernel then stops early,
 * or, for bit 2, writes outputs that are not valid). The word is sticky until
 * cleared: `clear` != 0 resets it after reading. Synchronous (a
 * device-to-host copy). Returns RN_OK, RN_ERR_NULL or RN_ERR_CUDA. The
 * kernels find the word's device address once per CUDA context (a device
 * reset gives the device a new context and a new lookup); make one call of
 * each configuration before capturing calls into a CUDA graph. */
enum { RN_DEVERR_STAGED_TIMEOUT = 1, RN_DEVERR_CLUSTER_TIMEOUT = 2, RN_DEVERR_PARAMS_TIMEOUT = 4 };
int rn_device_error(unsigned int *flags, int clear);

/* Self-test of the failure path above (library infrastructure; the paper has
 * no counterpart): launches one CTA on `stream` whose thread waits, through
 * the same bounded wait the staged kernels use, on an mbarrier that nothing
 * ever arrives at. After timeout_us microseconds (1 .. 1000000, else
 * RN_ERR_SIZE) the wait gives up, sets RN_DEVERR_STAGED_TIMEOUT in the
 * device error word and the kernel returns; the context stays usable. No
 * memory other than that word is touched. */
int rn_selftest_bounded_wait(unsigned int timeout_us, void *stream);

/* Whether the current GPU reads ordinary (pageable, unregistered) host
 * memory coherently, through the host's page tables, so that such memory may
 * be passed wherever the Memory convention above allows host memory (GB300
 * over NVLink-C2C does): *pageable = 1 if the device attribute
 * cudaDevAttrPageableMemoryAccess is set, else 0. Pinned memory
 * (cudaHostAlloc / cudaHostRegister) is accepted either way. Host-only (a
 * device attribute query). Returns RN_OK, RN_ERR_NULL or RN_ERR_CUDA. */
int rn_pageable_host_access(int *pageable);

/* Measurement aid: launch an empty kernel with `grid` CTAs of `threads`
 * threads on `stream` (the launch-latency floor small shapes are compared
 * against). grid in [1, 2^31), threads in [1, 1024], else RN_ERR_SIZE. */
int rn_launch_empty(int64_t grid, int threads, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* ROWNORM_H */
