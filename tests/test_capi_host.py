"""The C-ABI library on the host: it loads, exports every symbol the header
declares, and validates arguments before touching CUDA (no GPU needed)."""
import ctypes
import math
import os
import re

import pytest

from row_wise_normalization_gb300 import capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rownorm.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b([A-Za-z_]\w*)\s*\([^;{)]*(?:\([^)]*\)[^;{)]*)*\)\s*;", src)
    return sorted(set(n for n in names if n not in ("if", "return", "sizeof")))


@pytest.fixture(scope="module")
def lib():
    return capi.load()


def test_header_functions_parsed():
    names = _declared_functions()
    assert {"ln_fwd", "rms_fwd", "rn_status_str"} <= set(names)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"librownorm.so does not export {name}"
        assert name in capi.SIGNATURES, f"capi.py does not declare {name}"


def test_status_strings(lib):
    seen = set()
    for s in range(0, capi.RN_ERR_HOSTMEM + 1):
        assert capi.status_str(s) != "unknown status", s
        seen.add(capi.status_str(s))
    assert len(seen) == capi.RN_ERR_HOSTMEM + 1, "two statuses share a string"
    for v in range(capi.RN_VARIANT_COUNT):
        assert capi.variant_name(v) != "unknown"
    assert capi.status_str(99) == "unknown status"
    assert capi.variant_name(capi.RN_VARIANT_WARP) == "warp"


A = 1 << 20   # fake, 16-byte aligned "device" addresses; never dereferenced


def _ln(**kw):
    args = dict(x=A, gamma=A + 0x100000, beta=A + 0x200000, y=A + 0x300000,
                mean_out=0, rstd_out=0, rows=4, d=8, eps=1e-5, stream=0)
    args.update(kw)
    return capi.ln_fwd(**args)


def test_validation_errors_without_launch(lib):
    assert _ln(rows=-1) == capi.RN_ERR_SIZE
    assert _ln(d=0) == capi.RN_ERR_SIZE
    assert _ln(d=-3) == capi.RN_ERR_SIZE
    assert _ln(rows=1 << 40, d=1 << 30) == capi.RN_ERR_SIZE
    assert _ln(eps=-1e-5) == capi.RN_ERR_EPS
    assert _ln(eps=math.nan) == capi.RN_ERR_EPS
    assert _ln(eps=math.inf) == capi.RN_ERR_EPS
    assert _ln(x=0) == capi.RN_ERR_NULL
    assert _ln(y=0) == capi.RN_ERR_NULL
    assert _ln(gamma=0) == capi.RN_ERR_NULL
    assert _ln(beta=0) == capi.RN_ERR_NULL
    assert _ln(x=A + 2) == capi.RN_ERR_ALIGN
    assert _ln(mean_out=A + 0x400001) == capi.RN_ERR_ALIGN
    # outputs overlapping inputs or each other
    assert _ln(y=A + 4) == capi.RN_ERR_ALIAS
    assert _ln(y=A + 0x100000 - 8) == capi.RN_ERR_ALIAS          # y's tail over gamma
    assert _ln(mean_out=A + 0x200000 + 4) == capi.RN_ERR_ALIAS    # mean inside beta
    assert _ln(mean_out=A + 0x400000, rstd_out=A + 0x400008) == capi.RN_ERR_ALIAS
    assert capi.rms_fwd(A, A + 0x1000, A + 16, 4, 8, 1e-5, 0) == capi.RN_ERR_ALIAS
    assert capi.rms_fwd(A, 0, A + 0x1000, 4, 8, 1e-5, 0) == capi.RN_ERR_NULL


def test_empty_is_a_noop(lib):
    assert _ln(rows=0, x=0, y=0, gamma=0, beta=0) == capi.RN_OK
    assert capi.rms_fwd(0, 0, 0, 0, 5, 1e-5, 0) == capi.RN_OK
    # eps zero is allowed
    assert _ln(rows=0, eps=0.0) == capi.RN_OK


def test_bad_variant(lib):
    assert capi.ln_fwd_variant(99, A, A + 0x100000, A + 0x200000, A + 0x300000, 0, 0, 4, 8,
                               1e-5, 0) == capi.RN_ERR_VARIANT
    assert capi.rms_fwd_variant(-1, A, A + 0x1000, A + 0x2000, 4, 8, 1e-5, 0) == capi.RN_ERR_VARIANT


@pytest.mark.parametrize("d,variant,tpr,slots", [
    (1, capi.RN_VARIANT_WARP, 32, 1),
    (128, capi.RN_VARIANT_WARP, 32, 1),
    (768, capi.RN_VARIANT_WARP, 32, 6),
    (1027, capi.RN_VARIANT_WARP, 32, 8),
    (1028, capi.RN_VARIANT_BLOCK, 64, 5),
    (4096, capi.RN_VARIANT_BLOCK, 128, 8),
    (8193, capi.RN_VARIANT_BLOCK, 256, 8),
    (8196, capi.RN_VARIANT_BLOCK, 512, 5),
    (16384, capi.RN_VARIANT_BLOCK, 512, 8),
    (32771, capi.RN_VARIANT_BLOCK, 1024, 8),
    (32772, capi.RN_VARIANT_CLUSTER, 8 * 256, 6),
    (65536, capi.RN_VARIANT_CLUSTER, 8 * 256, 8),
    (131072, capi.RN_VARIANT_CLUSTER, 16 * 256, 8),
    (262144, capi.RN_VARIANT_CLUSTER, 16 * 512, 8),
    (524288, capi.RN_VARIANT_CLUSTER, 16 * 1024, 8),
    (524292, capi.RN_VARIANT_STREAM, 512, 0),
])
def test_plan_by_width(lib, d, variant, tpr, slots):
    p = capi.plan(capi.RN_OP_LN, capi.RN_VARIANT_AUTO, d, A, A + 0x1000000)
    assert (p.variant, p.vec, p.threads_per_row, p.slots) == (variant, 4, tpr, slots)


@pytest.mark.parametrize("d,op,variant,cl", [
    (16384, capi.RN_OP_LN, capi.RN_VARIANT_BLOCK, 1),      # 512 threads
    (16388, capi.RN_OP_LN, capi.RN_VARIANT_CLUSTER, 4),    # past 512 threads: cluster
    (20000, capi.RN_OP_LN, capi.RN_VARIANT_CLUSTER, 4),
    (32768, capi.RN_OP_LN, capi.RN_VARIANT_CLUSTER, 4),
    (20000, capi.RN_OP_RMS, capi.RN_VARIANT_BLOCK, 1),     # RMSNorm: one CTA per row
    (32768, capi.RN_OP_RMS, capi.RN_VARIANT_BLOCK, 1),
])
def test_aligned_layernorm_rows_past_512_threads_take_the_cluster(lib, d, op, variant, cl):
    p = capi.plan(op, capi.RN_VARIANT_AUTO, d, A, A + 0x1000000, A + 0x2000000, A + 0x3000000)
    assert (p.variant, p.cluster) == (variant, cl)
    # rows whose accesses are not all aligned stay on one CTA per row
    p = capi.plan(op, capi.RN_VARIANT_AUTO, d, A, A + 0x1000000, A + 0x2000004, 0)
    assert p.variant == capi.RN_VARIANT_BLOCK


@pytest.mark.parametrize("d,stages", [(1, 4), (3, 4), (4, 4), (8192, 4), (14464, 4),
                                      (14468, 3), (19264, 3), (19268, 2), (28928, 2),
                                      (28932, 1), (57856, 1)])
def test_staged_ring_depth(lib, d, stages):
    """Row buffers of 16*(d/4) bytes (rounded to 128) fill at most 226 KiB, up to 4 of them."""
    p = capi.plan(capi.RN_OP_LN, capi.RN_VARIANT_STAGED, d, A, A + 0x1000000)
    assert p.variant == capi.RN_VARIANT_STAGED and p.slots == stages
    sb = ((d // 4) * 16 + 127) // 128 * 128
    assert p.smem_bytes == stages * sb and p.smem_bytes <= 232448 - 1024


@pytest.mark.parametrize("d,cl,threads,slots", [(8196, 2, 256, 6), (12288, 2, 256, 6),
                                               (12292, 2, 256, 8), (20000, 4, 256, 6),
                                               (100000, 16, 256, 8), (400000, 16, 1024, 8)])
def test_cluster_shape(lib, d, cl, threads, slots):
    """The fewest CTAs of 256 threads (then 512, 1024) whose slices hold the row."""
    p = capi.plan(capi.RN_OP_RMS, capi.RN_VARIANT_CLUSTER, d, A, A + 0x10000000)
    assert (p.cluster, p.threads_per_cta, p.slots) == (cl, threads, slots)
    assert p.cluster * p.threads_per_cta * p.slots * 4 >= d


def test_cluster_needs_matching_phases(lib):
    with pytest.raises(capi.RowNormError):
        capi.plan(capi.RN_OP_LN, capi.RN_VARIANT_CLUSTER, 40000, A, A + 4)
    with pytest.raises(capi.RowNormError):
        capi.plan(capi.RN_OP_LN, capi.RN_VARIANT_CLUSTER, 524292, A, A + 0x1000000)


def test_staged_needs_matching_phases(lib):
    with pytest.raises(capi.RowNormError):
        capi.plan(capi.RN_OP_LN, capi.RN_VARIANT_STAGED, 40000, A, A + 4)
    p = capi.plan(capi.RN_OP_LN, capi.RN_VARIANT_AUTO, 40000, A, A + 4)
    assert p.variant == capi.RN_VARIANT_STREAM and p.vec == 1
    p = capi.plan(capi.RN_OP_LN, capi.RN_VARIANT_STAGED, 40000, A, A + 0x1000000)
    assert p.variant == capi.RN_VARIANT_STAGED


def test_plan_phase_mismatch_goes_scalar(lib):
    p = capi.plan(capi.RN_OP_RMS, capi.RN_VARIANT_AUTO, 768, A, A + 4)
    assert p.vec == 1 and p.variant == capi.RN_VARIANT_BLOCK
    p = capi.plan(capi.RN_OP_RMS, capi.RN_VARIANT_AUTO, 200, A + 4, A + 0x1004)
    assert p.vec == 4 and p.variant == capi.RN_VARIANT_WARP


def test_forced_variant_limits(lib):
    with pytest.raises(capi.RowNormError):
        capi.plan(capi.RN_OP_LN, capi.RN_VARIANT_WARP, 1028, A, A + 0x100000)
    with pytest.raises(capi.RowNormError):
        capi.plan(capi.RN_OP_LN, capi.RN_VARIANT_BLOCK, 32772, A, A + 0x100000)
    p = capi.plan(capi.RN_OP_LN, capi.RN_VARIANT_STREAM, 5, A, A + 0x100000)
    assert p.variant == capi.RN_VARIANT_STREAM


def test_torch_binding_rejects_cpu_tensors():
    """Unpinned CPU tensors are refused unless the GPU reads pageable host
    memory (where they are accepted; the GPU tests cover that)."""
    torch = pytest.importorskip("torch")
    import row_wise_normalization_gb300 as rn
    if torch.cuda.is_available() and capi.pageable_host_access():
        pytest.skip("this GPU reads pageable host memory")
    x = torch.zeros(2, 4)
    with pytest.raises(ValueError):
        rn.ln_fwd(x, torch.ones(4), torch.zeros(4))
    with pytest.raises(ValueError):
        rn.rms_fwd(x, torch.ones(4))


def test_residual_validation(lib):
    R = A + 0x400000
    H = A + 0x500000
    f = lambda **k: capi.ln_fwd_residual(**{**dict(x=A, res=R, gamma=A + 0x100000,
                                                   beta=A + 0x200000, h_out=H, y=A + 0x300000,
                                                   mean_out=0, rstd_out=0, rows=4, d=8,
                                                   eps=1e-5, stream=0), **k})
    assert f(res=0) == capi.RN_ERR_NULL
    assert f(h_out=R) == capi.RN_ERR_ALIAS          # in place over the residual
    assert f(h_out=A) == capi.RN_ERR_ALIAS          # over x
    assert f(y=R + 16) == capi.RN_ERR_ALIAS         # y over the residual
    assert f(h_out=A + 0x300000) == capi.RN_ERR_ALIAS   # h over y
    assert f(res=R + 2) == capi.RN_ERR_ALIGN
    assert f(rows=0, x=0, res=0) == capi.RN_OK
    assert capi.rms_fwd_residual(A, 0, A + 0x1000, 0, A + 0x2000, 4, 8, 1e-5, 0) == capi.RN_ERR_NULL


def test_residual_plans(lib):
    X, Y = A, A + 0x1000000
    p = capi.plan_residual(capi.RN_OP_LN, capi.RN_VARIANT_AUTO, 768, X, X + 0x100000,
                           Y + 0x100000, Y)
    assert p.variant == capi.RN_VARIANT_WARP and p.vec == 4 and p.aligned == 1
    # a residual in another 16-byte phase makes every access scalar
    p = capi.plan_residual(capi.RN_OP_LN, capi.RN_VARIANT_AUTO, 768, X, X + 0x100004,
                           Y + 0x100000, Y)
    assert p.vec == 1
    # rows past 16384 floats stream
    p = capi.plan_residual(capi.RN_OP_RMS, capi.RN_VARIANT_AUTO, 20000, X, X + 0x1000000, 0, Y)
    assert p.variant == capi.RN_VARIANT_STREAM
    for v in (capi.RN_VARIANT_STAGED, capi.RN_VARIANT_CLUSTER):
        with pytest.raises(capi.RowNormError):
            capi.plan_residual(capi.RN_OP_LN, v, 40000, X, X + 0x1000000, 0, Y)


def test_typed_plans_and_validation(lib):
    X, Y = A, A + 0x1000000
    p = capi.plan_typed(capi.RN_DTYPE_BF16, capi.RN_OP_LN, capi.RN_VARIANT_AUTO, 768, X, Y, X, X)
    assert (p.variant, p.vec, p.slots, p.aligned) == (capi.RN_VARIANT_WARP, 8, 3, 1)
    p = capi.plan_typed(capi.RN_DTYPE_F16, capi.RN_OP_RMS, capi.RN_VARIANT_AUTO, 4096, X, Y)
    assert (p.variant, p.vec, p.threads_per_row, p.slots) == (capi.RN_VARIANT_BLOCK, 8, 128, 4)
    p = capi.plan_typed(capi.RN_DTYPE_BF16, capi.RN_OP_RMS, capi.RN_VARIANT_AUTO, 40000, X, Y)
    assert p.variant == capi.RN_VARIANT_STREAM
    # 2-byte phases differ from 16-byte phases: scalar path
    p = capi.plan_typed(capi.RN_DTYPE_BF16, capi.RN_OP_RMS, capi.RN_VARIANT_AUTO, 768, X + 2, Y)
    assert p.vec == 1
    with pytest.raises(capi.RowNormError):
        capi.plan_typed(capi.RN_DTYPE_BF16, capi.RN_OP_LN, capi.RN_VARIANT_CLUSTER, 40000, X, Y)
    with pytest.raises(capi.RowNormError):
        capi.plan_typed(7, capi.RN_OP_LN, capi.RN_VARIANT_AUTO, 64, X, Y)
    # validation: 2-byte alignment for 16-bit, unknown dtype
    assert capi.ln_fwd_typed(capi.RN_DTYPE_BF16, 0, X + 1, X + 0x100000, X + 0x200000, Y, 0, 0,
                             4, 8, 1e-5, 0) == capi.RN_ERR_ALIGN
    assert capi.ln_fwd_typed(9, 0, X, X + 0x100000, X + 0x200000, Y, 0, 0, 4, 8, 1e-5,
                             0) == capi.RN_ERR_DTYPE
    assert capi.rms_fwd_typed(capi.RN_DTYPE_F16, 0, X, X + 0x100000, X + 8, 4, 8, 1e-5,
                              0) == capi.RN_ERR_ALIAS
    # statistics stay FP32: 4-byte alignment even with 16-bit data
    assert capi.ln_fwd_typed(capi.RN_DTYPE_BF16, 0, X, X + 0x100000, X + 0x200000, Y,
                             X + 0x300002, 0, 4, 8, 1e-5, 0) == capi.RN_ERR_ALIGN


def test_strided_plans_and_validation(lib):
    X, Y = A, A + 0x1000000
    F32, BF16 = capi.RN_DTYPE_F32, capi.RN_DTYPE_BF16
    LN, AUTO = capi.RN_OP_LN, capi.RN_VARIANT_AUTO
    # a column block of a wider matrix: strides a multiple of 4, everything aligned
    p = capi.plan_strided(F32, LN, AUTO, 768, X, 3 * 768, Y, 768, X, X)
    assert (p.variant, p.vec, p.aligned) == (capi.RN_VARIANT_WARP, 4, 1)
    # strides that agree modulo 4 but are not multiples of 4: vector path with head peel
    p = capi.plan_strided(F32, LN, AUTO, 768, X, 771, Y, 775, X, X)
    assert (p.vec, p.aligned) == (4, 0)
    # strides that disagree modulo 4: rows change relative phase, scalar path
    p = capi.plan_strided(F32, LN, AUTO, 768, X, 770, Y, 768, X, X)
    assert p.vec == 1
    # 16-bit: agreement modulo 8 elements
    p = capi.plan_strided(BF16, LN, AUTO, 1024, X, 1032, Y, 1024, X, X)
    assert (p.vec, p.aligned) == (8, 1)
    p = capi.plan_strided(BF16, LN, AUTO, 1024, X, 1028, Y, 1024, X, X)
    assert p.vec == 1
    # wide rows keep their variants when the phases agree
    p = capi.plan_strided(F32, LN, AUTO, 65536, X, 65540, Y, 65536, X, X)
    assert p.variant == capi.RN_VARIANT_CLUSTER
    p = capi.plan_strided(F32, LN, capi.RN_VARIANT_STAGED, 20000, X, 20004, Y, 20000, X, X)
    assert p.variant == capi.RN_VARIANT_STAGED
    with pytest.raises(capi.RowNormError):
        capi.plan_strided(F32, LN, capi.RN_VARIANT_STAGED, 20000, X, 20002, Y, 20000, X, X)
    with pytest.raises(capi.RowNormError):
        capi.plan_strided(F32, LN, AUTO, 768, X, 700, Y, 768, X, X)
    G, B, M, S = X + 0x2000000, X + 0x2100000, X + 0x2200000, X + 0x2300000
    # strides below d are rejected before anything runs
    assert capi.ln_fwd_strided(F32, AUTO, X, 767, G, B, Y, 768, M, S, 4, 768, 1e-5,
                               0) == capi.RN_ERR_SIZE
    assert capi.ln_fwd_strided(F32, AUTO, X, 768, G, B, Y, 0, M, S, 4, 768, 1e-5,
                               0) == capi.RN_ERR_SIZE
    assert capi.rms_fwd_strided(F32, AUTO, X, -4, G, Y, 768, 4, 768, 1e-5, 0) == capi.RN_ERR_SIZE
    # spans: y interleaved with x's rows (y = x + d, both with stride 2d) is an alias
    assert capi.ln_fwd_strided(F32, AUTO, X, 1536, G, B, X + 4 * 768, 1536, M, S, 4, 768, 1e-5,
                               0) == capi.RN_ERR_ALIAS
    # a stride that makes the span overflow
    assert capi.ln_fwd_strided(F32, AUTO, X, 1 << 60, G, B, Y, 768, M, S, 16, 768, 1e-5,
                               0) == capi.RN_ERR_SIZE
    # empty batch: nothing runs
    assert capi.ln_fwd_strided(F32, AUTO, 0, 1000, 0, 0, 0, 1000, 0, 0, 0, 768, 1e-5,
                               0) == capi.RN_OK


def test_batched_validation_without_launch(lib):
    X = A
    F32 = capi.RN_DTYPE_F32
    ok = (X, X + 0x100000, X + 0x200000, X + 0x300000, 0, 0, 4, 64)
    assert capi.ln_fwd_batched(F32, capi.problems([]), 0, 1e-5, 0) == capi.RN_OK
    assert capi.ln_fwd_batched(F32, capi.problems([ok]), -1, 1e-5, 0) == capi.RN_ERR_SIZE
    assert capi.ln_fwd_batched(F32, None, 3, 1e-5, 0) == capi.RN_ERR_NULL
    assert capi.ln_fwd_batched(7, capi.problems([ok]), 1, 1e-5, 0) == capi.RN_ERR_DTYPE
    assert capi.ln_fwd_batched(F32, capi.problems([ok]), 1, -1.0, 0) == capi.RN_ERR_EPS
    # a bad problem anywhere stops the whole call before anything runs
    bad_null = (0, X + 0x100000, X + 0x200000, X + 0x400000, 0, 0, 4, 64)
    assert capi.ln_fwd_batched(F32, capi.problems([ok, bad_null]), 2, 1e-5,
                               0) == capi.RN_ERR_NULL
    bad_size = (X + 0x500000, X + 0x100000, X + 0x200000, X + 0x600000, 0, 0, 4, 0)
    assert capi.ln_fwd_batched(F32, capi.problems([ok, bad_size]), 2, 1e-5,
                               0) == capi.RN_ERR_SIZE
    # problem 2 writes problem 1's input
    clash = (X + 0x700000, X + 0x100000, X + 0x200000, X + 16, 0, 0, 4, 64)
    assert capi.ln_fwd_batched(F32, capi.problems([ok, clash]), 2, 1e-5,
                               0) == capi.RN_ERR_ALIAS
    # two problems writing the same y
    twin = (X + 0x800000, X + 0x100000, X + 0x200000, X + 0x300000, 0, 0, 4, 64)
    assert capi.rms_fwd_batched(F32, capi.problems([ok, twin]), 2, 1e-5,
                                0) == capi.RN_ERR_ALIAS
    # sharing read-only parameters is fine (only checked here up to validation:
    # rows == 0 problems run nothing)
    empty = [(X + 0x900000 * (i + 1), X + 0x100000, X + 0x200000, X + 0x300000 + 0x900000 * (i + 1),
              0, 0, 0, 64) for i in range(3)]
    assert capi.ln_fwd_batched(F32, capi.problems(empty), 3, 1e-5, 0) == capi.RN_OK


def test_bounded_wait_selftest_rejects_out_of_range_limits(lib):
    assert capi.selftest_bounded_wait(0, 0) == capi.RN_ERR_SIZE
    assert capi.selftest_bounded_wait(2000000, 0) == capi.RN_ERR_SIZE


def test_no_alloc_checks_arguments_before_its_width_limit(lib):
    """ln_bwd_noalloc reports what ln_bwd would report before its own width
    limit: rows == 0 is a no-op at any width, a NULL input is RN_ERR_NULL, and
    only a call that needs the static partials (parameter gradients wanted,
    rows > 0) is refused for d > RN_NOALLOC_MAX_D. None of these calls reaches
    CUDA."""
    d = capi.RN_NOALLOC_MAX_D + 904
    rows = 5
    nd, nr = rows * d * 4, rows * 4
    base = A
    ptrs = {}
    for name, n in (("dy", nd), ("x", nd), ("gamma", 4 * d), ("mean", nr), ("rstd", nr),
                    ("dx", nd), ("dgamma", 4 * d), ("dbeta", 4 * d)):
        ptrs[name] = base
        base += (n + 0xFFFF) & ~0xFFFF
    order = ("dy", "x", "gamma", "mean", "rstd", "dx", "dgamma", "dbeta")

    def call(rows_, **kw):
        p = dict(ptrs)
        p.update(kw)
        return capi.ln_bwd_noalloc(*[p[k] for k in order], rows_, d, 0)

    assert call(0, **{k: 0 for k in order}) == capi.RN_OK
    assert call(rows, dy=0) == capi.RN_ERR_NULL
    assert call(rows, dx=ptrs["x"]) == capi.RN_ERR_ALIAS
    assert call(rows, dgamma=ptrs["dgamma"] + 2) == capi.RN_ERR_ALIGN
    assert call(-1) == capi.RN_ERR_SIZE
    assert call(rows) == capi.RN_ERR_SCRATCH
    assert call(rows, dgamma=0) == capi.RN_ERR_SCRATCH


def _widths():
    ws = set(range(1, 300)) | {w + k for w in (384, 512, 768, 1024, 1536, 2048, 3072, 4096,
                                                6144, 8192, 12288, 16384, 24576, 32768,
                                                49152, 65536, 98304, 131072, 262144, 524288)
                               for k in range(-9, 10)}
    return sorted(w for w in ws if w > 0)


@pytest.mark.parametrize("dtype", [capi.RN_DTYPE_F32, capi.RN_DTYPE_BF16, capi.RN_DTYPE_F16])
def test_every_planned_configuration_is_compiled(lib, dtype):
    """Only the configurations the planner can choose are compiled. A call
    whose plan succeeds (any variant, forced or AUTO) must get as far as the
    launch: on a machine without a GPU that is RN_ERR_CUDA (the first CUDA
    call fails), while a configuration missing from the library returns
    RN_ERR_VARIANT before any CUDA call."""
    es = 4 if dtype == capi.RN_DTYPE_F32 else 2
    X, Y, P = A, A + (1 << 28), A + (1 << 29)
    for d in _widths():
        for xo, yo, po in ((0, 0, 0), (1, 1, 0), (3, 3, 2), (0, 1, 0)):
            x, y, g = X + es * xo, Y + es * yo, P + es * po
            b = g + (1 << 20)
            for v in range(capi.RN_VARIANT_COUNT):
                for op in (capi.RN_OP_LN, capi.RN_OP_RMS):
                    p1 = b if op == capi.RN_OP_LN else 0
                    try:
                        capi.plan_typed(dtype, op, v, d, x, y, g, p1)
                    except capi.RowNormError:
                        continue
                    if op == capi.RN_OP_LN:
                        st = capi.ln_fwd_typed(dtype, v, x, g, b, y, 0, 0, 3, d, 1e-5, 0)
                    else:
                        st = capi.rms_fwd_typed(dtype, v, x, g, y, 3, d, 1e-5, 0)
                    assert st == capi.RN_ERR_CUDA, (dtype, op, v, d, xo, yo, po, st)
                    if dtype != capi.RN_DTYPE_F32:
                        continue
                    # the residual forms of the same rows
                    r = A + (1 << 30) + 4 * xo
                    try:
                        capi.plan_residual(op, v, d, x, r, 0, y, g, p1)
                    except capi.RowNormError:
                        continue
                    if op == capi.RN_OP_LN:
                        st = capi.ln_fwd_residual_variant(v, x, r, g, b, 0, y, 0, 0, 3, d,
                                                          1e-5, 0)
                    else:
                        st = capi.rms_fwd_residual_variant(v, x, r, g, 0, y, 3, d, 1e-5, 0)
                    assert st == capi.RN_ERR_CUDA, ("res", op, v, d, xo, yo, po, st)
