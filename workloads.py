"""Seeded synthetic inputs for row-wise LayerNorm / RMSNorm.

This module is the one thing the CPU oracle (``oracle/``) and the CUDA path
share: it draws input tensors and holds none of the normalization arithmetic.
Tests, ``bench.py`` and ``__graft_entry__.smoke()`` take inputs from here and
hand the same FP32 arrays to both sides.

Distributions and shapes follow the workloads the pages measure:

* LayerNorm at the harness shape [4096, 768] and the sweep shapes [8192, 768],
  [1024, 2048], [4096, 4096] ("LayerNorm [4096,768] is about 10% behind
  Triton's kernel", hypothesis 1 comment) — contiguous FP32.
* RMSNorm at 512 rows with widths 1, 31, 33, 127, 4096, 8193 and the four
  input patterns normal / zeros / small / alternating signs ("RMSNorm on an
  RTX 5070 ...", section "Correctness before timing"), plus width 128 from
  the short-row timing case of the same page.

Readings of points the pages leave open (stated once here):

* ``N(m, s)`` takes ``s`` as the standard deviation.
* "alternating" is ``x[r, c] = +1`` for even column ``c`` and ``-1`` for odd.
* "small" is ``U(-1e-3, 1e-3)``.
* "offset" rows are ``N(0, 2)`` plus one per-row constant drawn from
  ``U(-100, 100)``, which stresses the centred variance.

Every row block of ``BLOCK_ROWS`` rows is drawn from its own generator
``default_rng([seed, stream, block])``, so any subset of rows of a large
workload can be regenerated on the host without materialising the whole
tensor (this is how full-size parity samples rows), and large tensors are
generated in parallel threads (NumPy's generators release the GIL).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

BLOCK_ROWS = 256
EPS = 1e-5

PATTERNS = ("normal", "zeros", "small", "alternating")

# generator stream ids (second seed word)
_S_X = 1
_S_OFFSET = 2
_S_PARAMS = 3


@dataclass(frozen=True)
class Workload:
    """One synthetic normalization problem.

    op      -- "ln" (LayerNorm) or "rms" (RMSNorm)
    rows, d -- x is a contiguous row-major FP32 [rows, d] array
    seed    -- base seed of every generator used
    x_dist  -- "normal" | "zeros" | "small" | "alternating" | "offset"
    x_std   -- standard deviation of the normal part of x
    eps     -- the FP32 epsilon handed to both sides
    """

    op: str
    rows: int
    d: int
    seed: int
    x_dist: str = "normal"
    x_std: float = 1.0
    eps: float = EPS
    tag: str = field(default="", compare=False)

    # ---- parameters -------------------------------------------------------
    def params(self):
        """(gamma, beta) for LayerNorm or (w,) for RMSNorm, FP32 [d].

        gamma and w ~ N(1, 0.1); beta ~ N(0, 0.1).
        """
        rng = np.random.default_rng([self.seed, _S_PARAMS, self.d])
        g = (1.0 + 0.1 * rng.standard_normal(self.d)).astype(np.float32)
        if self.op == "rms":
            return (g,)
        b = (0.1 * rng.standard_normal(self.d)).astype(np.float32)
        return (g, b)

    # ---- x --------------------------------------------------------------
    def _block(self, b: int) -> np.ndarray:
        r0 = b * BLOCK_ROWS
        r1 = min(self.rows, r0 + BLOCK_ROWS)
        n = r1 - r0
        shape = (n, self.d)
        dist = self.x_dist
        if dist == "zeros":
            return np.zeros(shape, np.float32)
        if dist == "alternating":
            row = np.where(np.arange(self.d) % 2 == 0, 1.0, -1.0).astype(np.float32)
            return np.broadcast_to(row, shape).copy()
        rng = np.random.default_rng([self.seed, _S_X, b])
        if dist == "small":
            return rng.uniform(-1e-3, 1e-3, size=shape).astype(np.float32)
        x = rng.standard_normal(shape, dtype=np.float32)
        if self.x_std != 1.0:
            x *= np.float32(self.x_std)
        if dist == "offset":
            orng = np.random.default_rng([self.seed, _S_OFFSET, b])
            off = orng.uniform(-100.0, 100.0, size=(n, 1)).astype(np.float32)
            x += off
        elif dist != "normal":
            raise ValueError(f"unknown x distribution {dist!r}")
        return x

    def x_rows(self, r0: int, r1: int) -> np.ndarray:
        """Rows [r0, r1) of x, FP32, regenerated block by block."""
        r0 = max(0, r0)
        r1 = min(self.rows, r1)
        if r1 <= r0:
            return np.zeros((0, self.d), np.float32)
        b0, b1 = r0 // BLOCK_ROWS, (r1 - 1) // BLOCK_ROWS
        parts = [self._block(b) for b in range(b0, b1 + 1)]
        blk = np.concatenate(parts, axis=0) if len(parts) > 1 else parts[0]
        off = b0 * BLOCK_ROWS
        return blk[r0 - off : r1 - off]

    def x_take(self, rows) -> np.ndarray:
        """The listed rows of x (any order), FP32 [len(rows), d]."""
        rows = np.asarray(rows, dtype=np.int64)
        out = np.empty((len(rows), self.d), np.float32)
        cache = {}
        for i, r in enumerate(rows):
            b = int(r) // BLOCK_ROWS
            if b not in cache:
                cache[b] = self._block(b)
            out[i] = cache[b][int(r) - b * BLOCK_ROWS]
        return out

    def x(self, out: np.ndarray | None = None, threads: int | None = None) -> np.ndarray:
        """All of x, FP32 [rows, d]; large tensors are drawn in threads."""
        if out is None:
            out = np.empty((self.rows, self.d), np.float32)
        nb = (self.rows + BLOCK_ROWS - 1) // BLOCK_ROWS
        if threads is None:
            threads = min(16, os.cpu_count() or 1)

        def fill(b):
            r0 = b * BLOCK_ROWS
            blk = self._block(b)
            out[r0 : r0 + blk.shape[0]] = blk

        if nb <= 4 or threads <= 1:
            for b in range(nb):
                fill(b)
        else:
            with ThreadPoolExecutor(threads) as ex:
                list(ex.map(fill, range(nb)))
        return out

    @property
    def nbytes_x(self) -> int:
        return 4 * self.rows * self.d


# --------------------------------------------------------------------------
# The five workload families, by what they are.
# --------------------------------------------------------------------------

def ln_512x128() -> Workload:
    """LayerNorm, 512 x 128, x ~ N(0,1), seed 0 (the small launch-bound case)."""
    return Workload("ln", 512, 128, seed=0, tag="ln_512x128")


def ln_4096x768() -> Workload:
    """LayerNorm at the pages' harness shape [4096, 768], seed 1."""
    return Workload("ln", 4096, 768, seed=1, tag="ln_4096x768")


RMS_WIDTHS = (1, 31, 33, 127, 128, 4096, 8193)


def rms_512_matrix():
    """RMSNorm, 512 rows x widths {1,31,33,127,128,4096,8193} x 4 patterns, seed 2."""
    out = []
    for d in RMS_WIDTHS:
        for p in PATTERNS:
            out.append(Workload("rms", 512, d, seed=2, x_dist=p, tag=f"rms_512x{d}_{p}"))
    return out


SWEEP_SHAPES = ((8192, 768), (1024, 2048), (4096, 4096), (16384, 1024))


def sweep_offset():
    """LN and RMS over the sweep shapes, x ~ N(0,2) + per-row U(-100,100), seed 3."""
    out = []
    for op in ("ln", "rms"):
        for rows, d in SWEEP_SHAPES:
            out.append(Workload(op, rows, d, seed=3, x_dist="offset", x_std=2.0,
                                tag=f"{op}_{rows}x{d}_offset"))
    return out


def large_32768x8192(op: str = "ln") -> Workload:
    """LN or RMS at 32768 x 8192 (1 GiB in, 1 GiB out), x ~ N(0,1), seed 4."""
    return Workload(op, 32768, 8192, seed=4, tag=f"{op}_32768x8192")


# --------------------------------------------------------------------------
# 16-bit storage: FP32 values rounded to BF16 or FP16 (nearest even). Returns
# the 16-bit patterns (uint16) and their exact FP32 values, which both sides
# use (the GPU receives the patterns, the oracle the widened values).
# --------------------------------------------------------------------------

def to_storage(a, dtype: str):
    a = np.ascontiguousarray(a, np.float32)
    if dtype == "f32":
        return a, a
    if dtype == "f16":
        h = a.astype(np.float16)
        return h.view(np.uint16), h.astype(np.float32)
    if dtype == "bf16":
        u = a.view(np.uint32)
        bits = ((u + (((u >> 16) & 1) + np.uint32(0x7FFF))) >> 16).astype(np.uint16)
        return bits, (bits.astype(np.uint32) << 16).view(np.float32)
    raise ValueError(dtype)


def from_storage(bits, dtype: str):
    """FP32 values of 16-bit patterns."""
    bits = np.asarray(bits)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float32)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32)
    raise ValueError(dtype)
