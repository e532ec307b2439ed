"""Seeded synthetic inputs for the fused residual-add + RMSNorm workloads.

This module only draws random numbers and rounds them to the storage type
(through torch's float32 -> bfloat16 conversion).  It holds none of the
normalisation arithmetic, so the CPU oracle and the CUDA path can both be fed
from it without sharing any of the method's code.

Determinism and row sampling
----------------------------
Every [T, H] tensor is drawn in blocks of ``ROW_BLOCK`` rows.  Block ``k`` of
tensor ``tag`` in workload ``seed`` has its own PCG64 stream keyed by
``SeedSequence([seed, tag, k])``.  A single row of a huge tensor can therefore
be regenerated on its own (``rows=...``) with exactly the values the full
tensor holds, which is how full-size parity checks sample rows without
materialising the whole tensor a second time.

Workloads (distributions as in the blog "CuTeDSL at Perplexity" discussion of
the regular RMS norm, with the sizes of the five hot-path configurations):

* ``fp32``    x[64, 1024] ~ N(0,1) fp32, w = 1 + 0.1 N(0,1) fp32, no residual,
              no bias, eps 1e-6.
* ``decode``  T in {1, 8, 32, 128, 256}, H = 4096, bf16 x, r ~ N(0,1),
              w = 1 + 0.1 N(0,1), eps 1e-6.
* ``prefill`` T = 16384, H = 8192, bf16, x ~ N(0,1) with 1 % of the channels
              (round(0.01 H) distinct columns picked by a seeded permutation)
              scaled by 50 before rounding, r ~ N(0, variance 4),
              w = 1 + 0.1 N(0,1), eps 1e-5.
* ``fp8``     T = 4096, H in {5120, 7168}, bf16 x, r ~ N(0,1),
              w = 1 + 0.1 N(0,1), per-channel bias 0.01 N(0,1), FP8-e4m3
              output with a per-token scale, eps 1e-6.
* ``sweep``   T in {1,4,16,64,256,1024,4096,16384,65536} x
              H in {2048,4096,8192,16384}, bf16, x ~ Student-t(3) clipped to
              +-1e4, r ~ N(0,1), w = 1 + 0.1 N(0,1), eps 1e-6.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

ROW_BLOCK = 64

# stream tags: one independent stream family per tensor role
TAG_X, TAG_R, TAG_W, TAG_B, TAG_OUTLIER = 1, 2, 3, 4, 5

DECODE_TOKENS = (1, 8, 32, 128, 256)
SWEEP_TOKENS = (1, 4, 16, 64, 256, 1024, 4096, 16384, 65536)
SWEEP_HIDDEN = (2048, 4096, 8192, 16384)
FP8_HIDDEN = (5120, 7168)


@dataclass(frozen=True)
class Workload:
    """Shape, dtypes, distributions and seed of one synthetic workload."""
    name: str
    n_tokens: int
    hidden: int
    seed: int
    in_dtype: str              # "f32" | "bf16" | "f16"
    out_dtype: str             # "f32" | "bf16" | "f16" | "fp8"
    eps: float
    has_residual: bool = True
    has_weight: bool = True
    has_bias: bool = False
    x_dist: str = "normal"     # "normal" | "student_t3"
    r_std: float = 1.0
    outlier_frac: float = 0.0  # fraction of channels of x scaled by outlier_scale
    outlier_scale: float = 50.0
    res_dtype: str | None = None  # residual stream storage; None = in_dtype ("f32" under bf16 / f16)
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def res_storage(self) -> str:
        return self.res_dtype or self.in_dtype

    @property
    def in_bytes(self) -> int:
        return 4 if self.in_dtype == "f32" else 2  # bf16 / f16

    @property
    def out_bytes(self) -> int:
        return {"f32": 4, "bf16": 2, "f16": 2, "fp8": 1}[self.out_dtype]

    def algorithmic_bytes(self) -> int:
        """Minimum HBM bytes one call must move (each tensor touched once)."""
        T, H = self.n_tokens, self.hidden
        b = T * H * self.in_bytes                      # read x
        if self.has_residual:
            rb = 4 if self.res_storage == "f32" else 2
            b += 2 * T * H * rb                        # read r, write residual_out
        b += T * H * self.out_bytes                    # write y (or q)
        if self.out_dtype == "fp8":
            b += 4 * T                                 # per-token scales
        if self.has_weight:
            b += H * self.in_bytes
        if self.has_bias:
            b += H * self.in_bytes
        return b


def fp32_workload() -> Workload:
    return Workload("fp32", 64, 1024, 1, "f32", "f32", 1e-6, has_residual=False)


def decode_workload(n_tokens: int) -> Workload:
    return Workload(f"decode_T{n_tokens}", n_tokens, 4096, 10 + n_tokens, "bf16", "bf16", 1e-6)


def prefill_workload(n_tokens: int = 16384, hidden: int = 8192) -> Workload:
    return Workload("prefill", n_tokens, hidden, 30, "bf16", "bf16", 1e-5,
                    r_std=2.0, outlier_frac=0.01)


def fp8_workload(hidden: int, n_tokens: int = 4096) -> Workload:
    return Workload(f"fp8_H{hidden}", n_tokens, hidden, 40, "bf16", "fp8", 1e-6, has_bias=True)


def sweep_workload(n_tokens: int, hidden: int) -> Workload:
    return Workload(f"sweep_T{n_tokens}_H{hidden}", n_tokens, hidden, 50, "bf16", "bf16", 1e-6,
                    x_dist="student_t3")


# ----------------------------------------------------------------------------
# raw draws


def _rng(seed: int, tag: int, block: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, block])))


def _draw_block(dist: str, seed: int, tag: int, block: int, rows: int, cols: int) -> np.ndarray:
    g = _rng(seed, tag, block)
    if dist == "normal":
        return g.standard_normal((rows, cols), dtype=np.float32)
    if dist == "student_t3":
        t = g.standard_t(3.0, size=(rows, cols))
        return np.clip(t, -1e4, 1e4).astype(np.float32)
    raise ValueError(dist)


def _draw_range(dist: str, seed: int, tag: int, lo: int, hi: int, cols: int) -> np.ndarray:
    """Rows [lo, hi) of a block-seeded draw, blocks generated in parallel."""
    out = np.empty((hi - lo, cols), dtype=np.float32)
    if hi <= lo:
        return out

    def fill(k: int) -> None:
        b = _draw_block(dist, seed, tag, k, ROW_BLOCK, cols)
        a, z = max(lo, k * ROW_BLOCK), min(hi, (k + 1) * ROW_BLOCK)
        out[a - lo:z - lo] = b[a - k * ROW_BLOCK:z - k * ROW_BLOCK]

    blocks = range(lo // ROW_BLOCK, (hi - 1) // ROW_BLOCK + 1)
    workers = min(len(blocks), os.cpu_count() or 1, 32)
    if workers > 1:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, blocks))
    else:
        for k in blocks:
            fill(k)
    return out


def _draw_rows(dist: str, seed: int, tag: int, n_rows: int, cols: int,
               rows) -> np.ndarray:
    """Rows of a [n_rows, cols] float32 draw: all rows, a ``range`` of rows,
    or the rows listed in an index array."""
    if rows is None:
        return _draw_range(dist, seed, tag, 0, n_rows, cols)
    if isinstance(rows, range) and rows.step == 1:
        if rows.start < 0 or rows.stop > n_rows:
            raise IndexError("row range out of bounds")
        return _draw_range(dist, seed, tag, rows.start, rows.stop, cols)
    rows = np.asarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= n_rows):
        raise IndexError("row index out of range")
    out = np.empty((rows.size, cols), dtype=np.float32)
    cache: dict[int, np.ndarray] = {}
    for i, t in enumerate(rows):
        k = int(t) // ROW_BLOCK
        if k not in cache:
            cache[k] = _draw_block(dist, seed, tag, k, ROW_BLOCK, cols)
        out[i] = cache[k][int(t) - k * ROW_BLOCK]
    return out


def outlier_channels(wl: Workload) -> np.ndarray:
    """Sorted indices of the channels of x that carry the outlier scale."""
    n = int(round(wl.outlier_frac * wl.hidden))
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    perm = _rng(wl.seed, TAG_OUTLIER, 0).permutation(wl.hidden)
    return np.sort(perm[:n]).astype(np.int64)


# ----------------------------------------------------------------------------
# storage rounding (library conversion, not part of the method)


def to_storage(a: np.ndarray, dtype: str):
    """float32 numpy array -> torch CPU tensor of the storage dtype."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    if dtype == "f32":
        return t
    if dtype == "bf16":
        return t.to(torch.bfloat16)
    if dtype == "f16":
        return t.to(torch.float16)
    raise ValueError(dtype)


def make_inputs(wl: Workload, rows=None) -> dict:
    """Seeded inputs of ``wl`` as torch CPU tensors in their storage dtype.

    ``rows`` (optional: an index array or a ``range``) restricts x and
    residual to those token indices; the values are the ones the full tensors
    hold at those rows.
    Returns keys ``x``, ``residual`` (or None), ``weight`` (or None),
    ``bias`` (or None).
    """
    T, H = wl.n_tokens, wl.hidden
    x = _draw_rows(wl.x_dist, wl.seed, TAG_X, T, H, rows)
    cols = outlier_channels(wl)
    if cols.size:
        x[:, cols] *= np.float32(wl.outlier_scale)
    r = None
    if wl.has_residual:
        r = _draw_rows("normal", wl.seed, TAG_R, T, H, rows)
        if wl.r_std != 1.0:
            r *= np.float32(wl.r_std)
    w = None
    if wl.has_weight:
        w = 1.0 + 0.1 * _rng(wl.seed, TAG_W, 0).standard_normal(H, dtype=np.float32)
    b = None
    if wl.has_bias:
        b = 0.01 * _rng(wl.seed, TAG_B, 0).standard_normal(H, dtype=np.float32)
    return {
        "x": to_storage(x, wl.in_dtype),
        "residual": None if r is None else to_storage(r, wl.res_storage),
        "weight": None if w is None else to_storage(w.astype(np.float32), wl.in_dtype),
        "bias": None if b is None else to_storage(b.astype(np.float32), wl.in_dtype),
    }


def sample_rows(n_tokens: int, n: int, seed: int = 12345) -> np.ndarray:
    """Sorted distinct row indices: the first, the last and n-2 seeded others."""
    if n >= n_tokens:
        return np.arange(n_tokens, dtype=np.int64)
    g = np.random.default_rng(seed)
    mid = g.choice(np.arange(1, n_tokens - 1), size=max(0, n - 2), replace=False)
    return np.unique(np.concatenate([[0, n_tokens - 1], mid]).astype(np.int64))


def qk_inputs(n_tokens: int, n_q_heads: int, n_k_heads: int, head_dim: int, dtype: str = "bf16",
              seed: int = 60, pad: int = 0) -> dict:
    """Seeded QK-norm inputs: a fused qkv matrix [T, (Hq + 2 Hk) * D + pad]
    ~ N(0,1) (query heads first, then key, then value heads), and query / key
    weights 1 + 0.1 N(0,1) of length D.  Returned as torch CPU tensors."""
    width = (n_q_heads + 2 * n_k_heads) * head_dim + pad
    qkv = _draw_range("normal", seed, TAG_X, 0, n_tokens, width)
    g = _rng(seed, TAG_W, 0)
    wq = (1.0 + 0.1 * g.standard_normal(head_dim, dtype=np.float32)).astype(np.float32)
    wk = (1.0 + 0.1 * g.standard_normal(head_dim, dtype=np.float32)).astype(np.float32)
    return {"qkv": to_storage(qkv, dtype), "q_weight": to_storage(wq, dtype),
            "k_weight": to_storage(wk, dtype)}
