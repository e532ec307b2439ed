"""CPU oracle for the fused residual-add + RMSNorm -- TEST INFRASTRUCTURE.

A plain fp64 C implementation (``rmsnorm_oracle.c``) of what the hot path
computes, wrapped with ctypes.  Only the tests, ``__graft_entry__.smoke()``
and the bench's CPU-baseline / reference arm may import this package; the
library's compute path never does, and this package imports nothing from the
library.

The norm follows the blog "CuTeDSL at Perplexity", section "QK norm"
(regular RMS norm, reciprocal square root of the mean square plus EPS, times
the weight plus the scalar WEIGHT_BIAS), fused with the residual add, an
optional per-channel bias and an optional per-token FP8-e4m3 absmax output
(section "Blackwell support").  See the C file's header for the exact steps.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "rmsnorm_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "liboracle_rmsnorm.so")

F32, BF16, FP8E4M3, F64, F16 = 0, 1, 2, 3, 4
MXFP8, MXFP4, NVFP4 = 10, 11, 12
_BLOCK = {"mxfp8": (MXFP8, 32, 1), "mxfp4": (MXFP4, 32, 2), "nvfp4": (NVFP4, 16, 2)}
_DTYPES = {"f32": F32, "bf16": BF16, "fp8": FP8E4M3, "f64": F64, "f16": F16}

_lock = threading.Lock()
_default = None


def build(force: bool = False, src: str = SRC, out: str = LIB) -> str:
    """Compile the oracle with gcc (portable flags, no FMA contraction)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fPIC",
           "-shared", "-pthread", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        lib.oracle_rmsnorm.restype = ctypes.c_int
        lib.oracle_rmsnorm.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64,
                                       ctypes.c_double, ctypes.c_double,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_rmsnorm_res.restype = ctypes.c_int
        lib.oracle_rmsnorm_res.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64,
                                           ctypes.c_double, ctypes.c_double,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_bf16_from_f64.restype = ctypes.c_uint16
        lib.oracle_bf16_from_f64.argtypes = [ctypes.c_double]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_e4m3_from_f64.restype = ctypes.c_uint8
        lib.oracle_e4m3_from_f64.argtypes = [ctypes.c_double]
        lib.oracle_e4m3_to_f64.restype = ctypes.c_double
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_num_cpus.restype = ctypes.c_int
        lib.oracle_f16_from_f64.restype = ctypes.c_uint16
        lib.oracle_f16_from_f64.argtypes = [ctypes.c_double]
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_e2m1_to_f64.restype = ctypes.c_double
        lib.oracle_e2m1_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_from_f64.restype = ctypes.c_uint8
        lib.oracle_e2m1_from_f64.argtypes = [ctypes.c_double]
        lib.oracle_e8m0_to_f64.restype = ctypes.c_double
        lib.oracle_e8m0_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_block_quantize.restype = ctypes.c_int
        lib.oracle_block_quantize.argtypes = [vp, i64, i64, ctypes.c_int, vp, vp, vp]
        lib.oracle_qk_norm.restype = ctypes.c_int
        lib.oracle_qk_norm.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                       ctypes.c_double, ctypes.c_double, ctypes.c_int]
        self.lib = lib
        self.path = path

    def num_cpus(self) -> int:
        return int(self.lib.oracle_num_cpus())

    def bf16_from_f64(self, v: float) -> int:
        return int(self.lib.oracle_bf16_from_f64(float(v)))

    def bf16_to_f64(self, b: int) -> float:
        return float(self.lib.oracle_bf16_to_f64(int(b)))

    def e4m3_from_f64(self, v: float) -> int:
        return int(self.lib.oracle_e4m3_from_f64(float(v)))

    def e4m3_to_f64(self, c: int) -> float:
        return float(self.lib.oracle_e4m3_to_f64(int(c)))

    def f16_from_f64(self, v: float) -> int:
        return int(self.lib.oracle_f16_from_f64(float(v)))

    def f16_to_f64(self, h: int) -> float:
        return float(self.lib.oracle_f16_to_f64(int(h)))

    def e2m1_from_f64(self, v: float) -> int:
        return int(self.lib.oracle_e2m1_from_f64(float(v)))

    def e2m1_to_f64(self, c: int) -> float:
        return float(self.lib.oracle_e2m1_to_f64(int(c)))

    def e8m0_to_f64(self, c: int) -> float:
        return float(self.lib.oracle_e8m0_to_f64(int(c)))

    def block_quantize(self, y64: np.ndarray, fmt: str) -> dict:
        """Block-scaled quantisation of fp64 rows [T, H] (see the C file):
        returns ``q`` (bytes; FP4 packed two per byte), ``block_scale`` and,
        for NVFP4, ``token_scale``."""
        code, blk, per_byte = _BLOCK[fmt]
        y = np.ascontiguousarray(y64, dtype=np.float64)
        T, H = y.shape
        q = np.zeros((T, H // per_byte), dtype=np.uint8)
        bs = np.zeros((T, H // blk), dtype=np.uint8)
        ts = np.zeros(T, dtype=np.float32) if fmt == "nvfp4" else None
        st = self.lib.oracle_block_quantize(y.ctypes.data, T, H, code, q.ctypes.data,
                                            bs.ctypes.data, None if ts is None else ts.ctypes.data)
        if st != 0:
            raise RuntimeError(f"oracle_block_quantize failed with status {st}")
        return {"q": q, "block_scale": bs, "token_scale": ts}

    def rmsnorm_block(self, x, residual=None, weight=None, bias=None, *, eps: float,
                      in_dtype: str, fmt: str, weight_offset: float = 0.0) -> dict:
        """The norm (fp64 output) followed by the block-scaled quantisation."""
        o = self.rmsnorm(x, residual, weight, bias, eps=eps, in_dtype=in_dtype, out_dtype="f64",
                         weight_offset=weight_offset)
        b = self.block_quantize(o["out"], fmt)
        b["residual_out"] = o["residual_out"]
        b["y64"] = o["out"]
        return b

    def qk_norm(self, q, k, q_weight=None, k_weight=None, *, n_q_heads: int, n_k_heads: int,
                head_dim: int, eps: float, dtype: str, weight_offset: float = 0.0):
        """Per-head norm of q [T, q_stride] and k [T, k_stride] (copies are
        returned; the inputs are not modified).  Row t of q holds its n_q_heads
        heads of head_dim elements at the start of the row."""
        qb = None if q is None else _host_bits(q, dtype).copy()
        kb = None if k is None else _host_bits(k, dtype).copy()
        T = (qb if qb is not None else kb).shape[0]
        qs = qb.shape[1] if qb is not None else 0
        ks = kb.shape[1] if kb is not None else 0
        wq = None if q_weight is None else _host_bits(q_weight, dtype)
        wk = None if k_weight is None else _host_bits(k_weight, dtype)

        def ptr(a):
            return None if a is None else a.ctypes.data

        st = self.lib.oracle_qk_norm(ptr(qb), ptr(kb), ptr(wq), ptr(wk), T, n_q_heads,
                                     n_k_heads, head_dim, qs, ks, float(eps),
                                     float(weight_offset), _DTYPES[dtype])
        if st != 0:
            raise RuntimeError(f"oracle_qk_norm failed with status {st}")
        return qb, kb

    def rmsnorm(self, x, residual=None, weight=None, bias=None, *, eps: float,
                in_dtype: str, out_dtype: str, weight_offset: float = 0.0,
                n_threads: int = 0, residual_dtype: str | None = None) -> dict:
        return _rmsnorm(self.lib, x, residual, weight, bias, eps=eps, in_dtype=in_dtype,
                        out_dtype=out_dtype, weight_offset=weight_offset,
                        n_threads=n_threads, residual_dtype=residual_dtype)


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def num_cpus() -> int:
    return default().num_cpus()


def bf16_from_f64(v: float) -> int:
    return default().bf16_from_f64(v)


def bf16_to_f64(b: int) -> float:
    return default().bf16_to_f64(b)


def e4m3_from_f64(v: float) -> int:
    return default().e4m3_from_f64(v)


def e4m3_to_f64(c: int) -> float:
    return default().e4m3_to_f64(c)


def _host_bits(a, dtype: str) -> np.ndarray:
    """Contiguous numpy view of the raw storage bits of a CPU tensor/array."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if dtype in ("bf16", "f16"):
                return a.view(torch.int16).numpy().view(np.uint16)
            return a.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if dtype in ("bf16", "f16"):
        return a.view(np.uint16)
    return a.astype(np.float32, copy=False)


def rmsnorm(x, residual=None, weight=None, bias=None, *, eps: float, in_dtype: str,
            out_dtype: str, weight_offset: float = 0.0, n_threads: int = 0,
            residual_dtype: str | None = None) -> dict:
    """Run the oracle on CPU inputs; see ``_rmsnorm``."""
    return default().rmsnorm(x, residual, weight, bias, eps=eps, in_dtype=in_dtype,
                             out_dtype=out_dtype, weight_offset=weight_offset,
                             n_threads=n_threads, residual_dtype=residual_dtype)


def _rmsnorm(lib, x, residual=None, weight=None, bias=None, *, eps: float, in_dtype: str,
             out_dtype: str, weight_offset: float = 0.0, n_threads: int = 0,
             residual_dtype: str | None = None) -> dict:
    """Run the oracle on CPU inputs ([T, H] x / residual, [H] weight / bias).

    Inputs are torch CPU tensors or numpy arrays of the storage dtype
    (bf16 given as uint16 bits when numpy).  Returns numpy arrays:
    ``out`` (float32 for f32, uint16 bits for bf16 / f16, uint8 codes for fp8,
    float64 for f64), ``residual_out`` (storage of the residual, which is the
    input dtype unless ``residual_dtype`` says otherwise; or None)
    and ``out_scale`` (float32 [T], fp8 only).
    """
    xb = _host_bits(x, in_dtype)
    if xb.ndim != 2:
        raise ValueError("x must be [T, H]")
    T, H = xb.shape
    res_dt = residual_dtype or in_dtype
    rb = None if residual is None else _host_bits(residual, res_dt)
    wb = None if weight is None else _host_bits(weight, in_dtype)
    bb = None if bias is None else _host_bits(bias, in_dtype)
    out_np = {"f32": np.float32, "bf16": np.uint16, "fp8": np.uint8, "f64": np.float64,
              "f16": np.uint16}[out_dtype]
    out = np.empty((T, H), dtype=out_np)
    res_out = None if rb is None else np.empty_like(rb)
    scale = np.empty(T, dtype=np.float32) if out_dtype == "fp8" else None

    def ptr(a):
        return None if a is None else a.ctypes.data

    st = lib.oracle_rmsnorm_res(ptr(xb), ptr(rb), ptr(wb), ptr(bb), ptr(out), ptr(res_out),
                                ptr(scale), T, H, float(eps), float(weight_offset),
                                _DTYPES[in_dtype], _DTYPES[res_dt], _DTYPES[out_dtype],
                                int(n_threads))
    if st != 0:
        raise RuntimeError(f"oracle_rmsnorm failed with status {st}")
    return {"out": out, "residual_out": res_out, "out_scale": scale}


def qk_norm(q, k, q_weight=None, k_weight=None, **kw):
    """Per-head QK norm on CPU copies; see ``Oracle.qk_norm``."""
    return default().qk_norm(q, k, q_weight, k_weight, **kw)


def rmsnorm_block(x, residual=None, weight=None, bias=None, **kw):
    """Norm + block-scaled quantisation on CPU; see ``Oracle.rmsnorm_block``."""
    return default().rmsnorm_block(x, residual, weight, bias, **kw)
