"""ctypes binding of the C ABI in include/rmsnorm.h (argument marshalling only).

The shared library must have been built (``residual_add_rmsnorm_vec_gb300.build``
or ``__graft_entry__.build()``); a missing library raises instead of falling
back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH as _DEFAULT_LIB

# RMSNORM_GB300_LIB names another build of the library to load instead (the
# bounds-checked debug build, for instance); by default the in-tree one.
LIB_PATH = os.environ.get("RMSNORM_GB300_LIB") or _DEFAULT_LIB

RMSN_OK = 0
RMSN_EINVAL = -1
RMSN_EALIGN = -2
RMSN_EUNSUPPORTED = -3
RMSN_ECUDA = -4

RMSN_IN_F32 = 0x0
RMSN_IN_BF16 = 0x1
RMSN_IN_F16 = 0x2
RMSN_OUT_F32 = 0x0
RMSN_OUT_BF16 = 0x4
RMSN_OUT_FP8E4M3 = 0x8
RMSN_OUT_F16 = 0xC
RMSN_HAS_RESIDUAL = 0x10
RMSN_HAS_WEIGHT = 0x20
RMSN_HAS_BIAS = 0x40
RMSN_PDL = 0x80
RMSN_RESIDUAL_F32 = 0x200
RMSN_PDL_EARLY_PARAMS = 0x100
RMSN_QK_RING = 0x400
RMSN_QK_DIRECT = 0x800

VARIANT_WARP_ROWS = 0
VARIANT_BLOCK_ROW = 1
VARIANT_BULK_ROW = 2
VARIANT_GENERIC = 3
VARIANT_RAGGED = 4
VARIANT_CLUSTER = 5
VARIANT_BULK_PIPE = 6
VARIANT_NAMES = {0: "warp_rows", 1: "block_row", 2: "bulk_row", 3: "generic", 4: "ragged",
                 5: "cluster", 6: "bulk_pipe"}

RMSN_FMT_MXFP8 = 1
RMSN_FMT_MXFP4 = 2
RMSN_FMT_NVFP4 = 3
BLOCK_FORMATS = {"mxfp8": (RMSN_FMT_MXFP8, 32, 1), "mxfp4": (RMSN_FMT_MXFP4, 32, 2),
                 "nvfp4": (RMSN_FMT_NVFP4, 16, 2)}

EXPORTED = ("rmsnorm_fwd", "rmsnorm_fwd_ex", "rmsnorm_fwd_blockscaled", "rmsnorm_fwd_host",
            "rmsnorm_qk_fwd",
            "rmsnorm_query_config", "rmsnorm_list_configs", "rmsnorm_read_status",
            "rmsnorm_set_wait_limit", "rmsnorm_status_string")


class RmsnConfig(ctypes.Structure):
    """Mirror of ``rmsn_config``."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "variant", "vec_bytes", "warps_per_block", "warps_per_row", "chunks", "max_warps",
        "stages", "grid", "smem_bytes", "num_sms", "ring_copy", "cluster")]

    def as_dict(self) -> dict:
        d = {n: int(getattr(self, n)) for n, _ in self._fields_}
        d["variant_name"] = VARIANT_NAMES.get(d["variant"], "?")
        return d

    @classmethod
    def from_dict(cls, d: dict) -> "RmsnConfig":
        c = cls()
        for n, _ in cls._fields_:
            if n in d:
                setattr(c, n, int(d[n]))
        return c


class RmsnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return LIB_PATH


def load() -> ctypes.CDLL:
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"the CUDA library {LIB_PATH} is not built; run "
                    "residual_add_rmsnorm_vec_gb300.build.build() first")
            lib = ctypes.CDLL(LIB_PATH)
            vp, i64, u32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint32, ctypes.c_float
            lib.rmsnorm_fwd.restype = ctypes.c_int
            lib.rmsnorm_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, f32, u32, vp]
            lib.rmsnorm_fwd_ex.restype = ctypes.c_int
            lib.rmsnorm_fwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, f32, u32, f32,
                                           ctypes.POINTER(RmsnConfig), vp]
            lib.rmsnorm_fwd_blockscaled.restype = ctypes.c_int
            lib.rmsnorm_fwd_blockscaled.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, f32,
                                                    u32, ctypes.c_int, f32,
                                                    ctypes.POINTER(RmsnConfig), vp]
            lib.rmsnorm_fwd_host.restype = ctypes.c_int
            lib.rmsnorm_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, f32, u32, f32,
                                             vp]
            lib.rmsnorm_qk_fwd.restype = ctypes.c_int
            lib.rmsnorm_qk_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, f32,
                                           u32, vp]
            lib.rmsnorm_query_config.restype = ctypes.c_int
            lib.rmsnorm_query_config.argtypes = [i64, i64, u32, ctypes.POINTER(RmsnConfig)]
            lib.rmsnorm_list_configs.restype = ctypes.c_int
            lib.rmsnorm_list_configs.argtypes = [i64, i64, u32, ctypes.POINTER(RmsnConfig),
                                                 ctypes.c_int]
            lib.rmsnorm_read_status.restype = ctypes.c_int
            lib.rmsnorm_read_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
            lib.rmsnorm_set_wait_limit.restype = ctypes.c_int
            lib.rmsnorm_set_wait_limit.argtypes = [i64]
            lib.rmsnorm_status_string.restype = ctypes.c_char_p
            lib.rmsnorm_status_string.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().rmsnorm_status_string(int(status)).decode()


def rmsnorm_fwd(x, residual, weight, bias, out, residual_out, out_scale, n_tokens: int,
                hidden: int, eps: float, flags: int, stream) -> int:
    """Direct call of ``rmsnorm_fwd`` with raw pointers (ints or None)."""
    return int(load().rmsnorm_fwd(x, residual, weight, bias, out, residual_out, out_scale,
                                  int(n_tokens), int(hidden), float(eps), int(flags), stream))


def rmsnorm_fwd_ex(x, residual, weight, bias, out, residual_out, out_scale, n_tokens: int,
                   hidden: int, eps: float, flags: int, weight_offset: float,
                   cfg: RmsnConfig | None, stream) -> int:
    """Direct call of ``rmsnorm_fwd_ex`` with raw pointers (ints or None)."""
    return int(load().rmsnorm_fwd_ex(x, residual, weight, bias, out, residual_out, out_scale,
                                     int(n_tokens), int(hidden), float(eps), int(flags),
                                     float(weight_offset),
                                     None if cfg is None else ctypes.byref(cfg), stream))


def rmsnorm_fwd_blockscaled(x, residual, weight, bias, out, block_scale, token_scale,
                            residual_out, n_tokens: int, hidden: int, eps: float, flags: int,
                            fmt: int, weight_offset: float, cfg: RmsnConfig | None, stream) -> int:
    """Direct call of ``rmsnorm_fwd_blockscaled`` with raw pointers."""
    return int(load().rmsnorm_fwd_blockscaled(x, residual, weight, bias, out, block_scale,
                                              token_scale, residual_out, int(n_tokens),
                                              int(hidden), float(eps), int(flags), int(fmt),
                                              float(weight_offset),
                                              None if cfg is None else ctypes.byref(cfg),
                                              stream))


def rmsnorm_fwd_host(x, residual, weight, bias, out, residual_out, out_scale, n_tokens: int,
                     hidden: int, eps: float, flags: int, weight_offset: float, stream) -> int:
    """Direct call of ``rmsnorm_fwd_host`` (pointers may be host memory)."""
    return int(load().rmsnorm_fwd_host(x, residual, weight, bias, out, residual_out, out_scale,
                                       int(n_tokens), int(hidden), float(eps), int(flags),
                                       float(weight_offset), stream))


def rmsnorm_qk_fwd(q, k, q_weight, k_weight, n_tokens: int, n_q_heads: int, n_k_heads: int,
                   head_dim: int, q_token_stride: int, k_token_stride: int, eps: float,
                   weight_offset: float, flags: int, stream) -> int:
    """Direct call of ``rmsnorm_qk_fwd`` (in place on q and k)."""
    return int(load().rmsnorm_qk_fwd(q, k, q_weight, k_weight, int(n_tokens), int(n_q_heads),
                                     int(n_k_heads), int(head_dim), int(q_token_stride),
                                     int(k_token_stride), float(eps), float(weight_offset),
                                     int(flags), stream))


def rmsnorm_query_config(n_tokens: int, hidden: int, flags: int) -> RmsnConfig:
    c = RmsnConfig()
    st = load().rmsnorm_query_config(int(n_tokens), int(hidden), int(flags), ctypes.byref(c))
    if st != RMSN_OK:
        raise RmsnError(st, "rmsnorm_query_config")
    return c


def rmsnorm_list_configs(n_tokens: int, hidden: int, flags: int) -> list[RmsnConfig]:
    lib = load()
    n = lib.rmsnorm_list_configs(int(n_tokens), int(hidden), int(flags), None, 0)
    if n < 0:
        raise RmsnError(n, "rmsnorm_list_configs")
    arr = (RmsnConfig * max(1, n))()
    m = lib.rmsnorm_list_configs(int(n_tokens), int(hidden), int(flags), arr, n)
    if m < 0:
        raise RmsnError(m, "rmsnorm_list_configs")
    return [arr[i] for i in range(min(n, m))]


def rmsnorm_read_status(clear: bool = False) -> int:
    """Kernel status word of the current device (0 = no bounded wait ran out)."""
    v = ctypes.c_uint32(0)
    st = load().rmsnorm_read_status(ctypes.byref(v), int(bool(clear)))
    if st != RMSN_OK:
        raise RmsnError(st, "rmsnorm_read_status")
    return int(v.value)


def rmsnorm_set_wait_limit(cycles: int) -> int:
    """Testing hook: the bound of the bulk-copy kernel's row waits on the
    current device (0 = the default; negative = test each barrier once and
    do not wait)."""
    return int(load().rmsnorm_set_wait_limit(int(cycles)))
