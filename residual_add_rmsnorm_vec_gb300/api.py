"""Tensor-level entry point over the C ABI (marshalling only).

``fused_add_rmsnorm`` takes CUDA tensors, allocates the outputs that are not
given with torch, and calls ``rmsnorm_fwd_ex`` on the current torch stream.
Nothing here computes: a failed call raises ``RmsnError``.
"""
from __future__ import annotations

import torch

from . import _lib

_IN = {torch.float32: _lib.RMSN_IN_F32, torch.bfloat16: _lib.RMSN_IN_BF16,
       torch.float16: _lib.RMSN_IN_F16}
_OUT = {"f32": (_lib.RMSN_OUT_F32, torch.float32), "bf16": (_lib.RMSN_OUT_BF16, torch.bfloat16),
        "fp8": (_lib.RMSN_OUT_FP8E4M3, torch.uint8), "f16": (_lib.RMSN_OUT_F16, torch.float16)}
_DT_NAME = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}


def make_flags(in_dtype: str, out_dtype: str, residual: bool, weight: bool, bias: bool,
               pdl: bool = False, early_params: bool = False) -> int:
    f = {"f32": _lib.RMSN_IN_F32, "bf16": _lib.RMSN_IN_BF16, "f16": _lib.RMSN_IN_F16}[in_dtype]
    if pdl:
        f |= _lib.RMSN_PDL
    if early_params:
        f |= _lib.RMSN_PDL_EARLY_PARAMS
    f |= _OUT[out_dtype][0]
    if residual:
        f |= _lib.RMSN_HAS_RESIDUAL
    if weight:
        f |= _lib.RMSN_HAS_WEIGHT
    if bias:
        f |= _lib.RMSN_HAS_BIAS
    return f


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check(name, t, shape, dtypes, device=None):
    """A tensor the kernels will index as `shape`: anything else is refused
    here, before a launch could read or write past it."""
    if t is None:
        return
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must be one of {[str(d) for d in dtypes]}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def check_row_args(x, residual, weight, bias, out, residual_out, out_scale, out_dtype,
                   device=None):
    """Shapes, dtypes, devices and layout of the row norm's tensors.

    x is [T, H] bf16 / fp16 / fp32; the residual and residual_out are [T, H]
    of x's dtype, or both fp32 over bf16 / fp16 x (an fp32 residual stream);
    weight and bias are [H] of x's dtype; out is [T, H] of the output dtype
    (uint8 codes for FP8); out_scale is [T] fp32.  ``device``: where every
    tensor must live (None: anywhere, as for the host-memory entry)."""
    if x.dim() != 2:
        raise ValueError("x must be [n_tokens, hidden]")
    if x.dtype not in _IN:
        raise TypeError(f"unsupported input dtype {x.dtype}")
    T, H = x.shape
    _check("x", x, (T, H), (x.dtype,), device)
    res_dtypes = (x.dtype,) if x.dtype == torch.float32 else (x.dtype, torch.float32)
    _check("residual", residual, (T, H), res_dtypes, device)
    if residual_out is not None and residual is None:
        raise ValueError("residual_out needs a residual")
    if residual is not None:
        _check("residual_out", residual_out, (T, H), (residual.dtype,), device)
    _check("weight", weight, (H,), (x.dtype,), device)
    _check("bias", bias, (H,), (x.dtype,), device)
    _check("out", out, (T, H), (_OUT[out_dtype][1],), device)
    if out_scale is not None and out_dtype != "fp8":
        raise ValueError("out_scale is only written for the fp8 output")
    _check("out_scale", out_scale, (T,), (torch.float32,), device)


def fused_add_rmsnorm(x: torch.Tensor, residual: torch.Tensor | None = None,
                      weight: torch.Tensor | None = None, bias: torch.Tensor | None = None, *,
                      eps: float, out_dtype: str | None = None, weight_offset: float = 0.0,
                      out: torch.Tensor | None = None, residual_out: torch.Tensor | None = None,
                      out_scale: torch.Tensor | None = None, config: _lib.RmsnConfig | None = None,
                      stream: torch.cuda.Stream | None = None, pdl: bool = False,
                      early_params: bool = False):
    """Fused residual-add + RMSNorm of x[T, H] on the GPU.

    Returns ``(out, residual_out, out_scale)``; ``residual_out`` is None
    without a residual, ``out_scale`` is None unless ``out_dtype == "fp8"``
    (``out`` then holds E4M3 codes as uint8).  Tensors must be contiguous and
    on the same CUDA device; weight and bias are [H] of x's dtype.  ``pdl``
    launches with programmatic dependent launch (``early_params``: weight and
    bias are not written by the preceding kernel).
    """
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor (host rows: fused_add_rmsnorm_host)")
    out_dtype = out_dtype or _DT_NAME.get(x.dtype, "")
    if out_dtype not in _OUT:
        raise ValueError(f"unsupported output dtype {out_dtype!r}")
    check_row_args(x, residual, weight, bias, out, residual_out, out_scale, out_dtype, x.device)
    T, H = x.shape
    in_name = _DT_NAME[x.dtype]
    out_flag, out_torch = _OUT[out_dtype]
    if out is None:
        out = torch.empty((T, H), dtype=out_torch, device=x.device)
    # an fp32 residual under bf16 / fp16 activations is an fp32 residual stream
    res_f32 = residual is not None and residual.dtype == torch.float32 and x.dtype != torch.float32
    if residual is not None and residual_out is None:
        residual_out = torch.empty_like(residual)
    if out_dtype == "fp8" and out_scale is None:
        out_scale = torch.empty((T,), dtype=torch.float32, device=x.device)
    flags = make_flags(in_name, out_dtype, residual is not None, weight is not None,
                       bias is not None, pdl, early_params)
    if res_f32:
        flags |= _lib.RMSN_RESIDUAL_F32
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    st = _lib.rmsnorm_fwd_ex(_ptr(x), _ptr(residual), _ptr(weight), _ptr(bias),
                             _ptr(out), _ptr(residual_out), _ptr(out_scale), T, H, eps, flags,
                             weight_offset, config, s.cuda_stream)
    if st != _lib.RMSN_OK:
        raise _lib.RmsnError(st, "rmsnorm_fwd_ex")
    return out, residual_out, (out_scale if out_dtype == "fp8" else None)


def fused_add_rmsnorm_host(x: torch.Tensor, residual: torch.Tensor | None = None,
                           weight: torch.Tensor | None = None, bias: torch.Tensor | None = None, *,
                           eps: float, out_dtype: str | None = None, weight_offset: float = 0.0,
                           out: torch.Tensor | None = None,
                           residual_out: torch.Tensor | None = None,
                           out_scale: torch.Tensor | None = None, device: int | None = None,
                           stream: torch.cuda.Stream | None = None):
    """Fused residual-add + RMSNorm on tensors in host memory (``rmsnorm_fwd_host``).

    The GPU reads the rows straight from host memory and writes the results
    back there.  Inputs should be page-locked (``pin_memory()``); outputs
    that are not given are allocated page-locked.  Returns
    ``(out, residual_out, out_scale)`` like ``fused_add_rmsnorm``; the call is
    asynchronous, so synchronise ``stream`` before reading them.
    """
    out_dtype = out_dtype or _DT_NAME.get(x.dtype, "")
    if out_dtype not in _OUT:
        raise ValueError(f"unsupported output dtype {out_dtype!r}")
    check_row_args(x, residual, weight, bias, out, residual_out, out_scale, out_dtype)
    T, H = x.shape
    in_name = _DT_NAME[x.dtype]
    _, out_torch = _OUT[out_dtype]
    if out is None:
        out = torch.empty((T, H), dtype=out_torch, pin_memory=True)
    if residual is not None and residual_out is None:
        residual_out = torch.empty((T, H), dtype=residual.dtype, pin_memory=True)
    if out_dtype == "fp8" and out_scale is None:
        out_scale = torch.empty((T,), dtype=torch.float32, pin_memory=True)
    flags = make_flags(in_name, out_dtype, residual is not None, weight is not None,
                       bias is not None)
    if residual is not None and residual.dtype == torch.float32 and x.dtype != torch.float32:
        flags |= _lib.RMSN_RESIDUAL_F32
    dev = torch.cuda.current_device() if device is None else device
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        st = _lib.rmsnorm_fwd_host(_ptr(x), _ptr(residual), _ptr(weight), _ptr(bias), _ptr(out),
                                   _ptr(residual_out), _ptr(out_scale), T, H, eps, flags,
                                   weight_offset, s.cuda_stream)
    if st != _lib.RMSN_OK:
        raise _lib.RmsnError(st, "rmsnorm_fwd_host")
    return out, residual_out, (out_scale if out_dtype == "fp8" else None)


def qk_norm_(q: torch.Tensor | None, k: torch.Tensor | None, q_weight: torch.Tensor | None = None,
             k_weight: torch.Tensor | None = None, *, head_dim: int, eps: float,
             weight_offset: float = 0.0, stream: torch.cuda.Stream | None = None,
             pdl: bool = False, variant: str | None = None):
    """Per-head QK norm of q and k IN PLACE (``rmsnorm_qk_fwd``).

    q is [T, Hq * head_dim] or [T, Hq, head_dim], or a column slice of a
    fused qkv matrix (its row stride is used as the token stride); likewise
    k.  Either may be None.  ``variant``: None (the library's choice), "ring"
    or "direct" (force one kernel; for tests and tuning).  Returns (q, k).
    """
    def view2d(t):
        if t is None:
            return None, 0, 0
        if t.dim() == 3:
            t2 = t.reshape(t.shape[0], -1) if t.is_contiguous() else None
            if t2 is None:
                raise ValueError("3-D q/k must be contiguous")
            return t2, t2.shape[1] // head_dim, t2.stride(0)
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("q/k must be [T, heads*head_dim] with unit column stride")
        return t, t.shape[1] // head_dim, t.stride(0)

    if head_dim < 1:
        raise ValueError("head_dim must be positive")
    for name, t in (("q", q), ("k", k)):
        if t is None:
            continue
        if (t.shape[-1] != head_dim) if t.dim() == 3 else (t.shape[-1] % head_dim != 0):
            raise ValueError(f"{name}: rows must hold whole heads of head_dim elements")
    q2, hq, qs = view2d(q)
    k2, hk, ks = view2d(k)
    ref = q2 if q2 is not None else k2
    if ref is None:
        return q, k
    if q2 is not None and k2 is not None:
        if q2.shape[0] != k2.shape[0]:
            raise ValueError("q and k need the same number of tokens")
        if q2.dtype != k2.dtype or q2.device != k2.device:
            raise TypeError("q and k need the same dtype and device")
    if ref.dtype not in _IN:
        raise TypeError(f"unsupported dtype {ref.dtype}")
    if not ref.is_cuda:
        raise ValueError("q / k must be CUDA tensors")
    _check("q_weight", q_weight, (head_dim,), (ref.dtype,), ref.device)
    _check("k_weight", k_weight, (head_dim,), (ref.dtype,), ref.device)
    flags = _IN[ref.dtype] | (_lib.RMSN_PDL if pdl else 0)
    flags |= {None: 0, "ring": _lib.RMSN_QK_RING, "direct": _lib.RMSN_QK_DIRECT}[variant]
    s = stream if stream is not None else torch.cuda.current_stream(ref.device)
    st = _lib.rmsnorm_qk_fwd(_ptr(q2), _ptr(k2), _ptr(q_weight), _ptr(k_weight), ref.shape[0],
                             hq, hk, head_dim, qs, ks, eps, weight_offset, flags, s.cuda_stream)
    if st != _lib.RMSN_OK:
        raise _lib.RmsnError(st, "rmsnorm_qk_fwd")
    return q, k


def fused_add_rmsnorm_blockscaled(x: torch.Tensor, residual: torch.Tensor | None = None,
                                  weight: torch.Tensor | None = None,
                                  bias: torch.Tensor | None = None, *, eps: float, fmt: str,
                                  weight_offset: float = 0.0,
                                  residual_out: torch.Tensor | None = None,
                                  config: _lib.RmsnConfig | None = None,
                                  stream: torch.cuda.Stream | None = None, pdl: bool = False):
    """Fused residual-add + RMSNorm with an MXFP8 / MXFP4 / NVFP4 output
    (``rmsnorm_fwd_blockscaled``).  Returns ``(q, block_scale, token_scale,
    residual_out)``: q uint8 [T, H] (MXFP8) or [T, H / 2] (FP4, two codes per
    byte, low nibble first), block_scale uint8 [T, H / block], token_scale
    float32 [T] for NVFP4 (else None).  ``pdl``: launch with programmatic
    dependent launch."""
    if x.dim() != 2 or x.dtype != torch.bfloat16:
        raise TypeError("x must be a 2-D bfloat16 tensor")
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    if fmt not in _lib.BLOCK_FORMATS:
        raise ValueError(f"unknown block format {fmt!r}")
    T, H = x.shape
    bf16 = (torch.bfloat16,)
    _check("x", x, (T, H), bf16, x.device)
    _check("residual", residual, (T, H), bf16, x.device)
    if residual_out is not None and residual is None:
        raise ValueError("residual_out needs a residual")
    _check("residual_out", residual_out, (T, H), bf16, x.device)
    _check("weight", weight, (H,), bf16, x.device)
    _check("bias", bias, (H,), bf16, x.device)
    code, block, per_byte = _lib.BLOCK_FORMATS[fmt]
    q = torch.empty((T, H // per_byte), dtype=torch.uint8, device=x.device)
    bs = torch.empty((T, H // block), dtype=torch.uint8, device=x.device)
    ts = torch.empty((T,), dtype=torch.float32, device=x.device) if fmt == "nvfp4" else None
    if residual is not None and residual_out is None:
        residual_out = torch.empty_like(x)
    flags = make_flags("bf16", "f32", residual is not None, weight is not None, bias is not None,
                       pdl)
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    st = _lib.rmsnorm_fwd_blockscaled(_ptr(x), _ptr(residual), _ptr(weight), _ptr(bias), _ptr(q),
                                      _ptr(bs), _ptr(ts), _ptr(residual_out), T, H, eps, flags,
                                      code, weight_offset, config, s.cuda_stream)
    if st != _lib.RMSN_OK:
        raise _lib.RmsnError(st, "rmsnorm_fwd_blockscaled")
    return q, bs, ts, residual_out


def block_format_configs(n_tokens: int, hidden: int, fmt: str, residual: bool = True,
                         bias: bool = True) -> list:
    """Launch configurations a block-scaled output can be forced to: the
    vector kernels listed for the per-token FP8 output of the same shape
    (the block formats are built on the same launch shapes), less the
    element-wise kernels and, for the MX formats, the two-row pipelined ring
    (built for per-token FP8 and NVFP4 only)."""
    if fmt not in _lib.BLOCK_FORMATS:
        raise ValueError(f"unknown block format {fmt!r}")
    flags = make_flags("bf16", "fp8", residual, True, bias)
    skip = {_lib.VARIANT_GENERIC, _lib.VARIANT_RAGGED}
    if fmt != "nvfp4":
        skip.add(_lib.VARIANT_BULK_PIPE)
    return [c for c in _lib.rmsnorm_list_configs(n_tokens, hidden, flags) if c.variant not in skip]
