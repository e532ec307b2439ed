"""Helpers for GPU-vs-oracle parity: run both sides on the same seeded inputs
and compare with the tolerances of the fused residual-add + RMSNorm:

* residual_out: bit-exact;
* bf16 / fp16 output: at most 1 ulp of the output type (signed-magnitude
  ordering, +0 == -0); with a bias, an element further off must be one
  where the bias cancels, |y| <= 2^-8 (|w*h*inv| + |b_j|) by the oracle's
  fp64 values, and lie within the fp32 bound below (there y can be far
  smaller than the fp32 rounding of w*h*inv, and so many of its own ulps
  away);
* fp32 output: relative error <= 1e-5, measured against |y| + |b_j| when a
  bias is present (the fp32 rounding of w*h*inv is carried into y even where
  the bias cancels it; without a bias this is the plain relative error);
* FP8-E4M3 output: same code or the adjacent one; per-token scale relative
  error <= 1e-6.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

BF16_ULP = 1
F32_RTOL = 1e-5
FP8_STEPS = 1
SCALE_RTOL = 1e-6


def ordered16(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def ordered8(codes: np.ndarray) -> np.ndarray:
    c = codes.astype(np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def to_device(inp: dict, dev) -> dict:
    return {k: (None if v is None else v.to(dev)) for k, v in inp.items()}


CANCEL = 2.0 ** -8  # |y| at most this fraction of |w h inv| + |b_j|: the bias cancels


def oracle_run(wl, inp: dict, weight_offset: float = 0.0) -> dict:
    kw = dict(eps=float(np.float32(wl.eps)), in_dtype=wl.in_dtype, weight_offset=weight_offset,
              residual_dtype=wl.res_storage)
    ref = oracle.rmsnorm(inp["x"], inp["residual"], inp["weight"], inp["bias"],
                         out_dtype=wl.out_dtype, **kw)
    if inp["bias"] is not None and wl.out_dtype in ("bf16", "f16"):
        # the unrounded y decides which elements may take the cancellation bound
        ref["y64"] = oracle.rmsnorm(inp["x"], inp["residual"], inp["weight"], inp["bias"],
                                    out_dtype="f64", **kw)["out"]
    return ref


def gpu_outputs_to_host(wl, out, res, scale) -> dict:
    if wl.out_dtype in ("bf16", "f16"):
        o = bits16(out)
    elif wl.out_dtype == "fp8":
        o = out.detach().cpu().numpy()
    else:
        o = out.detach().cpu().numpy()
    r = None
    if res is not None:
        r = bits16(res) if wl.res_storage in ("bf16", "f16") else res.detach().cpu().numpy()
    s = None if scale is None else scale.detach().cpu().numpy()
    return {"out": o, "residual_out": r, "out_scale": s}


def to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Values of bf16 / fp16 bit patterns."""
    t = torch.from_numpy(bits.astype(np.uint16).view(np.int16))
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16).double().numpy()


def compare(wl, got: dict, ref: dict, where: str = "", bias=None) -> dict:
    """Assert the tolerances; return statistics.  ``bias`` (CPU tensor [H])
    widens the fp32 bound to 1e-5 * (|y| + |b_j|)."""
    stats = {}
    if ref["residual_out"] is not None:
        g, r = got["residual_out"], ref["residual_out"]
        if wl.res_storage in ("bf16", "f16"):
            bad = np.count_nonzero(g != r)
        else:
            bad = np.count_nonzero(g.view(np.uint32) != r.view(np.uint32))
        assert bad == 0, f"{where}: residual_out differs in {bad} elements"
    if wl.out_dtype in ("bf16", "f16"):
        # 1 ulp of the output type (signed-magnitude order works for both)
        d = np.abs(ordered16(got["out"]) - ordered16(ref["out"]))
        stats["exact_frac"] = float((d == 0).mean()) if d.size else 1.0
        if bias is not None and d.size and d.max() > BF16_ULP:
            # only elements where the bias cancels may be further off: the
            # fp32 bound on |y| + |b_j| applies to them
            far = d > BF16_ULP
            assert "y64" in ref, f"{where}: the oracle's fp64 y is needed to decide cancellation"
            bs = np.broadcast_to(bias.double().numpy()[None, :], d.shape)[far]
            y64 = ref["y64"][far]
            cancels = np.abs(y64) <= CANCEL * (np.abs(y64 - bs) + np.abs(bs))
            assert cancels.all(), (f"{where}: {int((~cancels).sum())} elements more than "
                                   f"{BF16_ULP} ulp off where the bias does not cancel")
            g = to_f64(got["out"], wl.out_dtype)[far]
            r = to_f64(ref["out"], wl.out_dtype)[far]
            b = np.abs(bs)
            rel = np.abs(g - r) / np.maximum(np.abs(r) + b, np.finfo(np.float32).tiny)
            stats["cancelled"] = int(far.sum())
            stats["cancelled_max_rel"] = float(rel.max())
            assert stats["cancelled_max_rel"] <= F32_RTOL, \
                f"{where}: 16-bit output off by {int(d.max())} ulp, rel {rel.max()} of |y| + |b|"
            d = np.where(far, 0, d)
        stats["max_ulp"] = int(d.max()) if d.size else 0
        assert stats["max_ulp"] <= BF16_ULP, f"{where}: bf16 output off by {stats['max_ulp']} ulp"
    elif wl.out_dtype == "f32":
        g = got["out"].astype(np.float64)
        r = ref["out"].astype(np.float64)
        mag = np.abs(r)
        if bias is not None:
            mag = mag + np.abs(bias.double().numpy())[None, :]
        rel = np.abs(g - r) / np.maximum(mag, np.finfo(np.float32).tiny)
        stats["max_rel"] = float(rel.max()) if rel.size else 0.0
        assert stats["max_rel"] <= F32_RTOL, f"{where}: f32 output rel err {stats['max_rel']}"
    else:
        d = np.abs(ordered8(got["out"]) - ordered8(ref["out"]))
        stats["max_steps"] = int(d.max()) if d.size else 0
        stats["exact_frac"] = float((d == 0).mean()) if d.size else 1.0
        assert stats["max_steps"] <= FP8_STEPS, f"{where}: fp8 codes {stats['max_steps']} steps apart"
        gs = got["out_scale"].astype(np.float64)
        rs = ref["out_scale"].astype(np.float64)
        rel = np.where(rs == 0, np.abs(gs), np.abs(gs - rs) / np.where(rs == 0, 1, np.abs(rs)))
        stats["scale_max_rel"] = float(rel.max()) if rel.size else 0.0
        assert stats["scale_max_rel"] <= SCALE_RTOL, f"{where}: scale rel err {stats['scale_max_rel']}"
    return stats
