"""Pins for the CPU oracle: each test checks it against something other than
itself -- library conversions, the OCP FP8 format definition, hand-derived
closed forms (tests/golden), invariants of the RMS norm and exact-rational
brute force on tiny rows.  CPU only.

The norm is the regular RMS norm of the blog "CuTeDSL at Perplexity"
(section "QK norm"), fused with the residual add and an optional bias /
FP8-e4m3 per-token output (section "Blackwell support").
"""
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers


def bf16_tensor(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def exact_bf16_neighbours(v: Fraction):
    """The two consecutive bf16 values around v > 0 (brute force over codes)."""
    lo, hi = 0x0000, 0x7F80
    # binary search over positive finite codes: value(code) is increasing
    def val(c):
        return Fraction(float(bf16_bits_to_float(np.array([c], dtype=np.uint16))[0]))
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if val(mid) <= v:
            lo = mid
        else:
            hi = mid
    return lo, val(lo), hi, val(hi)


def exact_round_bf16(v: Fraction) -> int:
    """bf16 bits of v rounded to nearest, ties to the even code (v finite)."""
    neg = v < 0
    a = -v if neg else v
    if a == 0:
        return 0x8000 if neg else 0
    c0, v0, c1, v1 = exact_bf16_neighbours(a)
    d0, d1 = a - v0, v1 - a
    if d0 < d1 or (d0 == d1 and c0 % 2 == 0):
        c = c0
    else:
        c = c1
    return c | (0x8000 if neg else 0)


# ---------------------------------------------------------------- bf16 encoder


def test_bf16_encoder_matches_torch_on_random_f32(oracle_mod):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals)]
    ref = torch.from_numpy(vals.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle_mod.bf16_from_f64(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_encoder_ties_and_boundaries(oracle_mod):
    # every midpoint between consecutive bf16 values in a few binades, +-1 f32 ulp
    base = np.arange(0x3F00, 0x3F80, dtype=np.uint32)            # [0.5, 1)
    sub = np.arange(0x0000, 0x0080, dtype=np.uint32)             # subnormals
    top = np.arange(0x7F00, 0x7F7F, dtype=np.uint32)             # near max
    codes = np.concatenate([base, sub, top])
    mids = ((codes << 16) + 0x8000).astype(np.uint32)           # exact midpoints in f32
    cand = np.concatenate([mids, mids - 1, mids + 1]).view(np.float32)
    ref = torch.from_numpy(cand.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle_mod.bf16_from_f64(float(v)) for v in cand], dtype=np.uint16)
    assert np.array_equal(got, ref)
    # overflow to infinity exactly at max + half ulp, and signed zero
    maxf = float(bf16_bits_to_float(np.array([0x7F7F], dtype=np.uint16))[0])
    assert oracle_mod.bf16_from_f64(maxf) == 0x7F7F
    assert oracle_mod.bf16_from_f64(maxf + 2.0**119) == 0x7F80
    assert oracle_mod.bf16_from_f64(maxf + 2.0**119 - 2.0**90) == 0x7F7F
    assert oracle_mod.bf16_from_f64(-0.0) == 0x8000


def test_bf16_encoder_rounds_f64_once(oracle_mod):
    # values just off a midpoint by less than an f32 ulp: a double-rounding
    # encoder (f64 -> f32 -> bf16) gets these wrong; exact rational rounding decides
    rng = np.random.default_rng(11)
    for c in rng.integers(0x0100, 0x7F00, size=300):
        mid = float(bf16_bits_to_float(np.array([c], dtype=np.uint16))[0]) * (1 + 2.0**-8)
        for delta in (2.0**-40, -2.0**-40):
            v = mid * (1 + delta)
            assert oracle_mod.bf16_from_f64(v) == exact_round_bf16(Fraction(v))


# ---------------------------------------------------------------- f16 encoder


def _f16_value(h: int) -> Fraction:
    return Fraction(float(np.array([h], dtype=np.uint16).view(np.float16)[0]))


def exact_round_f16(v: Fraction) -> int:
    """binary16 bits of finite v rounded to nearest, ties to the even code."""
    neg = v < 0
    a = -v if neg else v
    if a == 0:
        return 0x8000 if neg else 0
    lo, hi = 0x0000, 0x7C00
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if _f16_value(mid) <= a:
            lo = mid
        else:
            hi = mid
    d0, d1 = a - _f16_value(lo), (_f16_value(hi) - a) if hi < 0x7C00 else None
    if hi == 0x7C00:  # beyond the largest finite: overflow threshold max + half ulp
        c = lo if a - _f16_value(0x7BFF) < Fraction(16) else 0x7C00
    elif d0 < d1 or (d0 == d1 and lo % 2 == 0):
        c = lo
    else:
        c = hi
    return c | (0x8000 if neg else 0)


def _check_f16_encoder(orc):
    rng = np.random.default_rng(60)
    bits = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals)]
    ref = torch.from_numpy(vals.copy()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.f16_from_f64(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)
    # every tie and its f32 neighbours in a normal and the subnormal binade, overflow edge
    codes = np.concatenate([np.arange(0x3800, 0x3C00), np.arange(0x0000, 0x0400)]).astype(np.uint16)
    f = codes.view(np.float16).astype(np.float32)
    nxt = (codes + 1).astype(np.uint16).view(np.float16).astype(np.float32)
    mids = ((f.astype(np.float64) + nxt) / 2).astype(np.float32)
    cand = np.concatenate([mids, np.nextafter(mids, 0), np.nextafter(mids, 1)])
    ref = torch.from_numpy(cand).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.f16_from_f64(float(v)) for v in cand], dtype=np.uint16)
    assert np.array_equal(got, ref)
    assert orc.f16_from_f64(65504.0) == 0x7BFF and orc.f16_from_f64(65519.99) == 0x7BFF
    assert orc.f16_from_f64(65520.0) == 0x7C00 and orc.f16_from_f64(-1e9) == 0xFC00
    for c in rng.integers(0x0400, 0x7B00, size=200):
        mid = float(_f16_value(int(c)) + _f16_value(int(c) + 1)) / 2
        for v in (mid * (1 + 2.0**-40), mid * (1 - 2.0**-40)):
            assert orc.f16_from_f64(v) == exact_round_f16(Fraction(v))


def test_f16_encoder(oracle_mod):
    _check_f16_encoder(oracle_mod.default())


def _check_f16_norm(orc):
    # residual: the f32 sum of two fp16 values rounded to fp16 (torch) equals
    # the exact sum rounded once; the fp16 output is the f64 output rounded
    rng = np.random.default_rng(61)
    x = torch.from_numpy(rng.standard_normal((8, 256)).astype(np.float32) * 30).to(torch.float16)
    r = torch.from_numpy(rng.standard_normal((8, 256)).astype(np.float32)).to(torch.float16)
    w = torch.from_numpy((1 + 0.1 * rng.standard_normal(256)).astype(np.float32)).to(torch.float16)
    o = orc.rmsnorm(x, r, w, None, eps=1e-6, in_dtype="f16", out_dtype="f16")
    ref_res = (x.float() + r.float()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(o["residual_out"], ref_res)
    y = orc.rmsnorm(x, r, w, None, eps=1e-6, in_dtype="f16", out_dtype="f64")["out"]
    for i in range(0, 8 * 256, 29):
        assert o["out"].flat[i] == exact_round_f16(Fraction(float(y.flat[i])))
    # the fp16 norm equals the fp32-input norm of the widened rounded residual
    h = torch.from_numpy(o["residual_out"].view(np.int16)).view(torch.float16).float()
    o_h = orc.rmsnorm(h, None, w.float(), None, eps=1e-6, in_dtype="f32", out_dtype="f64")["out"]
    assert np.array_equal(y, o_h)


def _check_f32_residual_stream(orc):
    # bf16 / fp16 activations with an fp32 residual stream: h is the fp32 sum
    # (torch's f32 add of the widened values, correctly rounded), not rounded
    # to the activation type, and the norm is taken on that h
    rng = np.random.default_rng(62)
    for dt, tdt in (("bf16", torch.bfloat16), ("f16", torch.float16)):
        x = torch.from_numpy(rng.standard_normal((6, 320)).astype(np.float32)).to(tdt)
        r = torch.from_numpy(rng.standard_normal((6, 320)).astype(np.float32) * 7)
        w = torch.from_numpy((1 + 0.1 * rng.standard_normal(320)).astype(np.float32)).to(tdt)
        o = orc.rmsnorm(x, r, w, None, eps=1e-6, in_dtype=dt, out_dtype="f64",
                        residual_dtype="f32")
        assert np.array_equal(o["residual_out"], (x.float() + r).numpy())
        h = torch.from_numpy(o["residual_out"])
        ref = orc.rmsnorm(h, None, w.float(), None, eps=1e-6, in_dtype="f32", out_dtype="f64")
        assert np.array_equal(o["out"], ref["out"])


def test_f32_residual_stream(oracle_mod):
    _check_f32_residual_stream(oracle_mod.default())


def test_f16_norm_paths(oracle_mod):
    _check_f16_norm(oracle_mod.default())


# ---------------------------------------------------------------- e4m3 encoder


def read_e4m3_golden():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_spec_values.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                c, v = line.split()
                rows.append((int(c, 16), float(v)))
    return rows


def test_e4m3_decoder_matches_spec_table(oracle_mod):
    for code, val in read_e4m3_golden():
        got = oracle_mod.e4m3_to_f64(code)
        if math.isnan(val):
            assert math.isnan(got)
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), hex(code)


def test_e4m3_decoder_matches_torch_all_codes(oracle_mod):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle_mod.e4m3_to_f64(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_round_trip_all_codes(oracle_mod):
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle_mod.e4m3_from_f64(oracle_mod.e4m3_to_f64(c)) == c, hex(c)


def test_e4m3_encoder_matches_torch_dense_sweep(oracle_mod):
    # torch's fp32 -> float8_e4m3fn is RNE without saturation; below the first
    # value that rounds past 448 (464 is the tie, rounding to even 448) they agree
    v = np.linspace(-463.9, 463.9, 200001, dtype=np.float32)
    v = np.concatenate([v, np.linspace(-0.03, 0.03, 20001, dtype=np.float32)])
    ref = torch.from_numpy(v.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_mod.e4m3_from_f64(float(x)) for x in v], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_midpoints_round_to_even_and_saturate(oracle_mod):
    for c in range(0x00, 0x7E):
        lo, hi = oracle_mod.e4m3_to_f64(c), oracle_mod.e4m3_to_f64(c + 1)
        mid = (lo + hi) / 2
        want = c if c % 2 == 0 else c + 1
        assert oracle_mod.e4m3_from_f64(mid) == want, hex(c)
        assert oracle_mod.e4m3_from_f64(-mid) == want | 0x80
    for v in (448.0, 449.0, 463.99, 464.0, 479.0, 480.0, 1e6, float("inf")):
        assert oracle_mod.e4m3_from_f64(v) == 0x7E
        assert oracle_mod.e4m3_from_f64(-v) == 0xFE
    assert oracle_mod.e4m3_from_f64(float("nan")) & 0x7F == 0x7F


# ---------------------------------------------------------------- the norm


def read_closed_forms():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "rmsnorm_closed_forms.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            if line == "case":
                cur = {}
            elif line == "end":
                cases.append(cur)
                cur = None
            else:
                k, *vals = line.split()
                cur[k] = [float(v) for v in vals]
    return cases


def test_golden_closed_forms(oracle_mod):
    cases = read_closed_forms()
    assert len(cases) == 3
    for c in cases:
        x = bf16_tensor([c["x"]])
        r = bf16_tensor([c["r"]]) if "r" in c else None
        w = bf16_tensor(c["w"]) if "w" in c else None
        b = bf16_tensor(c["b"]) if "b" in c else None
        o = oracle_mod.rmsnorm(x, r, w, b, eps=c["eps"][0], in_dtype="bf16", out_dtype="bf16",
                               weight_offset=c.get("off", [0.0])[0])
        got = bf16_bits_to_float(o["out"][0])
        assert np.array_equal(got, np.array(c["y"], dtype=np.float32)), (c, got)
        if "res" in c:
            assert np.array_equal(bf16_bits_to_float(o["residual_out"][0]),
                                  np.array(c["res"], dtype=np.float32))


@pytest.mark.parametrize("c", [2.0**-10, 0.75, -3.5, 40.0])
@pytest.mark.parametrize("eps", [0.0, 1e-6, 1e-5, 0.5])
def test_constant_row_closed_form(oracle_mod, c, eps):
    H = 48
    rng = np.random.default_rng(3)
    w = bf16_tensor(1 + 0.1 * rng.standard_normal(H))
    b = bf16_tensor(0.01 * rng.standard_normal(H))
    off = 0.25
    x = bf16_tensor(np.full((2, H), c))
    eps32 = float(np.float32(eps))
    o = oracle_mod.rmsnorm(x, None, w, b, eps=eps32, in_dtype="bf16", out_dtype="f64",
                           weight_offset=off)["out"]
    want = (w.double().numpy() + off) * c / math.sqrt(c * c + eps32) + b.double().numpy()
    assert np.allclose(o, want[None, :], rtol=1e-14, atol=1e-15)


def test_mean_square_of_output(oracle_mod):
    # w = 1, b = 0: mean(y^2) = ms / (ms + eps); = 1 when eps = 0
    rng = np.random.default_rng(5)
    for H in (1, 7, 64, 1000, 4096):
        x = torch.from_numpy(rng.standard_normal((3, H)).astype(np.float32))
        for eps in (0.0, 1e-5, 0.3):
            y = oracle_mod.rmsnorm(x, None, None, None, eps=eps, in_dtype="f32",
                                   out_dtype="f64")["out"]
            ms = (x.double().numpy() ** 2).mean(axis=1)
            assert np.allclose((y ** 2).mean(axis=1), ms / (ms + eps), rtol=1e-12, atol=0)


def test_power_of_two_scale_invariance_bitexact(oracle_mod):
    rng = np.random.default_rng(9)
    x = bf16_tensor(rng.standard_normal((4, 300)))
    w = bf16_tensor(1 + 0.1 * rng.standard_normal(300))
    y0 = oracle_mod.rmsnorm(x, None, w, None, eps=0.0, in_dtype="bf16", out_dtype="bf16")["out"]
    for k in (-20, -3, 1, 5, 30):
        xs = (x.float() * 2.0**k).to(torch.bfloat16)   # exact
        yk = oracle_mod.rmsnorm(xs, None, w, None, eps=0.0, in_dtype="bf16",
                                out_dtype="bf16")["out"]
        assert np.array_equal(y0, yk), k


def test_general_scale_invariance(oracle_mod):
    rng = np.random.default_rng(10)
    x = torch.from_numpy(rng.standard_normal((4, 257)).astype(np.float32))
    a = 3.3
    y0 = oracle_mod.rmsnorm(x, None, None, None, eps=0.0, in_dtype="f32", out_dtype="f64")["out"]
    xa = torch.from_numpy((x.double().numpy() * a).astype(np.float32))
    ya = oracle_mod.rmsnorm(xa, None, None, None, eps=0.0, in_dtype="f32", out_dtype="f64")["out"]
    # xa is a rounded copy of a*x: equal to within the f32 rounding of the input
    assert np.allclose(y0, ya, rtol=2e-7, atol=1e-7)


def test_residual_is_sum_rounded_once(oracle_mod):
    rng = np.random.default_rng(12)
    x = bf16_tensor(rng.standard_normal((16, 512)) * np.exp(rng.uniform(-8, 8, (16, 512))))
    r = bf16_tensor(rng.standard_normal((16, 512)) * np.exp(rng.uniform(-8, 8, (16, 512))))
    o = oracle_mod.rmsnorm(x, r, None, None, eps=1e-6, in_dtype="bf16", out_dtype="bf16")
    # f32 sum of two bf16 values rounded to bf16 by torch equals the exact sum rounded once
    ref = (x.float() + r.float()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(o["residual_out"], ref)
    # commutative
    o2 = oracle_mod.rmsnorm(r, x, None, None, eps=1e-6, in_dtype="bf16", out_dtype="bf16")
    assert np.array_equal(o["residual_out"], o2["residual_out"])
    assert np.array_equal(o["out"], o2["out"])


def test_norm_is_taken_on_rounded_residual(oracle_mod):
    rng = np.random.default_rng(13)
    x = bf16_tensor(rng.standard_normal((8, 384)))
    r = bf16_tensor(rng.standard_normal((8, 384)) * 0.01)
    w = bf16_tensor(1 + 0.1 * rng.standard_normal(384))
    fused = oracle_mod.rmsnorm(x, r, w, None, eps=1e-6, in_dtype="bf16", out_dtype="f64")
    h = torch.from_numpy(fused["residual_out"].view(np.int16)).view(torch.bfloat16)
    plain = oracle_mod.rmsnorm(h, None, w, None, eps=1e-6, in_dtype="bf16", out_dtype="f64")
    assert np.array_equal(fused["out"], plain["out"])
    # and differs from normalising the unrounded f64 sum
    hx = x.double().numpy() + r.double().numpy()
    inv = 1 / np.sqrt((hx ** 2).mean(axis=1, keepdims=True) + float(np.float32(1e-6)))
    unrounded = w.double().numpy() * (hx * inv)
    assert not np.allclose(fused["out"], unrounded, rtol=1e-9, atol=0)


def test_bias_and_weight_offset_are_linear_terms(oracle_mod):
    rng = np.random.default_rng(14)
    H = 200
    x = bf16_tensor(rng.standard_normal((5, H)))
    # weights k/64 so that w + 1 is exactly representable in bf16
    wk = rng.integers(32, 96, size=H) / 64.0
    w = bf16_tensor(wk)
    w1 = bf16_tensor(wk + 1.0)
    b = bf16_tensor(0.01 * rng.standard_normal(H))
    y_b = oracle_mod.rmsnorm(x, None, w, b, eps=1e-6, in_dtype="bf16", out_dtype="f64")["out"]
    y_0 = oracle_mod.rmsnorm(x, None, w, None, eps=1e-6, in_dtype="bf16", out_dtype="f64")["out"]
    assert np.allclose(y_b - y_0, b.double().numpy()[None, :], rtol=0, atol=1e-14)
    y_off = oracle_mod.rmsnorm(x, None, w, None, eps=1e-6, in_dtype="bf16", out_dtype="f64",
                               weight_offset=1.0)["out"]
    y_w1 = oracle_mod.rmsnorm(x, None, w1, None, eps=1e-6, in_dtype="bf16", out_dtype="f64")["out"]
    assert np.array_equal(y_off, y_w1)
    # sign: a negative weight flips the output
    y_neg = oracle_mod.rmsnorm(x, None, bf16_tensor(-wk), None, eps=1e-6, in_dtype="bf16",
                               out_dtype="f64")["out"]
    assert np.array_equal(y_neg, -y_0)


def test_brute_force_tiny_rows_exact_rational(oracle_mod):
    # exact rational residual sum and mean square, 60-digit square root,
    # nearest-bf16 search; per element of rows of H <= 8
    rng = np.random.default_rng(15)
    getcontext().prec = 60
    for H in (1, 2, 3, 5, 8):
        for trial in range(6):
            x = bf16_tensor(rng.standard_normal((1, H)) * 2.0 ** rng.integers(-4, 5))
            r = bf16_tensor(rng.standard_normal((1, H)))
            w = bf16_tensor(1 + 0.1 * rng.standard_normal(H))
            b = bf16_tensor(0.01 * rng.standard_normal(H))
            eps = float(np.float32(1e-6))
            o = oracle_mod.rmsnorm(x, r, w, b, eps=eps, in_dtype="bf16", out_dtype="bf16")
            xs = [Fraction(float(v)) for v in x.float()[0]]
            rs = [Fraction(float(v)) for v in r.float()[0]]
            ws = [Fraction(float(v)) for v in w.float()]
            bs = [Fraction(float(v)) for v in b.float()]
            hbits = [exact_round_bf16(a + c) for a, c in zip(xs, rs)]
            assert list(o["residual_out"][0]) == hbits
            h = [Fraction(float(bf16_bits_to_float(np.array([hb], dtype=np.uint16))[0]))
                 for hb in hbits]
            ms = sum(v * v for v in h) / H + Fraction(eps)
            root = Decimal(ms.numerator) / Decimal(ms.denominator)
            inv = Fraction(Decimal(1) / root.sqrt())
            want = [exact_round_bf16(wj * (hj * inv) + bj) for wj, hj, bj in zip(ws, h, bs)]
            assert list(o["out"][0]) == want, (H, trial)


def test_fp32_and_bf16_outputs_are_the_f64_output_rounded(oracle_mod):
    rng = np.random.default_rng(16)
    x = torch.from_numpy(rng.standard_normal((6, 333)).astype(np.float32))
    w = torch.from_numpy((1 + 0.1 * rng.standard_normal(333)).astype(np.float32))
    y64 = oracle_mod.rmsnorm(x, None, w, None, eps=1e-6, in_dtype="f32", out_dtype="f64")["out"]
    y32 = oracle_mod.rmsnorm(x, None, w, None, eps=1e-6, in_dtype="f32", out_dtype="f32")["out"]
    assert np.array_equal(y32, y64.astype(np.float32))
    ybf = oracle_mod.rmsnorm(x, None, w, None, eps=1e-6, in_dtype="f32", out_dtype="bf16")["out"]
    for i in range(0, 6 * 333, 37):
        v = y64.flat[i]
        assert ybf.flat[i] == exact_round_bf16(Fraction(float(v)))


def test_fp8_output_properties(oracle_mod):
    rng = np.random.default_rng(17)
    T, H = 6, 5120
    x = bf16_tensor(rng.standard_normal((T, H)))
    r = bf16_tensor(rng.standard_normal((T, H)))
    w = bf16_tensor(1 + 0.1 * rng.standard_normal(H))
    b = bf16_tensor(0.01 * rng.standard_normal(H))
    q = oracle_mod.rmsnorm(x, r, w, b, eps=1e-6, in_dtype="bf16", out_dtype="fp8")
    y = oracle_mod.rmsnorm(x, r, w, b, eps=1e-6, in_dtype="bf16", out_dtype="f64")["out"]
    a = np.abs(y).max(axis=1)
    assert np.array_equal(q["out_scale"], (a / 448.0).astype(np.float32))
    codes = q["out"]
    dec = np.array([oracle_mod.e4m3_to_f64(c) for c in range(256)])[codes]
    for t in range(T):
        j = int(np.argmax(np.abs(y[t])))
        assert codes[t, j] in (0x7E, 0xFE)
        assert np.sign(dec[t, j]) == np.sign(y[t, j])
        s = a[t] / 448.0
        err = np.abs(dec[t] * s - y[t])
        normal = np.abs(y[t]) / s >= 2.0**-6
        # half a quantum: relative 2^-4 for normals, 2^-10 (absolute, in units of s) below
        assert np.all(err[normal] <= np.abs(y[t][normal]) * 2.0**-4 * (1 + 1e-12))
        assert np.all(err[~normal] <= s * 2.0**-10 * (1 + 1e-12))
    # zero row: scale 0 and all codes +0; constant row: every code is 448
    z = oracle_mod.rmsnorm(torch.zeros((1, 64), dtype=torch.bfloat16), None, None, None,
                           eps=1e-6, in_dtype="bf16", out_dtype="fp8")
    assert z["out_scale"][0] == 0 and not z["out"].any()
    cst = oracle_mod.rmsnorm(bf16_tensor(np.full((1, 64), -2.5)), None, None, None,
                             eps=1e-6, in_dtype="bf16", out_dtype="fp8")
    assert np.all(cst["out"] == 0xFE)


def test_threads_do_not_change_results_and_empty_input(oracle_mod):
    rng = np.random.default_rng(18)
    x = bf16_tensor(rng.standard_normal((37, 129)))
    r = bf16_tensor(rng.standard_normal((37, 129)))
    a = oracle_mod.rmsnorm(x, r, None, None, eps=1e-6, in_dtype="bf16", out_dtype="bf16",
                           n_threads=1)
    b = oracle_mod.rmsnorm(x, r, None, None, eps=1e-6, in_dtype="bf16", out_dtype="bf16",
                           n_threads=8)
    assert np.array_equal(a["out"], b["out"])
    assert np.array_equal(a["residual_out"], b["residual_out"])
    e = oracle_mod.rmsnorm(torch.zeros((0, 16), dtype=torch.bfloat16), None, None, None,
                           eps=1e-6, in_dtype="bf16", out_dtype="bf16")
    assert e["out"].shape == (0, 16)


# ---------------------------------------------------------------- QK norm


def test_qk_norm_equals_row_norm_of_heads(oracle_mod):
    # a contiguous [T, heads * D] q is the row norm of its [T * heads, D] view
    _check_qk_equals_rows(oracle_mod.default())


def _check_qk_equals_rows(orc):
    rng = np.random.default_rng(40)
    T, Hq, Hk, D = 5, 4, 2, 64
    q = bf16_tensor(rng.standard_normal((T, Hq * D)))
    k = bf16_tensor(rng.standard_normal((T, Hk * D)) * 3)
    wq = bf16_tensor(1 + 0.1 * rng.standard_normal(D))
    wk = bf16_tensor(1 + 0.2 * rng.standard_normal(D))
    qo, ko = orc.qk_norm(q, k, wq, wk, n_q_heads=Hq, n_k_heads=Hk, head_dim=D, eps=1e-6,
                         dtype="bf16", weight_offset=0.5)
    rq = orc.rmsnorm(q.reshape(T * Hq, D), None, wq, None, eps=1e-6, in_dtype="bf16",
                     out_dtype="bf16", weight_offset=0.5)["out"]
    rk = orc.rmsnorm(k.reshape(T * Hk, D), None, wk, None, eps=1e-6, in_dtype="bf16",
                     out_dtype="bf16", weight_offset=0.5)["out"]
    assert np.array_equal(qo.reshape(T * Hq, D), rq)
    assert np.array_equal(ko.reshape(T * Hk, D), rk)


def _check_qk_constant_heads(orc):
    # constant head c: every element becomes (w_j + off) * c / sqrt(c^2 + eps),
    # with the query weight on query heads and the key weight on key heads
    D, c, eps, off = 16, 0.25, 0.0625, 0.5
    wq = bf16_tensor(np.linspace(0.5, 2.0, D))
    wk = bf16_tensor(np.linspace(-1.0, 1.0, D))
    q = bf16_tensor(np.full((2, 3 * D), c))
    k = bf16_tensor(np.full((2, 1 * D), -c))
    qo, ko = orc.qk_norm(q, k, wq, wk, n_q_heads=3, n_k_heads=1, head_dim=D, eps=eps,
                         dtype="bf16", weight_offset=off)
    want_q = torch.from_numpy((wq.double().numpy() + off) * c / math.sqrt(c * c + eps)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    want_k = torch.from_numpy((wk.double().numpy() + off) * -c / math.sqrt(c * c + eps)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(qo.reshape(-1, D), np.tile(want_q, (6, 1)))
    assert np.array_equal(ko.reshape(-1, D), np.tile(want_k, (2, 1)))


def _check_qk_strided_fused_qkv(orc):
    # q and k inside a fused [T, (Hq + 2 Hk) * D + pad] qkv buffer: heads are
    # normalised like the contiguous case; v and the row padding are untouched
    rng = np.random.default_rng(41)
    T, Hq, Hk, D, pad = 3, 2, 1, 32, 16
    S = (Hq + 2 * Hk) * D + pad
    qkv = bf16_tensor(rng.standard_normal((T, S)))
    wq = bf16_tensor(1 + 0.1 * rng.standard_normal(D))
    wk = bf16_tensor(1 + 0.1 * rng.standard_normal(D))
    qo, _ = orc.qk_norm(qkv, None, wq, None, n_q_heads=Hq, n_k_heads=0, head_dim=D,
                        eps=1e-6, dtype="bf16")
    _, ko = orc.qk_norm(None, qkv[:, Hq * D:].contiguous(), None, wk, n_q_heads=0,
                        n_k_heads=Hk, head_dim=D, eps=1e-6, dtype="bf16")
    cq, ck = orc.qk_norm(qkv[:, :Hq * D].contiguous(), qkv[:, Hq * D:(Hq + Hk) * D].contiguous(),
                         wq, wk, n_q_heads=Hq, n_k_heads=Hk, head_dim=D, eps=1e-6, dtype="bf16")
    bits = qkv.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(qo[:, :Hq * D], cq)
    assert np.array_equal(qo[:, Hq * D:], bits[:, Hq * D:])
    assert np.array_equal(ko[:, :Hk * D], ck)
    assert np.array_equal(ko[:, Hk * D:], bits[:, (Hq + Hk) * D:])


def test_qk_norm_constant_heads(oracle_mod):
    _check_qk_constant_heads(oracle_mod.default())


def test_qk_norm_strided_fused_qkv(oracle_mod):
    _check_qk_strided_fused_qkv(oracle_mod.default())


# ---------------------------------------------------------------- block-scaled outputs


def test_e2m1_decoder_matches_spec_table(oracle_mod):
    orc = oracle_mod.default()
    with open(os.path.join(GOLDEN, "e2m1_spec_values.txt")) as f:
        rows = [l.split("#")[0].split() for l in f if l.split("#")[0].strip()]
    assert len(rows) == 16
    for c, v in rows:
        got = orc.e2m1_to_f64(int(c, 16))
        assert got == float(v) and math.copysign(1, got) == math.copysign(1, float(v))


def _check_e2m1_encoder(orc):
    for c in range(16):
        assert orc.e2m1_from_f64(orc.e2m1_to_f64(c)) == c
    for c in range(7):
        lo, hi = orc.e2m1_to_f64(c), orc.e2m1_to_f64(c + 1)
        want = c if c % 2 == 0 else c + 1
        assert orc.e2m1_from_f64((lo + hi) / 2) == want, c
        assert orc.e2m1_from_f64(-(lo + hi) / 2) == want | 8
        assert orc.e2m1_from_f64(lo + (hi - lo) * 0.49) == c
        assert orc.e2m1_from_f64(lo + (hi - lo) * 0.51) == c + 1
    for v in (6.0, 6.5, 7.0, 100.0, float("inf")):
        assert orc.e2m1_from_f64(v) == 7 and orc.e2m1_from_f64(-v) == 15


def test_e2m1_encoder_round_trip_ties_saturation(oracle_mod):
    _check_e2m1_encoder(oracle_mod.default())


def test_e8m0_decoder(oracle_mod):
    orc = oracle_mod.default()
    assert orc.e8m0_to_f64(127) == 1.0 and orc.e8m0_to_f64(128) == 2.0
    assert orc.e8m0_to_f64(0) == 2.0 ** -127 and orc.e8m0_to_f64(254) == 2.0 ** 127
    assert math.isnan(orc.e8m0_to_f64(255))


def _unpack_fp4(q):
    out = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = q & 0xF
    out[..., 1::2] = q >> 4
    return out


def _dequant(orc, fmt, b, H):
    T = b["q"].shape[0]
    if fmt == "mxfp8":
        el = np.array([orc.e4m3_to_f64(c) for c in range(256)])[b["q"]]
    else:
        el = np.array([orc.e2m1_to_f64(c) for c in range(16)])[_unpack_fp4(b["q"])]
    if fmt == "nvfp4":
        sb = np.array([orc.e4m3_to_f64(c) for c in range(256)])[b["block_scale"]]
        scale = np.repeat(sb, 16, axis=1) * b["token_scale"].astype(np.float64)[:, None]
    else:
        scale = np.repeat(np.array([orc.e8m0_to_f64(c) for c in range(256)])[b["block_scale"]],
                          32, axis=1)
    return el * scale


def _check_mx_exact_blocks(orc):
    # rows whose blocks hold exactly representable values: every block of 32
    # has max |y| = 2^k, so the scale is 2^(k - emax) and y / X is a value of
    # the element format -> dequantisation is exact
    rng = np.random.default_rng(50)
    T, H = 3, 128
    for fmt, vals in (("mxfp8", [1.0, 0.5, -0.75, 0.125, 1.5 / 4, -1.0]),
                      ("mxfp4", [1.0, 0.5, -0.75, 0.25, -1.0, 0.375])):
        kb = rng.integers(-20, 20, size=(T, H // 32)).astype(float)
        v = rng.choice(vals, size=(T, H))
        v[:, ::32] = 1.0                       # the block maximum, |v| <= 1 elsewhere
        y = v * 2.0 ** np.repeat(kb, 32, axis=1)
        b = orc.block_quantize(y, fmt)
        k = np.log2(np.abs(y[:, ::32]))
        emax = 8 if fmt == "mxfp8" else 2
        assert np.array_equal(b["block_scale"].astype(int), (k - emax + 127).astype(int))
        assert np.array_equal(_dequant(orc, fmt, b, H), y)


def _check_block_error_bounds(orc):
    rng = np.random.default_rng(51)
    T, H = 4, 256
    y = rng.standard_normal((T, H)) * np.exp(rng.uniform(-6, 6, (T, 1)))
    y[2] = 0.0
    for fmt, mant, top in (("mxfp8", 3, 448.0), ("mxfp4", 1, 6.0), ("nvfp4", 1, 6.0)):
        b = orc.block_quantize(y, fmt)
        d = _dequant(orc, fmt, b, H)
        blk = 16 if fmt == "nvfp4" else 32
        for t in range(T):
            for j0 in range(0, H, blk):
                yb, db = y[t, j0:j0 + blk], d[t, j0:j0 + blk]
                if not np.any(yb):
                    assert not np.any(db)
                    continue
                if fmt == "nvfp4":
                    s = orc.e4m3_to_f64(b["block_scale"][t, j0 // 16]) * float(b["token_scale"][t])
                else:
                    s = orc.e8m0_to_f64(b["block_scale"][t, j0 // 32])
                v = np.abs(yb) / s
                # half the spacing of the element format at v (normals), or the
                # subnormal spacing, plus the saturation above the largest value
                e = np.floor(np.log2(np.maximum(v, 1e-300)))
                e = np.maximum(e, 0 if fmt != "mxfp8" else -6)
                half = 2.0 ** (e - mant - 1)
                bound = (half + np.maximum(v - top, 0)) * s * (1 + 1e-12)
                assert np.all(np.abs(db - yb) <= bound), (fmt, t, j0)
        # each non-zero block's largest element lands at the top of the element
        # range: NVFP4 +-6 (the block scale is max / 6 up to its E4M3
        # rounding), MX in [2^emax, 2^(emax+1)) after the power-of-two scale
        codes = b["q"] if fmt == "mxfp8" else _unpack_fp4(b["q"])
        for t in range(T):
            for j0 in range(0, H, blk):
                yb = y[t, j0:j0 + blk]
                if not np.any(yb):
                    continue
                c = int(codes[t, j0 + int(np.argmax(np.abs(yb)))])
                if fmt == "nvfp4":
                    assert c & 7 == 7, (t, j0, c)
                elif fmt == "mxfp4":
                    assert c & 7 in (6, 7), (t, j0, c)
                else:
                    assert c & 0x7F >= 0x78, (t, j0, c)
        if fmt == "nvfp4":
            for t in (0, 1, 3):
                a = np.abs(y[t]).max()
                assert b["token_scale"][t] == np.float32(a / 2688.0)
                jb = int(np.argmax(np.abs(y[t]))) // 16
                assert b["block_scale"][t, jb] == 0x7E       # 448
                assert _unpack_fp4(b["q"])[t, int(np.argmax(np.abs(y[t])))] in (7, 15)
            assert b["token_scale"][2] == 0 and not b["block_scale"][2].any()
        else:
            assert not b["block_scale"][2].any() and not b["q"][2].any()


def test_mx_exact_blocks(oracle_mod):
    _check_mx_exact_blocks(oracle_mod.default())


def test_block_formats_error_bounds_and_scales(oracle_mod):
    _check_block_error_bounds(oracle_mod.default())


def test_rmsnorm_block_is_norm_then_quantize(oracle_mod):
    orc = oracle_mod.default()
    rng = np.random.default_rng(52)
    x = bf16_tensor(rng.standard_normal((3, 64)))
    r = bf16_tensor(rng.standard_normal((3, 64)))
    o = orc.rmsnorm_block(x, r, None, None, eps=1e-6, in_dtype="bf16", fmt="mxfp8")
    y = orc.rmsnorm(x, r, None, None, eps=1e-6, in_dtype="bf16", out_dtype="f64")
    assert np.array_equal(o["y64"], y["out"]) and np.array_equal(o["residual_out"], y["residual_out"])
    assert np.array_equal(o["q"], orc.block_quantize(y["out"], "mxfp8")["q"])


# ---------------------------------------------------------------- mutants

# Each mutant plants one plausible mistake in the oracle's C source: a dropped
# term, a wrong sign, a wrong divisor, a transposed index, a misplaced eps, a
# wrong FP8 constant, normalising the unrounded residual.
MUTANTS = {
    "divide_by_H_minus_1": ("ss / (double)H", "ss / (double)(H - 1)"),
    "eps_outside_sqrt": ("1.0 / sqrt(ms + J->eps)", "1.0 / (sqrt(ms) + J->eps)"),
    "eps_dropped": ("1.0 / sqrt(ms + J->eps)", "1.0 / sqrt(ms)"),
    "bias_dropped": ("* (h[j] * inv) + b;", "* (h[j] * inv);"),
    "offset_sign": ("(w + J->weight_offset)", "(w - J->weight_offset)"),
    "residual_sign": ("xv + rv)", "xv - rv)"),
    "weight_reversed": ("load_in(J->weight, J->in_dtype, j)",
                        "load_in(J->weight, J->in_dtype, H - 1 - j)"),
    "unrounded_norm": ("h[j] = round_store_in(J->residual_out, J->res_dtype, base + j, xv + rv);",
                       "round_store_in(J->residual_out, J->res_dtype, base + j, xv + rv); "
                       "h[j] = xv + rv;"),
    "residual_stream_rounded_to_input": (
        "h[j] = round_store_in(J->residual_out, J->res_dtype, base + j, xv + rv);",
        "h[j] = round_store_in(J->residual_out, J->res_dtype, base + j, "
        "oracle_bf16_to_f64(oracle_bf16_from_f64(xv + rv)));"),
    "fp8_max_240": ("a / 448.0", "a / 240.0"),
    "bf16_truncates": ("r = round_to_quantum(a, q);\n        const double maxf",
                       "r = ldexp(floor(ldexp(a, -q)), q);\n        const double maxf"),
    "qk_weights_swapped": ("k_weight, eps,\n                    weight_offset);",
                           "q_weight, eps,\n                    weight_offset);"),
    "qk_divisor_off_by_one": ("ss / (double)head_dim + eps", "ss / (double)(head_dim - 1) + eps"),
    "mx_emax_off_by_one": ("const int emax = elem_fp4 ? 2 : 8;", "const int emax = elem_fp4 ? 2 : 7;"),
    "nvfp4_scale_uses_4": ("amax / (6.0 * (double)g)", "amax / (4.0 * (double)g)"),
    "e2m1_ties_up": ("r = round_to_quantum(a, q);\n        if (r > 6.0)",
                     "r = ldexp(floor(ldexp(a, -q) + 0.5), q);\n        if (r > 6.0)"),
    "f16_max_wrong": ("if (r > 65504.0) r = INFINITY;", "if (r > 65472.0) r = INFINITY;"),
    "f16_loads_as_bf16": ("return dtype == ORC_F16 ? oracle_f16_to_f64(b) : oracle_bf16_to_f64(b);",
                          "return oracle_bf16_to_f64(b);"),
    "e4m3_ties_up": ("r = round_to_quantum(a, q);\n        if (r > 448.0)",
                     "r = ldexp(floor(ldexp(a, -q) + 0.5), q);\n        if (r > 448.0)"),
}


def all_pin_checks(orc):
    """Every norm / encoder pin above, run against one oracle build."""
    checks = [
        lambda: test_bf16_encoder_ties_and_boundaries(orc),
        lambda: test_e4m3_midpoints_round_to_even_and_saturate(orc),
        lambda: test_golden_closed_forms(orc),
        lambda: test_mean_square_of_output(orc),
        lambda: test_residual_is_sum_rounded_once(orc),
        lambda: test_norm_is_taken_on_rounded_residual(orc),
        lambda: test_bias_and_weight_offset_are_linear_terms(orc),
        lambda: test_fp8_output_properties(orc),
    ]
    for c, eps in ((2.0**-10, 1e-6), (0.75, 0.5), (-3.5, 0.0)):
        checks.append(lambda c=c, eps=eps: test_constant_row_closed_form(orc, c, eps))
    checks.append(lambda: test_brute_force_tiny_rows_exact_rational(orc))
    checks.append(lambda: _check_qk_equals_rows(orc))
    checks.append(lambda: _check_qk_constant_heads(orc))
    checks.append(lambda: _check_qk_strided_fused_qkv(orc))
    checks.append(lambda: _check_e2m1_encoder(orc))
    checks.append(lambda: _check_f16_encoder(orc))
    checks.append(lambda: _check_f16_norm(orc))
    checks.append(lambda: _check_f32_residual_stream(orc))
    checks.append(lambda: _check_mx_exact_blocks(orc))
    checks.append(lambda: _check_block_error_bounds(orc))
    failed = 0
    for chk in checks:
        try:
            chk()
        except AssertionError:
            failed += 1
    return failed


def test_pins_pass_on_the_oracle(oracle_mod):
    assert all_pin_checks(oracle_mod.default()) == 0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(oracle_mod, tmp_path, name):
    src = open(oracle_mod.SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutated = tmp_path / "oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle_mod.build(force=True, src=str(mutated), out=str(tmp_path / "libmut.so"))
    orc = oracle_mod.Oracle(lib)
    assert all_pin_checks(orc) >= 1, f"no pin catches mutant {name}"
