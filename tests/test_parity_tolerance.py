"""CPU checks of the comparison itself (tests/parity.py): an error planted in
a copy of the output (never in a kernel) must fail it, and the widened bound
for 16-bit outputs with a bias admits only elements where the bias cancels."""
import numpy as np
import pytest
import torch

import parity
from residual_add_rmsnorm_vec_gb300 import synth


def bf16_bits(v):
    return parity.bits16(torch.tensor(v, dtype=torch.float64).to(torch.bfloat16))


def case():
    # y64: the oracle's unrounded outputs; b: the bias.  Element 0 does not
    # cancel (w h inv = 0.5, b = 0.5), element 1 does (w h inv = 1 + 2^-20,
    # b = -1: y is 2^-20 of the operands' size)
    y64 = np.array([[1.0, 2.0 ** -20, -3.0, 0.25]])
    b = torch.tensor([0.5, -1.0, 0.0, 0.125], dtype=torch.bfloat16)
    wl = synth.Workload("tol", 1, 4, 0, "bf16", "bf16", 1e-6, has_residual=False, has_bias=True)
    ref = {"out": bf16_bits(y64), "residual_out": None, "out_scale": None, "y64": y64}
    return wl, ref, b


def got_with(ref, j, ulps):
    out = ref["out"].copy().astype(np.int32)
    out[0, j] += ulps  # same sign: ulps along the magnitude
    return {"out": out.astype(np.uint16), "residual_out": None, "out_scale": None}


def test_exact_copy_passes():
    wl, ref, b = case()
    st = parity.compare(wl, got_with(ref, 0, 0), ref, "copy", bias=b)
    assert st["max_ulp"] == 0


def test_one_ulp_passes_anywhere():
    wl, ref, b = case()
    for j in range(4):
        parity.compare(wl, got_with(ref, j, 1), ref, "1 ulp", bias=b)


def test_two_ulp_where_the_bias_does_not_cancel_fails():
    wl, ref, b = case()
    for j in (0, 2, 3):
        with pytest.raises(AssertionError, match="does not cancel"):
            parity.compare(wl, got_with(ref, j, 2), ref, "planted", bias=b)


def test_cancelled_element_may_be_further_off_within_the_fp32_bound():
    wl, ref, b = case()
    # 2^-20 has bf16 ulp 2^-27: 8 ulp is 2^-24 absolute, 6e-8 of |y| + |b|
    st = parity.compare(wl, got_with(ref, 1, 8), ref, "cancelled", bias=b)
    assert st["cancelled"] == 1 and st["cancelled_max_rel"] <= parity.F32_RTOL
    # but not beyond it: 2^14 ulp is 2^-13 absolute, 1.2e-4 of |y| + |b|
    with pytest.raises(AssertionError, match="rel"):
        parity.compare(wl, got_with(ref, 1, 1 << 14), ref, "cancelled, too far", bias=b)


def test_without_bias_two_ulp_fails():
    wl, ref, _ = case()
    with pytest.raises(AssertionError, match="ulp"):
        parity.compare(wl, got_with(ref, 1, 2), ref, "no bias", bias=None)


def test_residual_and_fp8_plants_fail():
    wl = synth.Workload("tol8", 2, 4, 0, "bf16", "fp8", 1e-6, has_bias=True)
    ref = {"out": np.array([[0x38, 0x40, 0xB8, 0x7E]] * 2, dtype=np.uint8),
           "residual_out": np.zeros((2, 4), dtype=np.uint16),
           "out_scale": np.array([1.0, 2.0], dtype=np.float32)}
    ok = {k: v.copy() for k, v in ref.items()}
    parity.compare(wl, ok, ref, "fp8 copy")
    bad = {k: v.copy() for k, v in ref.items()}
    bad["out"][1, 1] += 2
    with pytest.raises(AssertionError, match="steps"):
        parity.compare(wl, bad, ref, "fp8 two steps")
    bad = {k: v.copy() for k, v in ref.items()}
    bad["out_scale"][0] = np.nextafter(np.float32(1.0), np.float32(2.0)) + np.float32(1e-6)
    with pytest.raises(AssertionError, match="scale"):
        parity.compare(wl, bad, ref, "fp8 scale")
    bad = {k: v.copy() for k, v in ref.items()}
    bad["residual_out"][0, 3] ^= 1
    with pytest.raises(AssertionError, match="residual_out"):
        parity.compare(wl, bad, ref, "residual bit")
