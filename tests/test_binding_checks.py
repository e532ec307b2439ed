"""The tensor binding refuses, before any launch, every tensor the kernels
would index past or misread: wrong shape, dtype, device or layout.  These
checks run on CPU tensors (no GPU, no library call)."""
import pytest
import torch

import residual_add_rmsnorm_vec_gb300 as rn

T, H = 4, 64


def args(**kw):
    a = dict(x=torch.zeros(T, H, dtype=torch.bfloat16),
             residual=torch.zeros(T, H, dtype=torch.bfloat16),
             weight=torch.zeros(H, dtype=torch.bfloat16), bias=None, out=None,
             residual_out=None, out_scale=None, out_dtype="bf16")
    a.update(kw)
    return a


def test_valid_arguments_pass():
    rn.check_row_args(**args())
    rn.check_row_args(**args(out=torch.zeros(T, H, dtype=torch.bfloat16),
                             residual_out=torch.zeros(T, H, dtype=torch.bfloat16),
                             bias=torch.zeros(H, dtype=torch.bfloat16)))
    # fp32 residual stream under bf16 activations
    rn.check_row_args(**args(residual=torch.zeros(T, H), residual_out=torch.zeros(T, H)))
    rn.check_row_args(**args(out=torch.zeros(T, H, dtype=torch.uint8), out_dtype="fp8",
                             out_scale=torch.zeros(T)))
    rn.check_row_args(**args(residual=None, weight=None))


@pytest.mark.parametrize("kw,err", [
    (dict(x=torch.zeros(T, H, 1, dtype=torch.bfloat16)), ValueError),
    (dict(x=torch.zeros(T, H, dtype=torch.int32)), TypeError),
    (dict(x=torch.zeros(H, T, dtype=torch.bfloat16).t()), ValueError),  # not contiguous
    (dict(residual=torch.zeros(T, H + 1, dtype=torch.bfloat16)), ValueError),
    (dict(residual=torch.zeros(T - 1, H, dtype=torch.bfloat16)), ValueError),
    (dict(residual=torch.zeros(T, H, dtype=torch.float16)), TypeError),
    (dict(weight=torch.zeros(H // 2, dtype=torch.bfloat16)), ValueError),
    (dict(weight=torch.zeros(H)), TypeError),
    (dict(bias=torch.zeros(H + 8, dtype=torch.bfloat16)), ValueError),
    (dict(out=torch.zeros(T, H // 2, dtype=torch.bfloat16)), ValueError),
    (dict(out=torch.zeros(T, H, dtype=torch.float16)), TypeError),
    (dict(out=torch.zeros(T, H, dtype=torch.uint8), out_dtype="fp8",
          out_scale=torch.zeros(T - 1)), ValueError),
    (dict(out_scale=torch.zeros(T)), ValueError),  # no FP8 output
    (dict(residual_out=torch.zeros(T, H)), TypeError),  # bf16 residual, fp32 residual_out
    (dict(residual=None, residual_out=torch.zeros(T, H, dtype=torch.bfloat16)), ValueError),
    (dict(residual=torch.zeros(2 * T, H, dtype=torch.bfloat16)[::2]), ValueError),
])
def test_bad_arguments_are_refused(kw, err):
    with pytest.raises(err):
        rn.check_row_args(**args(**kw))


def test_device_is_checked():
    a = args()
    with pytest.raises(ValueError):
        rn.check_row_args(**a, device=torch.device("meta"))


def test_entry_points_refuse_host_tensors_for_device_calls():
    x = torch.zeros(T, H, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        rn.fused_add_rmsnorm(x, eps=1e-6)
    with pytest.raises(ValueError):
        rn.fused_add_rmsnorm_blockscaled(x, eps=1e-6, fmt="mxfp8")
    with pytest.raises(ValueError):
        rn.qk_norm_(x, None, head_dim=32, eps=1e-6)


def test_qk_head_width_checked():
    with pytest.raises(ValueError):
        rn.qk_norm_(torch.zeros(T, 100, dtype=torch.bfloat16), None, head_dim=64, eps=1e-6)
    with pytest.raises(ValueError):
        rn.qk_norm_(torch.zeros(T, 2, 32, dtype=torch.bfloat16), None, head_dim=64, eps=1e-6)
    with pytest.raises(TypeError):
        rn.qk_norm_(torch.zeros(T, 128, dtype=torch.bfloat16), torch.zeros(T, 64), head_dim=64,
                    eps=1e-6)


def test_host_entry_checks_shapes_before_the_call():
    x = torch.zeros(T, H, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        rn.fused_add_rmsnorm_host(x, torch.zeros(T, H + 2, dtype=torch.bfloat16), eps=1e-6)
    with pytest.raises(ValueError):
        rn.fused_add_rmsnorm_host(x, None, torch.zeros(H - 1, dtype=torch.bfloat16), eps=1e-6)
