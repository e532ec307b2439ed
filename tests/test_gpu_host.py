"""GPU parity of rmsnorm_fwd_host: rows in host memory, read and written by
the kernel across the CPU-GPU link, checked against the CPU oracle with the
same tolerances as the device path (tests/parity.py)."""
import numpy as np
import pytest
import torch

import parity
from residual_add_rmsnorm_vec_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from residual_add_rmsnorm_vec_gb300 import build

    build.build()
    import residual_add_rmsnorm_vec_gb300 as p

    torch.cuda.set_device(0)
    return p


def pinned(inp):
    return {k: (None if v is None else v.pin_memory()) for k, v in inp.items()}


def run_host(pkg, wl, inp, weight_offset=0.0):
    out, res, scale = pkg.fused_add_rmsnorm_host(inp["x"], inp["residual"], inp["weight"],
                                                 inp["bias"], eps=wl.eps,
                                                 out_dtype=wl.out_dtype,
                                                 weight_offset=weight_offset)
    torch.cuda.synchronize()
    return parity.gpu_outputs_to_host(wl, out, res, scale)


@pytest.mark.parametrize("wl", [
    synth.prefill_workload(2048, 8192),
    synth.decode_workload(8),
    synth.fp8_workload(5120, n_tokens=512),
    synth.fp8_workload(7168, n_tokens=256),
    synth.fp32_workload(),
    synth.Workload("host_ragged", 33, 1000, 9, "bf16", "bf16", 1e-6, has_bias=True),
    synth.Workload("host_wide", 64, 16384, 5, "bf16", "bf16", 1e-6),
], ids=lambda w: w.name)
def test_host_memory_parity(pkg, wl):
    inp = synth.make_inputs(wl)
    got = run_host(pkg, wl, pinned(inp))
    parity.compare(wl, got, parity.oracle_run(wl, inp), f"host {wl.name}", bias=inp["bias"])
    assert pkg.rmsnorm_read_status() == 0


def test_host_and_device_pointers_mixed(pkg):
    # x and residual in pinned host memory, weight and outputs on the device
    wl = synth.prefill_workload(512, 4096)
    inp = synth.make_inputs(wl)
    x, r = inp["x"].pin_memory(), inp["residual"].pin_memory()
    w = inp["weight"].cuda()
    out = torch.empty((wl.n_tokens, wl.hidden), dtype=torch.bfloat16, device="cuda")
    res = torch.empty_like(out)
    pkg.fused_add_rmsnorm_host(x, r, w, None, eps=wl.eps, out=out, residual_out=res)
    torch.cuda.synchronize()
    got = parity.gpu_outputs_to_host(wl, out, res, None)
    parity.compare(wl, got, parity.oracle_run(wl, inp), "mixed host/device")


def test_pageable_memory_is_used_or_rejected(pkg):
    # ordinary (not page-locked) host memory: the library either runs the
    # kernel on it (the device reports pageable-memory access) or rejects it
    # with RMSN_EINVAL before any launch; both outcomes are checked
    wl = synth.decode_workload(32)
    inp = synth.make_inputs(wl)
    try:
        out, res, _ = pkg.fused_add_rmsnorm_host(
            inp["x"], inp["residual"], inp["weight"], None, eps=wl.eps,
            out=torch.empty((32, 4096), dtype=torch.bfloat16),
            residual_out=torch.empty((32, 4096), dtype=torch.bfloat16))
    except pkg.RmsnError as e:
        assert e.status == pkg.RMSN_EINVAL
        return
    torch.cuda.synchronize()
    got = parity.gpu_outputs_to_host(wl, out, res, None)
    parity.compare(wl, got, parity.oracle_run(wl, inp), "pageable host memory")


def test_host_entry_validates_before_launch(pkg):
    x = torch.zeros((4, 64), dtype=torch.bfloat16).pin_memory()
    flags = pkg.make_flags("bf16", "bf16", True, False, False)
    # residual flag without a residual pointer
    st = pkg.rmsnorm_fwd_host(x.data_ptr(), None, None, None, x.data_ptr(), x.data_ptr(), None,
                              4, 64, 1e-6, flags, 0.0, None)
    assert st == pkg.RMSN_EINVAL
    assert pkg.rmsnorm_fwd_host(None, None, None, None, None, None, None, 0, 64, 1e-6,
                                pkg.make_flags("bf16", "bf16", False, False, False), 0.0,
                                None) == pkg.RMSN_OK


def test_other_gpu_memory_refused_before_launch(pkg):
    # device memory of another GPU cannot be read without peer access: the
    # host entry refuses it on the host, before anything is launched
    if torch.cuda.device_count() < 2:
        pytest.skip("needs a second GPU to hold the foreign buffer")
    T, H = 4, 256
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda:1")
    out = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    torch.cuda.set_device(0)
    st = pkg.rmsnorm_fwd_host(x.data_ptr(), None, None, None, out.data_ptr(), None, None, T, H,
                              1e-6, pkg.make_flags("bf16", "bf16", False, False, False), 0.0,
                              torch.cuda.current_stream(0).cuda_stream)
    assert st == pkg.RMSN_EINVAL


def test_own_device_memory_accepted(pkg):
    # the same call with the buffer on the current GPU runs and is correct
    wl = synth.Workload("host_own_dev", 4, 256, 3, "bf16", "bf16", 1e-6, has_residual=False,
                        has_weight=False)
    inp = synth.make_inputs(wl)
    x = inp["x"].to("cuda:0")
    out = torch.empty((4, 256), dtype=torch.bfloat16).pin_memory()
    st = pkg.rmsnorm_fwd_host(x.data_ptr(), None, None, None, out.data_ptr(), None, None, 4, 256,
                              1e-6, pkg.make_flags("bf16", "bf16", False, False, False), 0.0,
                              torch.cuda.current_stream(0).cuda_stream)
    assert st == pkg.RMSN_OK
    torch.cuda.synchronize()
    parity.compare(wl, parity.gpu_outputs_to_host(wl, out, None, None),
                   parity.oracle_run(wl, inp), "own device")
