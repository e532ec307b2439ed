"""Seeded random cases of the row norm against the CPU oracle: shapes drawn
from the sizes that change the launch (one warp, one block, the ring with
swizzled or linear copies, the ragged-row and generic kernels), every input
/ output dtype pair, the optional residual / weight / bias, a weight
offset, an fp32 residual stream, programmatic dependent launch, and buffers
offset from their allocation by the same or by different element counts.
Each case uses the tolerances of tests/parity.py."""
import numpy as np
import pytest
import torch

import parity
from residual_add_rmsnorm_vec_gb300 import synth

pytestmark = pytest.mark.gpu

N_CASES = 500
HIDDEN = [1, 3, 12, 64, 100, 256, 511, 1000, 1024, 2048, 2050, 4095, 4096, 5120, 7168, 8190, 8192,
          12288, 16384]
TOKENS = [1, 2, 7, 31, 64, 152, 300, 1024, 2500]
PAIRS = [("bf16", "bf16"), ("bf16", "fp8"), ("bf16", "f32"), ("f16", "f16"), ("f16", "fp8"),
         ("f16", "f32"), ("f32", "f32"), ("f32", "bf16"), ("f32", "fp8"), ("f32", "f16")]


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from residual_add_rmsnorm_vec_gb300 import build

    build.build()
    import residual_add_rmsnorm_vec_gb300 as p

    torch.cuda.set_device(0)
    return p


def draw_case(i):
    rng = np.random.default_rng(1000 + i)
    T = int(rng.choice(TOKENS))
    H = int(rng.choice(HIDDEN))
    while T * H > 8_000_000:
        T = max(1, T // 2)
    in_dt, out_dt = PAIRS[int(rng.integers(len(PAIRS)))]
    res = bool(rng.random() < 0.75)
    # the fp32 residual stream is built for outputs of the input dtype and FP8
    r32 = res and in_dt != "f32" and out_dt in (in_dt, "fp8") and bool(rng.random() < 0.35)
    return dict(
        T=T, H=H, in_dt=in_dt, out_dt=out_dt, res=res, r32=r32,
        weight=bool(rng.random() < 0.85), bias=bool(rng.random() < 0.4),
        woff=float(rng.choice([0.0, 0.0, 1.0, -0.25])),
        eps=float(rng.choice([1e-6, 1e-5])), pdl=bool(rng.random() < 0.3),
        # element offsets of x / residual / out / residual_out from a fresh allocation
        offs=[int(v) for v in (rng.integers(0, 3, 4) if rng.random() < 0.3 else [0, 0, 0, 0])],
        same_off=bool(rng.random() < 0.5))


def placed(t, off, dev):
    """A copy of t on `dev` that starts `off` elements into its allocation."""
    flat = torch.zeros(t.numel() + off + 8, dtype=t.dtype, device=dev)
    v = flat[off:off + t.numel()].view(t.shape)
    v.copy_(t)
    return v


def empty_placed(shape, dtype, off, dev):
    n = int(np.prod(shape))
    return torch.empty(n + off + 8, dtype=dtype, device=dev)[off:off + n].view(shape)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case(pkg, i):
    c = draw_case(i)
    wl = synth.Workload(f"fuzz{i}", c["T"], c["H"], 2000 + i, c["in_dt"], c["out_dt"], c["eps"],
                        has_residual=c["res"], has_weight=c["weight"], has_bias=c["bias"],
                        res_dtype="f32" if c["r32"] else None, r_std=2.0)
    inp = synth.make_inputs(wl)
    ref = parity.oracle_run(wl, inp, weight_offset=c["woff"])
    dev = "cuda"
    offs = [c["offs"][0]] * 4 if c["same_off"] else c["offs"]
    x = placed(inp["x"], offs[0], dev)
    r = None if inp["residual"] is None else placed(inp["residual"], offs[1], dev)
    w = None if inp["weight"] is None else inp["weight"].to(dev)
    b = None if inp["bias"] is None else inp["bias"].to(dev)
    out_t = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32,
             "fp8": torch.uint8}[c["out_dt"]]
    out = empty_placed((c["T"], c["H"]), out_t, offs[2], dev)
    ro = None if r is None else empty_placed((c["T"], c["H"]), r.dtype, offs[3], dev)
    y, res, scale = pkg.fused_add_rmsnorm(x, r, w, b, eps=c["eps"], out_dtype=c["out_dt"],
                                          weight_offset=c["woff"], out=out, residual_out=ro,
                                          pdl=c["pdl"])
    torch.cuda.synchronize()
    parity.compare(wl, parity.gpu_outputs_to_host(wl, y, res, scale), ref, f"case {i}: {c}",
                   bias=inp["bias"])
    assert pkg.rmsnorm_read_status() == 0
