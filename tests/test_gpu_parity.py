"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs, element by element.  Tolerances are in tests/parity.py:
residual_out bit-exact, bf16 <= 1 ulp, fp32 relative <= 1e-5, FP8 <= 1 code
step with per-token scale relative error <= 1e-6.

Workloads are the five hot-path configurations (fp32 plain norm; bf16 decode
T in {1..256} x H=4096; bf16 prefill 16384 x 8192 with outlier channels;
FP8 output with bias at H in {5120, 7168}; the tokens x hidden sweep), plus
ragged, misaligned, aliased and degenerate shapes.
"""
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


DEV = "cuda:0"


def run_gpu(pkg, wl, inp, config=None, weight_offset=0.0):
    g = parity.to_device(inp, DEV)
    out, res, scale = pkg.fused_add_rmsnorm(g["x"], g["residual"], g["weight"], g["bias"],
                                            eps=wl.eps, out_dtype=wl.out_dtype,
                                            weight_offset=weight_offset, config=config)
    torch.cuda.synchronize()
    return parity.gpu_outputs_to_host(wl, out, res, scale)


def check(pkg, wl, rows=None, config=None, weight_offset=0.0, where=""):
    """Full tensors on the GPU; oracle on all rows or the sampled ``rows``."""
    inp = synth.make_inputs(wl)
    got = run_gpu(pkg, wl, inp, config, weight_offset)
    if rows is not None:
        sub = synth.make_inputs(wl, rows=rows)
        ref = parity.oracle_run(wl, sub, weight_offset)
        got = {k: (None if v is None else v[rows]) for k, v in got.items()}
    else:
        ref = parity.oracle_run(wl, inp, weight_offset)
    return parity.compare(wl, got, ref, where or wl.name, bias=inp["bias"])


# ---------------------------------------------------------------- the five configs


def test_fp32_plain_norm(pkg):
    st = check(pkg, synth.fp32_workload())
    assert st["max_rel"] <= 1e-5


@pytest.mark.parametrize("T", synth.DECODE_TOKENS)
def test_decode(pkg, T):
    check(pkg, synth.decode_workload(T))


def test_prefill_full_size(pkg):
    # every row of the 16384 x 8192 workload, the shape the bench times
    wl = synth.prefill_workload()
    st = check(pkg, wl)
    assert st["exact_frac"] > 0.99


@pytest.mark.parametrize("stages", [2, 3, 6])
@pytest.mark.parametrize("ch,wmax", [(2, 16), (1, 16), (2, 8)])
def test_prefill_full_size_bulk_ring(pkg, stages, ch, wmax):
    # the shared-memory ring variant at every row of the bench workload
    wl = synth.prefill_workload()
    cfg = pkg.RmsnConfig.from_dict({"variant": pkg.VARIANT_BULK_ROW, "chunks": ch,
                                    "max_warps": wmax, "stages": stages})
    check(pkg, wl, config=cfg)
    assert pkg.rmsnorm_read_status() == 0


@pytest.mark.parametrize("stages", [2, 5, 8])
@pytest.mark.parametrize("grid", [0, 7])
def test_deep_ring_wraps(pkg, stages, grid):
    # short rows through a deep ring: every stage is refilled many times
    # (3000 rows over 7 blocks: ~430 rows per block)
    wl = synth.Workload(f"ring_st{stages}", 3000, 2048, 78, "bf16", "bf16", 1e-6, has_bias=True)
    cfg = pkg.RmsnConfig.from_dict({"variant": pkg.VARIANT_BULK_ROW, "chunks": 1,
                                    "max_warps": 8, "stages": stages, "grid": grid})
    check(pkg, wl, config=cfg)
    assert pkg.rmsnorm_read_status() == 0


@pytest.mark.parametrize("H", synth.FP8_HIDDEN)
def test_fp8_bias(pkg, H):
    st = check(pkg, synth.fp8_workload(H))
    assert st["exact_frac"] > 0.99


@pytest.mark.parametrize("H", synth.SWEEP_HIDDEN)
@pytest.mark.parametrize("T", synth.SWEEP_TOKENS)
def test_sweep(pkg, T, H):
    wl = synth.sweep_workload(T, H)
    rows = None
    if T * H > 64 * 2**20:
        rows = synth.sample_rows(T, 1024)
    check(pkg, wl, rows=rows)


# ---------------------------------------------------------------- every built variant


FLAG_SETS = [
    ("bf16", "bf16", True, True, False),
    ("bf16", "bf16", True, True, True),
    ("bf16", "bf16", False, False, False),
    ("bf16", "f32", True, True, True),
    ("bf16", "fp8", True, True, True),
    ("bf16", "fp8", False, True, False),
    ("f32", "f32", False, True, False),
    ("f32", "f32", True, True, True),
    ("f32", "bf16", True, True, False),
    ("f32", "fp8", True, True, True),
    ("f16", "f16", True, True, False),
    ("f16", "f16", True, True, True),
    ("f16", "fp8", True, True, True),
    ("f16", "f32", False, True, False),
    ("f32", "f16", True, True, False),
]


@pytest.mark.parametrize("fs", FLAG_SETS, ids=lambda f: "-".join(map(str, f)))
@pytest.mark.parametrize("H", [256, 2048, 5120])
def test_every_config(pkg, fs, H):
    in_dt, out_dt, res, w, b = fs
    T = 37
    wl = synth.Workload(f"cfg_{in_dt}_{out_dt}", T, H, 77, in_dt, out_dt, 1e-6,
                        has_residual=res, has_weight=w, has_bias=b)
    flags = pkg.make_flags(in_dt, out_dt, res, w, b)
    cfgs = pkg.rmsnorm_list_configs(T, H, flags)
    assert cfgs, "no configuration for a vector-aligned shape"
    inp = synth.make_inputs(wl)
    ref = parity.oracle_run(wl, inp)
    variants = set()
    for c in cfgs:
        got = run_gpu(pkg, wl, inp, config=c)
        parity.compare(wl, got, ref, f"{wl.name} {c.as_dict()}", bias=inp["bias"])
        variants.add(c.variant)
        # a small explicit grid exercises the grid-stride row loop
        c2 = pkg.RmsnConfig.from_dict({**c.as_dict(), "grid": 3})
        got = run_gpu(pkg, wl, inp, config=c2)
        parity.compare(wl, got, ref, f"{wl.name} grid=3 {c.as_dict()}", bias=inp["bias"])
    assert pkg.VARIANT_GENERIC in variants and pkg.VARIANT_BLOCK_ROW in variants
    assert pkg.VARIANT_BULK_ROW in variants
    assert pkg.rmsnorm_read_status() == 0


@pytest.mark.parametrize("T", synth.DECODE_TOKENS)
def test_cluster_variant_decode(pkg, T):
    # the split-row variant: each row over a cluster of one-warp blocks that
    # exchange partial sums through distributed shared memory, every built
    # cluster size, on the decode workload (and with a bias and an offset)
    wl = synth.decode_workload(T)
    flags = pkg.make_flags("bf16", "bf16", True, True, False)
    cfgs = [c for c in pkg.rmsnorm_list_configs(T, 4096, flags)
            if c.variant == pkg.VARIANT_CLUSTER]
    assert {c.cluster for c in cfgs} == {2, 4, 8}
    for c in cfgs:
        assert c.grid == T * c.cluster and c.warps_per_block == 1
        check(pkg, wl, config=c, where=f"cluster {c.as_dict()}")
    wlb = synth.Workload(f"cluster_bias_T{T}", T, 4096, 83, "bf16", "bf16", 1e-6, has_bias=True)
    for c in pkg.rmsnorm_list_configs(T, 4096, pkg.make_flags("bf16", "bf16", True, True, True)):
        if c.variant == pkg.VARIANT_CLUSTER:
            check(pkg, wlb, config=c, weight_offset=0.5, where=f"cluster bias {c.as_dict()}")


@pytest.mark.parametrize("T,H", [(1, 4096), (256, 4096), (2048, 8192), (4096, 5120)])
def test_fp16_io(pkg, T, H):
    wl = synth.Workload(f"f16_T{T}_H{H}", T, H, 80, "f16", "f16", 1e-6, has_bias=H == 5120,
                        r_std=2.0)
    st = check(pkg, wl)
    assert st["exact_frac"] > 0.99


@pytest.mark.parametrize("T,H,in_dt,out_dt,bias", [
    (1, 4096, "bf16", "bf16", False), (256, 4096, "bf16", "bf16", False),
    (2048, 8192, "bf16", "bf16", False), (4096, 5120, "bf16", "fp8", True),
    (64, 4096, "f16", "f16", True), (300, 2048, "f16", "fp8", False),
    (33, 1000, "bf16", "bf16", True), (5, 12, "f16", "f16", False),
    (16384, 8192, "bf16", "bf16", False), (4096, 8192, "f16", "f16", True),
])
def test_f32_residual_stream(pkg, T, H, in_dt, out_dt, bias):
    # bf16 / fp16 activations, fp32 residual stream: residual_out is the fp32
    # sum (bit-exact), the norm is taken on it
    wl = synth.Workload(f"r32_{in_dt}_{out_dt}_T{T}_H{H}", T, H, 90, in_dt, out_dt, 1e-6,
                        has_bias=bias, r_std=4.0, res_dtype="f32")
    check(pkg, wl)


@pytest.mark.parametrize("in_dt,out_dt", [("bf16", "bf16"), ("f16", "f16"), ("bf16", "fp8")])
def test_f32_residual_stream_every_config_and_in_place(pkg, in_dt, out_dt):
    wl = synth.Workload(f"r32_cfg_{in_dt}_{out_dt}", 37, 2048, 91, in_dt, out_dt, 1e-6,
                        has_bias=True, res_dtype="f32")
    flags = pkg.make_flags(in_dt, out_dt, True, True, True) | pkg.RMSN_RESIDUAL_F32
    cfgs = pkg.rmsnorm_list_configs(37, 2048, flags)
    assert cfgs and any(c.variant == pkg.VARIANT_BULK_ROW for c in cfgs)
    inp = synth.make_inputs(wl)
    ref = parity.oracle_run(wl, inp)
    for c in cfgs:
        parity.compare(wl, run_gpu(pkg, wl, inp, config=c), ref, f"r32 {c.as_dict()}",
                       bias=inp["bias"])
    # residual_out written over the residual itself (the usual in-place
    # update), with the selector's launch and with every ring shape
    for c in [None] + [c for c in cfgs if c.variant == pkg.VARIANT_BULK_ROW]:
        g = parity.to_device(inp, DEV)
        out, res, scale = pkg.fused_add_rmsnorm(g["x"], g["residual"], g["weight"], g["bias"],
                                                eps=wl.eps, out_dtype=out_dt,
                                                residual_out=g["residual"], config=c)
        torch.cuda.synchronize()
        parity.compare(wl, parity.gpu_outputs_to_host(wl, out, res, scale), ref,
                       f"r32 in place {c}", bias=inp["bias"])


@pytest.mark.parametrize("H", [1, 7, 1000, 4097])
def test_fp16_ragged_generic(pkg, H):
    check(pkg, synth.Workload(f"f16_ragged_H{H}", 21, H, 81, "f16", "f16", 1e-6, has_bias=True))


def test_weight_offset(pkg):
    wl = synth.Workload("woff", 16, 4096, 5, "bf16", "bf16", 1e-6, has_bias=True)
    for off in (1.0, -0.5):
        check(pkg, wl, weight_offset=off)


# ---------------------------------------------------------------- edge cases


@pytest.mark.parametrize("H", [1, 3, 7, 8, 15, 17, 100, 1000, 4095, 4097, 6000])
@pytest.mark.parametrize("out_dt", ["bf16", "fp8", "f32"])
def test_ragged_hidden_out_dtypes(pkg, H, out_dt):
    # odd hidden sizes with a bias: the ragged-row kernel for each output
    wl = synth.Workload(f"ragged_H{H}", 33, H, 9, "bf16", out_dt, 1e-6, has_bias=True)
    check(pkg, wl)


@pytest.mark.parametrize("H", [1, 5, 8, 1001])
def test_ragged_hidden_f32(pkg, H):
    wl = synth.Workload(f"ragged32_H{H}", 19, H, 9, "f32", "f32", 1e-6)
    check(pkg, wl)


def test_empty_batch(pkg):
    x = torch.empty((0, 4096), dtype=torch.bfloat16, device=DEV)
    r = torch.empty_like(x)
    out, res, _ = pkg.fused_add_rmsnorm(x, r, None, None, eps=1e-6)
    assert out.shape == (0, 4096) and res.shape == (0, 4096)


def test_misaligned_pointers_take_generic_path(pkg):
    # views offset by one bf16 element: 2-byte aligned, not 32-byte aligned
    wl = synth.Workload("misaligned", 24, 2048, 11, "bf16", "bf16", 1e-6)
    inp = synth.make_inputs(wl)
    ref = parity.oracle_run(wl, inp)
    T, H = wl.n_tokens, wl.hidden
    bufs = {k: torch.zeros(T * H + 1, dtype=torch.bfloat16, device=DEV) for k in ("x", "r", "o", "ro")}
    x = bufs["x"][1:].view(T, H)
    r = bufs["r"][1:].view(T, H)
    x.copy_(inp["x"])
    r.copy_(inp["residual"])
    wbuf = torch.zeros(H + 1, dtype=torch.bfloat16, device=DEV)
    w = wbuf[1:]
    w.copy_(inp["weight"])
    out = bufs["o"][1:].view(T, H)
    res = bufs["ro"][1:].view(T, H)
    pkg.fused_add_rmsnorm(x, r, w, None, eps=wl.eps, out=out, residual_out=res)
    torch.cuda.synchronize()
    got = parity.gpu_outputs_to_host(wl, out, res, None)
    parity.compare(wl, got, ref, "misaligned")


def test_unequally_misaligned_pointers_take_generic_path(pkg):
    # x one element off a 16-byte boundary, the residual two: the ragged-row
    # kernel needs every row pointer equally aligned, so the generic one runs
    wl = synth.Workload("misaligned2", 24, 2048, 12, "bf16", "bf16", 1e-6)
    inp = synth.make_inputs(wl)
    ref = parity.oracle_run(wl, inp)
    T, H = wl.n_tokens, wl.hidden
    xb = torch.zeros(T * H + 8, dtype=torch.bfloat16, device=DEV)
    rb = torch.zeros(T * H + 8, dtype=torch.bfloat16, device=DEV)
    x, r = xb[1:1 + T * H].view(T, H), rb[2:2 + T * H].view(T, H)
    x.copy_(inp["x"])
    r.copy_(inp["residual"])
    out, res, _ = pkg.fused_add_rmsnorm(x, r, inp["weight"].to(DEV), None, eps=wl.eps)
    torch.cuda.synchronize()
    parity.compare(wl, parity.gpu_outputs_to_host(wl, out, res, None), ref, "unequal offsets")


RAGGED_H = [1, 7, 9, 100, 1000, 4097, 8190]


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("out", ["same", "fp8", "mixed"])
@pytest.mark.parametrize("res,bias", [(True, True), (True, False), (False, True), (False, False)])
@pytest.mark.parametrize("H", RAGGED_H)
def test_ragged_kernel_every_config(pkg, dt, out, res, bias, H):
    # rows off the 32-byte grid: the selector takes the ragged-row kernel, and
    # every listed shape of it (and a 3-block grid looping over rows) matches
    # the oracle, for the input's dtype out, a per-token FP8 output, and fp32
    # out of 16-bit rows / bf16 out of fp32 rows
    T = 37
    if H * (4 if dt == "f32" else 2) % 32 == 0:
        pytest.skip("rows on the 32-byte grid take the vector kernels")
    odt = {"same": dt, "fp8": "fp8", "mixed": "bf16" if dt == "f32" else "f32"}[out]
    wl = synth.Workload(f"rag_{dt}_{odt}_H{H}", T, H, 79, dt, odt, 1e-6, has_residual=res,
                        has_bias=bias)
    flags = pkg.make_flags(dt, odt, res, True, bias)
    assert pkg.rmsnorm_query_config(T, H, flags).variant == pkg.VARIANT_RAGGED
    cfgs = [c for c in pkg.rmsnorm_list_configs(T, H, flags) if c.variant == pkg.VARIANT_RAGGED]
    assert cfgs
    inp = synth.make_inputs(wl)
    ref = parity.oracle_run(wl, inp)
    for c in cfgs:
        for grid in (0, 3):
            c2 = pkg.RmsnConfig.from_dict({**c.as_dict(), "grid": grid})
            parity.compare(wl, run_gpu(pkg, wl, inp, config=c2), ref,
                           f"{wl.name} {c2.as_dict()}", bias=inp["bias"])
    assert pkg.rmsnorm_read_status() == 0


@pytest.mark.parametrize("T,H,dt,odt", [(3000, 4097, "bf16", "bf16"), (2048, 8190, "bf16", "bf16"),
                                        (16384, 8190, "bf16", "bf16"), (1000, 6001, "f32", "f32"),
                                        (4096, 5118, "bf16", "fp8"), (16384, 8190, "bf16", "fp8"),
                                        (999, 7167, "f16", "fp8"), (777, 3001, "f32", "fp8"),
                                        (16384, 8190, "bf16", "f32"), (555, 4097, "f32", "f16")])
def test_ragged_kernel_large(pkg, T, H, dt, odt):
    rows = synth.sample_rows(T, 1024) if T > 4096 else None
    check(pkg, synth.Workload(f"rag_large_T{T}_H{H}_{odt}", T, H, 80, dt, odt, 1e-5,
                              has_bias=True, r_std=2.0), rows=rows)


def test_ragged_fp8_output_alignment(pkg):
    # views offset by one element: x, residual and the FP8 out one element
    # off their boundaries take the ragged-row kernel; an FP8 out offset
    # differently falls back to the generic kernel; both match the oracle
    wl = synth.Workload("rag_fp8_views", 24, 2048, 13, "bf16", "fp8", 1e-6, has_bias=True)
    inp = synth.make_inputs(wl)
    ref = parity.oracle_run(wl, inp)
    T, H = wl.n_tokens, wl.hidden
    w, b = inp["weight"].to(DEV), inp["bias"].to(DEV)  # alive until the kernels ran
    for q_off in (1, 2):
        xb = torch.zeros(T * H + 8, dtype=torch.bfloat16, device=DEV)
        rb = torch.zeros(T * H + 8, dtype=torch.bfloat16, device=DEV)
        rob = torch.zeros(T * H + 8, dtype=torch.bfloat16, device=DEV)
        qb = torch.zeros(T * H + 8, dtype=torch.uint8, device=DEV)
        x, r = xb[1:1 + T * H].view(T, H), rb[1:1 + T * H].view(T, H)
        ro, q = rob[1:1 + T * H].view(T, H), qb[q_off:q_off + T * H].view(T, H)
        x.copy_(inp["x"])
        r.copy_(inp["residual"])
        scale = torch.zeros(T, dtype=torch.float32, device=DEV)
        s = torch.cuda.current_stream().cuda_stream
        st = pkg.rmsnorm_fwd(x.data_ptr(), r.data_ptr(), w.data_ptr(), b.data_ptr(),
                             q.data_ptr(), ro.data_ptr(),
                             scale.data_ptr(), T, H, wl.eps,
                             pkg.make_flags("bf16", "fp8", True, True, True), s)
        assert st == pkg.RMSN_OK
        torch.cuda.synchronize()
        parity.compare(wl, parity.gpu_outputs_to_host(wl, q, ro, scale), ref,
                       f"fp8 out offset {q_off}", bias=inp["bias"])


@pytest.mark.parametrize("alias", ["residual_out=residual", "out=x", "out=residual"])
def test_ragged_kernel_in_place(pkg, alias):
    wl = synth.Workload("rag_inplace", 29, 1000, 81, "bf16", "bf16", 1e-6, has_bias=True)
    inp = synth.make_inputs(wl)
    ref = parity.oracle_run(wl, inp)
    g = parity.to_device(inp, DEV)
    kw = {"residual_out=residual": dict(residual_out=g["residual"]),
          "out=x": dict(out=g["x"]),
          "out=residual": dict(out=g["residual"], residual_out=torch.empty_like(g["residual"]))}[alias]
    out, res, _ = pkg.fused_add_rmsnorm(g["x"], g["residual"], g["weight"], g["bias"],
                                        eps=wl.eps, **kw)
    torch.cuda.synchronize()
    parity.compare(wl, parity.gpu_outputs_to_host(wl, out, res, None), ref, alias,
                   bias=inp["bias"])


def test_odd_byte_pointer_rejected(pkg):
    buf = torch.zeros(2 * 64 * 64 + 2, dtype=torch.uint8, device=DEV)
    base = buf.data_ptr()
    st = pkg.rmsnorm_fwd(base + 1, base + 1, None, None, base + 1, base + 1, None, 4, 64, 1e-6,
                         pkg.make_flags("bf16", "bf16", True, False, False),
                         torch.cuda.current_stream().cuda_stream)
    assert st == pkg.RMSN_EALIGN


@pytest.mark.parametrize("alias", ["residual_out=residual", "residual_out=x", "out=x",
                                   "out=residual"])
def test_in_place_aliasing(pkg, alias):
    wl = synth.Workload("alias", 40, 4096, 13, "bf16", "bf16", 1e-6)
    inp = synth.make_inputs(wl)
    ref = parity.oracle_run(wl, inp)
    g = parity.to_device(inp, DEV)
    x, r = g["x"].clone(), g["residual"].clone()
    out = res = None
    if alias == "residual_out=residual":
        res = r
    elif alias == "residual_out=x":
        res = x
    elif alias == "out=x":
        out = x
    else:
        out = r
    o, ro, _ = pkg.fused_add_rmsnorm(x, r, g["weight"], None, eps=wl.eps, out=out, residual_out=res)
    torch.cuda.synchronize()
    got = parity.gpu_outputs_to_host(wl, o, ro, None)
    parity.compare(wl, got, ref, alias)


def test_in_place_no_residual_generic(pkg):
    wl = synth.Workload("alias_gen", 9, 1000, 14, "bf16", "bf16", 1e-6, has_residual=False)
    inp = synth.make_inputs(wl)
    ref = parity.oracle_run(wl, inp)
    x = inp["x"].to(DEV)
    o, _, _ = pkg.fused_add_rmsnorm(x, None, inp["weight"].to(DEV), None, eps=wl.eps, out=x)
    torch.cuda.synchronize()
    parity.compare(wl, parity.gpu_outputs_to_host(wl, o, None, None), ref, "in-place generic")


def test_degenerate_rows(pkg):
    # zero rows (FP8 scale 0, codes +0), constant rows, large and tiny values.
    # The fp32 sum of squares bounds the range: rows need sum(h^2) < FLT_MAX,
    # i.e. rms(h) < sqrt(FLT_MAX / H) (about 4e17 at H = 2048); 1e15 is inside.
    T, H = 8, 2048
    x = torch.zeros((T, H), dtype=torch.float32)
    x[1] = 3.0
    x[2] = -1e15
    x[3, ::2] = 1e-30
    x[4] = torch.linspace(-100, 100, H)
    xb = x.to(torch.bfloat16)
    for out_dt in ("bf16", "fp8", "f32"):
        wl = synth.Workload("degenerate", T, H, 0, "bf16", out_dt, 1e-6, has_residual=False,
                            has_weight=False)
        inp = {"x": xb, "residual": None, "weight": None, "bias": None}
        got = run_gpu(pkg, wl, inp)
        ref = parity.oracle_run(wl, inp)
        parity.compare(wl, got, ref, f"degenerate {out_dt}")
        if out_dt == "fp8":
            assert got["out_scale"][0] == 0 and not got["out"][0].any()
            assert np.all(got["out"][1] == 0x7E)


def test_forced_unbuilt_config_rejected(pkg):
    wl = synth.decode_workload(8)
    inp = parity.to_device(synth.make_inputs(wl), DEV)
    bad = pkg.RmsnConfig.from_dict({"variant": pkg.VARIANT_BLOCK_ROW, "chunks": 3, "max_warps": 8})
    with pytest.raises(pkg.RmsnError) as e:
        pkg.fused_add_rmsnorm(inp["x"], inp["residual"], inp["weight"], None, eps=1e-6, config=bad)
    assert e.value.status == pkg.RMSN_EUNSUPPORTED
    # a row wider than one warp's registers cannot take the one-warp shape
    big = pkg.RmsnConfig.from_dict({"variant": pkg.VARIANT_WARP_ROWS, "chunks": 1, "max_warps": 1})
    with pytest.raises(pkg.RmsnError):
        pkg.fused_add_rmsnorm(inp["x"], inp["residual"], inp["weight"], None, eps=1e-6, config=big)


def _same_shape(a, b):
    keys = ("variant", "chunks", "max_warps", "warps_per_block", "stages")
    return all(getattr(a, k) == getattr(b, k) for k in keys)


def test_selector_decode_vs_prefill(pkg):
    flags = pkg.make_flags("bf16", "bf16", True, True, False)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # a hidden size without measured rows but a measured neighbour within 2x
    # (2560: 3072 is nearest) takes the neighbour's launch shape
    keys = ("variant", "chunks", "max_warps", "stages")
    for T in (8, 4096):
        c = pkg.rmsnorm_query_config(T, 2560, flags)
        n = pkg.rmsnorm_query_config(T, 3072, flags)
        assert all(getattr(c, k) == getattr(n, k) for k in keys) and c.num_sms == sms, \
            (T, c.as_dict(), n.as_dict())
    # no measured hidden size within 2x (bf16 512: the nearest, 2048, is 4x
    # away): the decode rule (one warp per block while the problem needs
    # fewer warps than there are SMs), else one block per row
    c = pkg.rmsnorm_query_config(8, 512, flags)
    assert c.variant == pkg.VARIANT_WARP_ROWS and c.warps_per_block == 1
    c = pkg.rmsnorm_query_config(16384, 512, flags)
    assert c.variant == pkg.VARIANT_BLOCK_ROW
    # measured shapes: whatever the table picked is a valid built configuration
    for T, H in ((1, 4096), (8, 4096), (256, 4096), (16384, 8192), (4096, 16384), (8, 3072),
                 (4096, 6144), (16384, 7168)):
        c = pkg.rmsnorm_query_config(T, H, flags)
        assert any(_same_shape(c, o) for o in pkg.rmsnorm_list_configs(T, H, flags)), (T, H)
        assert 1 <= c.grid <= max(T, 1)
        # PDL calls take the rows measured with PDL where the hidden size has
        # them, else the plain rows: a built shape either way
        cp = pkg.rmsnorm_query_config(T, H, flags | pkg.RMSN_PDL)
        assert any(_same_shape(cp, o) for o in pkg.rmsnorm_list_configs(T, H, flags)), (T, H)
    # hidden 3072 has no PDL rows: a PDL call takes its plain rows, not a
    # PDL neighbour's
    c, cp = (pkg.rmsnorm_query_config(256, 3072, flags | f) for f in (0, pkg.RMSN_PDL))
    assert _same_shape(c, cp)
    # rows off the 32-byte grid: the ragged-row kernel for the same dtype in
    # and out, a per-token FP8 output and fp32 out of 16-bit rows; the generic
    # one otherwise (here: bf16 activations over an fp32 residual stream)
    for out in ("bf16", "fp8", "f32"):
        c = pkg.rmsnorm_query_config(16, 1000, pkg.make_flags("bf16", out, True, True, False))
        assert c.variant == pkg.VARIANT_RAGGED, out
    c = pkg.rmsnorm_query_config(16, 1001, flags | pkg.RMSN_RESIDUAL_F32)
    assert c.variant == pkg.VARIANT_GENERIC


def test_register_launch_grid(pkg):
    # the register kernels take one unit per block where a unit moves at
    # least 4 KiB of x (grid = rows, or row groups for one warp per row);
    # smaller units, and the rings, stay on a grid of resident blocks
    flags = pkg.make_flags("bf16", "bf16", True, True, False)
    for c in pkg.rmsnorm_list_configs(16384, 8192, flags):
        if c.variant == pkg.VARIANT_BLOCK_ROW:
            assert c.grid == 16384, c.as_dict()
        elif c.variant in (pkg.VARIANT_BULK_ROW, pkg.VARIANT_BULK_PIPE):
            assert c.grid <= 8 * c.num_sms, c.as_dict()
    for c in pkg.rmsnorm_list_configs(65536, 2048, flags):
        if c.variant == pkg.VARIANT_WARP_ROWS:
            assert c.grid == -(-65536 // c.warps_per_block), c.as_dict()
    small = [c for c in pkg.rmsnorm_list_configs(65536, 128, flags)
             if c.variant in (pkg.VARIANT_BLOCK_ROW, pkg.VARIANT_WARP_ROWS)]
    assert small and all(c.grid < 65536 // c.warps_per_block for c in small
                         if c.variant == pkg.VARIANT_WARP_ROWS)
    assert all(c.grid < 65536 for c in small if c.variant == pkg.VARIANT_BLOCK_ROW)
    # the selected bench launch is the one-row register launch, and its
    # parity at full size is covered by test_prefill_full_size
    c = pkg.rmsnorm_query_config(16384, 8192, flags)
    assert c.variant == pkg.VARIANT_BLOCK_ROW and c.grid == 16384


def test_ring_copy_mode(pkg):
    # the ring launches of the bench shape fill their stages with swizzled
    # tensor copies; rows that are not whole 1 KiB units fall back to 1-D
    # bulk copies
    flags = pkg.make_flags("bf16", "bf16", True, True, False)
    rings = [c for c in pkg.rmsnorm_list_configs(16384, 8192, flags)
             if c.variant == pkg.VARIANT_BULK_ROW]
    assert rings and all(c.ring_copy == 2 for c in rings)
    rings = [c for c in pkg.rmsnorm_list_configs(37, 256, flags)
             if c.variant == pkg.VARIANT_BULK_ROW]
    assert rings and all(c.ring_copy == 1 for c in rings)
    rings = (pkg.VARIANT_BULK_ROW, pkg.VARIANT_BULK_PIPE)
    assert all(c.ring_copy == 0 for c in pkg.rmsnorm_list_configs(37, 256, flags)
               if c.variant not in rings)


def test_selection_cache_keeps_colliding_problems_apart(pkg):
    # (8 x 8) and (2 x 384), fp32 with residual and weight, hash alike in the
    # launch cache: the second call must get its own launch (the first one's
    # single-warp shape would leave a third of its row unwritten)
    for i, (T, H) in enumerate(((8, 8), (2, 384), (8, 8))):
        check(pkg, synth.Workload(f"cache_{T}x{H}", T, H, 300 + i, "f32", "f32", 1e-6))


def test_status_word_clear_after_all_runs(pkg):
    # no bounded wait in any kernel ran out during the suite
    assert pkg.rmsnorm_read_status(clear=False) == 0


def test_streams_are_respected(pkg):
    wl = synth.decode_workload(128)
    inp = synth.make_inputs(wl)
    ref = parity.oracle_run(wl, inp)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = parity.to_device(inp, DEV)
        out, res, _ = pkg.fused_add_rmsnorm(g["x"], g["residual"], g["weight"], None, eps=wl.eps)
    s.synchronize()
    parity.compare(wl, parity.gpu_outputs_to_host(wl, out, res, None), ref, "side stream")
