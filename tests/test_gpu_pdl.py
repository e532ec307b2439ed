"""Programmatic dependent launch (RMSN_PDL): chained calls where each call
reads what the previous one wrote (y and residual_out feed the next call's
x and residual, as consecutive norms of a layer stack do).  With PDL the next
kernel may start before the previous one ends, so a missing wait would read
stale rows; the chain must be bit-identical to the chain launched without
PDL (same launch shapes), eagerly and in a CUDA graph, and its first call
must match the oracle.  The 16384 x 8192 case is the prefill step that
bench.py times, in its launch configuration (selector's choice + RMSN_PDL)."""
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


def chain(pkg, inp, eps, n, pdl, early, graph=False, config=None):
    x0 = inp["x"].cuda()
    r0 = inp["residual"].cuda()
    w = inp["weight"].cuda()
    T, H = x0.shape
    xs = [x0] + [torch.empty_like(x0) for _ in range(n)]
    rs = [r0] + [torch.empty_like(x0) for _ in range(n)]

    def run():
        for k in range(n):
            pkg.fused_add_rmsnorm(xs[k], rs[k], w, None, eps=eps, out=xs[k + 1],
                                  residual_out=rs[k + 1], pdl=pdl, early_params=early,
                                  config=config)

    if graph:
        run()  # warm the launch-shape caches before capture
        torch.cuda.synchronize()
        for t in xs[1:] + rs[1:]:
            t.zero_()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                run()
        torch.cuda.current_stream().wait_stream(s)
        g.replay()
    else:
        run()
    torch.cuda.synchronize()
    return [parity.bits16(t) for t in xs[1:] + rs[1:]]


@pytest.mark.parametrize("T,H", [(1, 4096), (8, 4096), (256, 4096), (2048, 8192), (37, 1000),
                                 (16384, 8192)])
@pytest.mark.parametrize("early", [False, True])
def test_pdl_chain_matches_plain_chain(pkg, T, H, early):
    # both chains take the launch the selector picks for PDL calls (the table
    # has rows measured with PDL), so only the launch attribute differs
    wl = synth.Workload(f"pdl_T{T}_H{H}", T, H, 21, "bf16", "bf16", 1e-6)
    inp = synth.make_inputs(wl)
    n = 6
    cfg = pkg.rmsnorm_query_config(T, H, pkg.make_flags("bf16", "bf16", True, True, False) |
                                   pkg.RMSN_PDL)
    ref = chain(pkg, inp, wl.eps, n, pdl=False, early=False, config=cfg)
    for graph in (False, True):
        got = chain(pkg, inp, wl.eps, n, pdl=True, early=early, graph=graph)
        for k, (a, b) in enumerate(zip(got, ref)):
            assert np.array_equal(a, b), (graph, k)
    # first link of the chain against the oracle
    o = parity.oracle_run(wl, inp)
    got = {"out": ref[0], "residual_out": ref[n], "out_scale": None}
    parity.compare(wl, got, o, "pdl chain first call")
    assert pkg.rmsnorm_read_status() == 0


@pytest.mark.parametrize("T", [1, 32, 256])
def test_pdl_chain_cluster_variant(pkg, T):
    # the split-row cluster launches chained by PDL (both launch attributes)
    # give the same bits as the plain chain, eagerly and in a graph
    wl = synth.Workload(f"pdl_cluster_T{T}", T, 4096, 23, "bf16", "bf16", 1e-6)
    inp = synth.make_inputs(wl)
    flags = pkg.make_flags("bf16", "bf16", True, True, False)
    for c in pkg.rmsnorm_list_configs(T, 4096, flags):
        if c.variant != pkg.VARIANT_CLUSTER:
            continue
        ref = chain(pkg, inp, wl.eps, 4, pdl=False, early=False, config=c)
        for graph in (False, True):
            got = chain(pkg, inp, wl.eps, 4, pdl=True, early=True, graph=graph, config=c)
            for k, (a, b) in enumerate(zip(got, ref)):
                assert np.array_equal(a, b), (c.cluster, graph, k)


def test_early_params_needs_pdl(pkg):
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    flags = pkg.make_flags("bf16", "bf16", False, False, False) | pkg.RMSN_PDL_EARLY_PARAMS
    st = pkg.rmsnorm_fwd(x.data_ptr(), None, None, None, x.data_ptr(), None, None, 4, 64, 1e-6,
                         flags, torch.cuda.current_stream().cuda_stream)
    assert st == pkg.RMSN_EINVAL


def quant_chain(pkg, inp, eps, n, fmt, pdl, config=None):
    """n calls where call k takes the residual_out of call k - 1 as its
    residual (x, weight and bias fixed); returns every call's outputs, then
    the residual stream."""
    x = inp["x"].cuda()
    w, b = inp["weight"].cuda(), inp["bias"].cuda()
    rs = [inp["residual"].cuda()] + [torch.empty_like(x) for _ in range(n)]
    outs = []
    for k in range(n):
        if fmt == "fp8":
            q, ro, sc = pkg.fused_add_rmsnorm(x, rs[k], w, b, eps=eps, out_dtype="fp8",
                                              residual_out=rs[k + 1], pdl=pdl, config=config)
            outs.append((q, sc))
        else:
            q, bs, ts, ro = pkg.fused_add_rmsnorm_blockscaled(x, rs[k], w, b, eps=eps, fmt=fmt,
                                                              residual_out=rs[k + 1], pdl=pdl,
                                                              config=config)
            outs.append((q, bs) if ts is None else (q, bs, ts))
    torch.cuda.synchronize()
    return [[t.cpu() for t in o] for o in outs] + [[r.cpu()] for r in rs[1:]]


@pytest.mark.parametrize("fmt", ["fp8", "mxfp8", "mxfp4", "nvfp4"])
@pytest.mark.parametrize("T,H", [(4096, 5120), (33, 2048)])
def test_pdl_chain_quantised_outputs(pkg, fmt, T, H):
    # the quantised launches chained by RMSN_PDL, as bench.py times them:
    # with one launch shape forced on both chains, every output is
    # bit-identical with and without PDL; with the selector's picks (the
    # table has rows measured with PDL, so the shapes may differ) the
    # residual stream, which no launch shape changes, still is
    wl = synth.Workload(f"pdlq_{fmt}_T{T}_H{H}", T, H, 22, "bf16", "bf16", 1e-6, has_bias=True)
    inp = synth.make_inputs(wl)
    cfgs = (pkg.rmsnorm_list_configs(T, H, pkg.make_flags("bf16", "fp8", True, True, True))
            if fmt == "fp8" else pkg.block_format_configs(T, H, fmt))
    rings = [c for c in cfgs if c.variant in (pkg.VARIANT_BULK_ROW, pkg.VARIANT_BULK_PIPE)]
    cfg = rings[0] if rings else cfgs[0]
    ref = quant_chain(pkg, inp, wl.eps, 4, fmt, pdl=False, config=cfg)
    got = quant_chain(pkg, inp, wl.eps, 4, fmt, pdl=True, config=cfg)
    for k, (a, b) in enumerate(zip(got, ref)):
        for ta, tb in zip(a, b):
            assert torch.equal(ta, tb), (fmt, k, cfg.as_dict())
    ref = quant_chain(pkg, inp, wl.eps, 4, fmt, pdl=False)
    got = quant_chain(pkg, inp, wl.eps, 4, fmt, pdl=True)
    for k in range(4):
        assert torch.equal(got[4 + k][0], ref[4 + k][0]), (fmt, "residual", k)
    assert pkg.rmsnorm_read_status() == 0
