"""The bulk-copy kernel's give-up path, run on a healthy GPU.

Every wait of the ring kernel for a row to land in shared memory is bounded.
rmsnorm_set_wait_limit(-1) makes each wait test its barrier once and not
wait, so on rows whose copies are still in flight the wait runs out while
the copies themselves complete normally.  The kernel must then return, set
bit 0 of the status word, leave every row it did not finish unwritten, and
have finished rows equal to the oracle's; the block drains its own copies
with the default bound before it exits, so the device stays usable.
"""
import numpy as np
import pytest
import torch

import parity
from residual_add_rmsnorm_vec_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
CANARY = 0x7FC1  # a bf16 NaN pattern the kernel never writes for finite inputs


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from residual_add_rmsnorm_vec_gb300 import build

    build.build()
    import residual_add_rmsnorm_vec_gb300 as p

    torch.cuda.set_device(0)
    return p


def ring_config(pkg, stages):
    return pkg.RmsnConfig.from_dict({"variant": pkg.VARIANT_BULK_ROW, "chunks": 2,
                                     "max_warps": 16, "stages": stages})


def run(pkg, g, cfg, T, H):
    out = torch.full((T, H), CANARY, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    res = torch.full((T, H), CANARY, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    pkg.fused_add_rmsnorm(g["x"], g["residual"], g["weight"], g["bias"], eps=1e-6, out=out,
                          residual_out=res, config=cfg)
    torch.cuda.synchronize()
    return parity.bits16(out), parity.bits16(res)


@pytest.mark.parametrize("stages", [2, 4])
def test_wait_that_runs_out_stops_cleanly(pkg, stages):
    T, H = 4096, 8192
    wl = synth.Workload("wait_expiry", T, H, 95, "bf16", "bf16", 1e-6, has_bias=True)
    inp = synth.make_inputs(wl)
    ref = parity.oracle_run(wl, inp)
    g = parity.to_device(inp, DEV)
    cfg = ring_config(pkg, stages)
    pkg.rmsnorm_read_status(clear=True)
    hits, finished = 0, 0
    try:
        assert pkg.rmsnorm_set_wait_limit(-1) == pkg.RMSN_OK
        for _ in range(4):
            out, res = run(pkg, g, cfg, T, H)
            status = pkg.rmsnorm_read_status(clear=True)
            done = ~np.all(out == CANARY, axis=1)  # rows the kernel wrote an output for
            # a row is written whole or not at all
            assert np.all(np.all(out[done] != CANARY, axis=1))
            # finished rows: exactly the oracle's residual, output within 1 ulp
            assert np.array_equal(res[done], ref["residual_out"][done])
            d = np.abs(parity.ordered16(out[done]) - parity.ordered16(ref["out"][done]))
            assert d.size == 0 or d.max() <= parity.BF16_ULP
            finished += int(done.sum())
            if status & 1:
                hits += 1
                assert not done.all(), "the status says a wait ran out, yet every row finished"
            else:
                assert done.all(), "rows were left unwritten with no wait reported"
    finally:
        pkg.rmsnorm_set_wait_limit(0)
        pkg.rmsnorm_read_status(clear=True)
    assert hits >= 1, "no wait ran out although none was allowed to wait"
    # the device is still usable: the default bound gives the full result
    out, res = run(pkg, g, cfg, T, H)
    assert pkg.rmsnorm_read_status() == 0
    got = {"out": out, "residual_out": res, "out_scale": None}
    parity.compare(wl, got, ref, "after the give-up path", bias=inp["bias"])


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_pipelined_ring_wait_that_runs_out_stops_cleanly(pkg, fmt):
    # the two-row pipelined ring (quantised outputs): every row is either
    # written exactly as a launch with the default bound writes it, or not
    # written at all (its canaries intact: FP8 code 0xFF and E4M3 block scale
    # 0xFF are NaN, which the saturating conversions never produce)
    T, H = 4096, 5120
    wl = synth.fp8_workload(H, n_tokens=T)
    g = parity.to_device(synth.make_inputs(wl), DEV)
    flags = pkg.make_flags("bf16", "fp8", True, True, True)
    cfg = [c for c in pkg.rmsnorm_list_configs(T, H, flags)
           if c.variant == pkg.VARIANT_BULK_PIPE and c.chunks == 2][0]
    s = torch.cuda.current_stream().cuda_stream
    code, blk, per_byte = pkg.BLOCK_FORMATS["nvfp4"]

    def launch():
        q = torch.full((T, H if fmt == "fp8" else H // 2), 0xFF, dtype=torch.uint8, device=DEV)
        bs = torch.full((T, H // blk), 0xFF, dtype=torch.uint8, device=DEV)
        sc = torch.zeros((T,), dtype=torch.float32, device=DEV)
        res = torch.full((T, H), CANARY, dtype=torch.int16, device=DEV).view(torch.bfloat16)
        ptr = [g["x"].data_ptr(), g["residual"].data_ptr(), g["weight"].data_ptr(),
               g["bias"].data_ptr()]
        if fmt == "fp8":
            st = pkg.rmsnorm_fwd_ex(*ptr, q.data_ptr(), res.data_ptr(), sc.data_ptr(), T, H,
                                    wl.eps, flags, 0.0, cfg, s)
        else:
            st = pkg.rmsnorm_fwd_blockscaled(*ptr, q.data_ptr(), bs.data_ptr(), sc.data_ptr(),
                                             res.data_ptr(), T, H, wl.eps,
                                             pkg.make_flags("bf16", "f32", True, True, True),
                                             code, 0.0, cfg, s)
        assert st == pkg.RMSN_OK
        torch.cuda.synchronize()
        return (q.cpu().numpy(), bs.cpu().numpy(), sc.cpu().numpy(), parity.bits16(res))

    want = launch()
    assert pkg.rmsnorm_read_status() == 0
    pkg.rmsnorm_read_status(clear=True)
    hits = 0
    try:
        pkg.rmsnorm_set_wait_limit(-1)
        for _ in range(4):
            q, bs, sc, res = launch()
            status = pkg.rmsnorm_read_status(clear=True)
            mark = q if fmt == "fp8" else bs
            done = ~np.all(mark == 0xFF, axis=1)
            assert np.all(mark[~done] == 0xFF) and np.all(q[~done] == 0xFF)
            assert np.all(mark[done] != 0xFF), "a row's output half written"
            assert np.array_equal(q[done], want[0][done]) and np.array_equal(sc[done], want[2][done])
            assert np.array_equal(res[done], want[3][done])
            if fmt == "nvfp4":
                assert np.array_equal(bs[done], want[1][done])
            if status & 1:
                hits += 1
                assert not done.all()
            else:
                assert done.all()
    finally:
        pkg.rmsnorm_set_wait_limit(0)
        pkg.rmsnorm_read_status(clear=True)
    assert hits >= 1, "no wait ran out although none was allowed to wait"


def test_qk_ring_wait_that_runs_out_stops_cleanly(pkg):
    # the QK norm's ring variant under the same limit: every head is either
    # normalised as the oracle does or left as it was
    import oracle

    T, Hq, Hk, D = 8192, 32, 8, 128
    inp = synth.qk_inputs(T, Hq, Hk, D, "bf16")
    qkv = inp["qkv"]
    ref_q, ref_k = oracle.qk_norm(qkv[:, :Hq * D].contiguous(),
                                  qkv[:, Hq * D:(Hq + Hk) * D].contiguous(), inp["q_weight"],
                                  inp["k_weight"], n_q_heads=Hq, n_k_heads=Hk, head_dim=D,
                                  eps=1e-6, dtype="bf16")
    orig = parity.bits16(qkv[:, :(Hq + Hk) * D])
    want = np.concatenate([ref_q, ref_k], axis=1)
    pkg.rmsnorm_read_status(clear=True)
    hits = 0
    try:
        pkg.rmsnorm_set_wait_limit(-1)
        for _ in range(4):
            g = qkv.cuda()
            pkg.qk_norm_(g[:, :Hq * D], g[:, Hq * D:(Hq + Hk) * D], inp["q_weight"].cuda(),
                         inp["k_weight"].cuda(), head_dim=D, eps=1e-6, variant="ring")
            torch.cuda.synchronize()
            got = parity.bits16(g[:, :(Hq + Hk) * D]).reshape(T, Hq + Hk, D)
            status = pkg.rmsnorm_read_status(clear=True)
            same_as_input = np.all(got == orig.reshape(T, Hq + Hk, D), axis=2)
            d = np.abs(parity.ordered16(got) -
                       parity.ordered16(want.reshape(T, Hq + Hk, D))).max(axis=2)
            assert np.all(same_as_input | (d <= 1)), "a head half written or wrong"
            if status & 1:
                hits += 1
            else:
                assert np.all(d <= 1)
    finally:
        pkg.rmsnorm_set_wait_limit(0)
        pkg.rmsnorm_read_status(clear=True)
    assert hits >= 1, "no wait ran out although none was allowed to wait"
