"""GPU parity of the QK norm (rmsnorm_qk_fwd): per-head RMS norm of query
and key heads in place, against the CPU oracle's per-head norm, with the
bf16 (1 ulp) and fp32 (1e-5 relative) tolerances of tests/parity.py; heads
inside a fused qkv row leave the value heads and the row padding untouched."""
import numpy as np
import pytest
import torch

import oracle
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


def bits(t, dtype):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if dtype in ("bf16", "f16") else t.numpy()


def compare(dtype, got, ref, where):
    if dtype in ("bf16", "f16"):
        d = np.abs(parity.ordered16(got) - parity.ordered16(ref))
        assert d.max() <= parity.BF16_ULP, f"{where}: {d.max()} ulp"
        return float((d == 0).mean())
    rel = np.abs(got.astype(np.float64) - ref) / np.maximum(np.abs(ref.astype(np.float64)), 1e-30)
    assert rel.max() <= parity.F32_RTOL, f"{where}: rel {rel.max()}"
    return 1.0


def ring_applies(Hq, Hk, D, dtype):
    """The ring variant's shapes: 4..32 whole 32-byte vectors per head (a power
    of two), at most 2048 per token."""
    nvec = D * (4 if dtype == "f32" else 2) // 32
    return nvec >= 4 and nvec & (nvec - 1) == 0 and nvec <= 32 and (Hq + Hk) * nvec <= 2048


@pytest.mark.parametrize("T,Hq,Hk,D,dtype", [
    (1, 32, 8, 128, "bf16"), (7, 16, 4, 64, "bf16"), (512, 32, 8, 128, "bf16"),
    (4096, 32, 8, 128, "bf16"), (16384, 32, 8, 128, "bf16"), (33, 8, 2, 256, "bf16"),
    (3, 2, 1, 512, "bf16"),
    (5, 4, 4, 128, "f32"), (65, 6, 2, 64, "f32"), (9, 3, 1, 256, "f32"), (2, 1, 1, 16, "bf16"),
    (17, 32, 8, 128, "f16"), (3, 4, 2, 64, "f16"), (5, 2, 2, 256, "f16"),
    (1100, 4, 2, 96, "bf16"), (37, 5, 3, 96, "bf16"), (29, 7, 5, 64, "f32"),
    (305, 6, 2, 64, "bf16"), (333, 3, 1, 128, "f32"), (641, 64, 8, 128, "bf16"),
])
@pytest.mark.parametrize("pad", [0, 16])
@pytest.mark.parametrize("variant", [None, "ring", "direct"])
@pytest.mark.parametrize("woff", [0.25, 0.0])
def test_qk_norm_fused_qkv(pkg, T, Hq, Hk, D, dtype, pad, variant, woff):
    if pad and dtype == "f32":
        pad = 8  # keep the row stride a multiple of 32 bytes
    if variant == "ring" and not ring_applies(Hq, Hk, D, dtype):
        pytest.skip("the ring variant does not take this head shape")
    inp = synth.qk_inputs(T, Hq, Hk, D, dtype, pad=pad)
    qkv = inp["qkv"]
    S = qkv.shape[1]
    ref_q, _ = oracle.qk_norm(qkv, None, inp["q_weight"], None, n_q_heads=Hq, n_k_heads=0,
                              head_dim=D, eps=1e-6, dtype=dtype, weight_offset=woff)
    _, ref_k = oracle.qk_norm(None, qkv[:, Hq * D:].contiguous(), None, inp["k_weight"],
                              n_q_heads=0, n_k_heads=Hk, head_dim=D, eps=1e-6, dtype=dtype,
                              weight_offset=woff)
    g = qkv.cuda()
    pkg.qk_norm_(g[:, :Hq * D], g[:, Hq * D:(Hq + Hk) * D], inp["q_weight"].cuda(),
                 inp["k_weight"].cuda(), head_dim=D, eps=1e-6, weight_offset=woff,
                 variant=variant)
    torch.cuda.synchronize()
    got = bits(g, dtype)
    orig = bits(qkv, dtype)
    compare(dtype, got[:, :Hq * D], ref_q[:, :Hq * D], "q heads")
    compare(dtype, got[:, Hq * D:(Hq + Hk) * D], ref_k[:, :Hk * D], "k heads")
    # value heads and padding untouched
    assert np.array_equal(got[:, (Hq + Hk) * D:], orig[:, (Hq + Hk) * D:])
    assert S == (Hq + 2 * Hk) * D + pad
    assert pkg.rmsnorm_read_status() == 0


def test_qk_norm_contiguous_heads_no_weights_and_pdl(pkg):
    T, Hq, Hk, D = 100, 8, 2, 128
    inp = synth.qk_inputs(T, Hq, Hk, D, "bf16")
    q = inp["qkv"][:, :Hq * D].contiguous()
    k = inp["qkv"][:, Hq * D:(Hq + Hk) * D].contiguous()
    rq, rk = oracle.qk_norm(q, k, None, None, n_q_heads=Hq, n_k_heads=Hk, head_dim=D,
                            eps=1e-5, dtype="bf16")
    gq, gk = q.cuda().view(T, Hq, D), k.cuda().view(T, Hk, D)
    pkg.qk_norm_(gq, gk, None, None, head_dim=D, eps=1e-5, pdl=True)
    torch.cuda.synchronize()
    compare("bf16", bits(gq, "bf16").reshape(T, -1), rq, "q")
    compare("bf16", bits(gk, "bf16").reshape(T, -1), rk, "k")


def test_qk_ring_rejects_shapes_it_does_not_take(pkg):
    # head_dim 96 bf16 is 6 vectors per head (not a power of two): the ring
    # variant cannot be forced, the default launch still runs
    T, Hq, Hk, D = 1100, 4, 2, 96
    x = torch.zeros((T, (Hq + Hk) * D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkg.RmsnError) as e:
        pkg.qk_norm_(x[:, :Hq * D], x[:, Hq * D:], None, None, head_dim=D, eps=1e-6,
                     variant="ring")
    assert e.value.status == pkg.RMSN_EUNSUPPORTED
    pkg.qk_norm_(x[:, :Hq * D], x[:, Hq * D:], None, None, head_dim=D, eps=1e-6)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream().cuda_stream
    assert pkg.rmsnorm_qk_fwd(x.data_ptr(), None, None, None, T, Hq, 0, D, (Hq + Hk) * D, 0,
                              1e-6, 0.0, pkg.RMSN_IN_BF16 | pkg.RMSN_QK_RING |
                              pkg.RMSN_QK_DIRECT, s) == pkg.RMSN_EINVAL


def test_qk_norm_only_q_or_only_k(pkg):
    T, H, D = 16, 4, 64
    inp = synth.qk_inputs(T, H, H, D, "bf16")
    x = inp["qkv"][:, :H * D].contiguous()
    rq, _ = oracle.qk_norm(x, None, inp["q_weight"], None, n_q_heads=H, n_k_heads=0,
                           head_dim=D, eps=1e-6, dtype="bf16")
    for variant in (None, "ring"):
        g = x.cuda()
        pkg.qk_norm_(g, None, inp["q_weight"].cuda(), None, head_dim=D, eps=1e-6,
                     variant=variant)
        torch.cuda.synchronize()
        compare("bf16", bits(g, "bf16"), rq, f"q only {variant}")
        g = x.cuda()
        pkg.qk_norm_(None, g, None, inp["q_weight"].cuda(), head_dim=D, eps=1e-6,
                     variant=variant)
        torch.cuda.synchronize()
        compare("bf16", bits(g, "bf16"), rq, f"k only {variant}")


def test_qk_norm_rejections(pkg):
    x = torch.zeros((4, 4 * 72), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    bf = pkg.RMSN_IN_BF16
    # head_dim 72 bf16 = 144 bytes: not whole 32-byte vectors
    assert pkg.rmsnorm_qk_fwd(x.data_ptr(), None, None, None, 4, 4, 0, 72, 4 * 72, 0, 1e-6, 0.0,
                              bf, s) == pkg.RMSN_EUNSUPPORTED
    y = torch.zeros((4, 4 * 64 + 8), dtype=torch.bfloat16, device="cuda")
    # token stride of 264 elements = 528 bytes: heads of token 1 not 32-byte aligned
    assert pkg.rmsnorm_qk_fwd(y.data_ptr(), None, None, None, 4, 4, 0, 64, 264, 0, 1e-6, 0.0, bf,
                              s) == pkg.RMSN_EUNSUPPORTED
    # stride shorter than the heads, bad flags, odd address
    assert pkg.rmsnorm_qk_fwd(y.data_ptr(), None, None, None, 4, 4, 0, 64, 100, 0, 1e-6, 0.0, bf,
                              s) == pkg.RMSN_EINVAL
    assert pkg.rmsnorm_qk_fwd(y.data_ptr(), None, None, None, 4, 4, 0, 64, 256, 0, 1e-6, 0.0,
                              bf | 0x4, s) == pkg.RMSN_EINVAL
    assert pkg.rmsnorm_qk_fwd(y.data_ptr() + 1, None, None, None, 4, 4, 0, 64, 256, 0, 1e-6, 0.0,
                              bf, s) == pkg.RMSN_EALIGN
    assert pkg.rmsnorm_qk_fwd(None, None, None, None, 0, 4, 0, 64, 256, 0, 1e-6, 0.0, bf,
                              s) == pkg.RMSN_OK
    # more head groups per token than the grid's y extent holds (head_dim 512
    # bf16, one head per warp: 2^20 + 16 heads); the buffers are the full
    # size, so even a launch would stay inside them
    Hq, Hk, D = 1 << 20, 16, 512
    q = torch.zeros((1, Hq * D), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, Hk * D), dtype=torch.bfloat16, device="cuda")
    assert pkg.rmsnorm_qk_fwd(q.data_ptr(), k.data_ptr(), None, None, 1, Hq, Hk, D, Hq * D,
                              Hk * D, 1e-6, 0.0, bf, s) == pkg.RMSN_EUNSUPPORTED
    del q, k
