"""Guard bands around every output: each output buffer is carved out of a
larger allocation whose bytes before and after it hold a canary pattern.
After the call every canary byte must be unchanged, so no kernel writes
outside its outputs.  This runs every launch configuration the library
lists (and a small explicit grid, which sends blocks round the row loop) on
aligned, ragged and one-row shapes, for the row norm on device and host
memory and for the block-scaled outputs."""
import pytest
import torch

from residual_add_rmsnorm_vec_gb300 import synth

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side; a multiple of 256 keeps the output aligned
CANARY = 0xA5


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from residual_add_rmsnorm_vec_gb300 import build

    build.build()
    import residual_add_rmsnorm_vec_gb300 as p

    torch.cuda.set_device(0)
    return p


class Guarded:
    """An output of `shape` and `dtype` between two canary regions."""

    def __init__(self, shape, dtype, device="cuda", pin=False):
        n = 1
        for s in shape:
            n *= s
        self.nbytes = n * torch.empty((), dtype=dtype).element_size()
        buf = torch.full((GUARD + self.nbytes + GUARD,), CANARY, dtype=torch.uint8)
        self.buf = buf.pin_memory() if pin else buf.to(device)
        self.t = self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(*shape)

    def intact(self):
        torch.cuda.synchronize()
        head = self.buf[:GUARD].cpu()
        tail = self.buf[GUARD + self.nbytes:].cpu()
        return bool((head == CANARY).all()) and bool((tail == CANARY).all())


def p(t):
    return None if t is None else t.data_ptr()


def row_case(pkg, wl, config, host=False):
    T, H = wl.n_tokens, wl.hidden
    inp = synth.make_inputs(wl)
    dev = "cpu" if host else "cuda"

    def put(t):
        if t is None:
            return None
        return t.pin_memory() if host else t.to(dev)

    x, r, w, b = (put(inp[k]) for k in ("x", "residual", "weight", "bias"))
    out_t = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32,
             "fp8": torch.uint8}[wl.out_dtype]
    out = Guarded((T, H), out_t, dev, pin=host)
    res = Guarded((T, H), r.dtype, dev, pin=host) if r is not None else None
    sc = Guarded((T,), torch.float32, dev, pin=host) if wl.out_dtype == "fp8" else None
    flags = pkg.make_flags(wl.in_dtype, wl.out_dtype, r is not None, w is not None, b is not None)
    if r is not None and r.dtype == torch.float32 and x.dtype != torch.float32:
        flags |= pkg.RMSN_RESIDUAL_F32
    s = torch.cuda.current_stream().cuda_stream
    args = (p(x), p(r), p(w), p(b), p(out.t), None if res is None else p(res.t),
            None if sc is None else p(sc.t), T, H, wl.eps, flags)
    if host:
        st = pkg.rmsnorm_fwd_host(*args, 0.0, s)
    else:
        st = pkg.rmsnorm_fwd_ex(*args, 0.0, config, s)
    assert st == pkg.RMSN_OK
    for g in (out, res, sc):
        if g is not None:
            assert g.intact(), f"{wl.name} {None if config is None else config.as_dict()}"


FLAG_CASES = [
    ("bf16", "bf16", True, True), ("bf16", "fp8", True, True), ("f32", "f32", False, False),
    ("f16", "f16", True, False), ("bf16", "f32", False, True),
]


@pytest.mark.parametrize("in_dt,out_dt,res,bias", FLAG_CASES)
@pytest.mark.parametrize("T,H", [(37, 2048), (1, 4096), (300, 5120), (7, 1000), (3, 12)])
def test_row_norm_writes_only_its_outputs(pkg, in_dt, out_dt, res, bias, T, H):
    wl = synth.Workload(f"guard_{in_dt}_{out_dt}_T{T}_H{H}", T, H, 95, in_dt, out_dt, 1e-6,
                        has_residual=res, has_bias=bias)
    flags = pkg.make_flags(in_dt, out_dt, res, True, bias)
    cfgs = pkg.rmsnorm_list_configs(T, H, flags)
    assert cfgs
    for c in cfgs:
        row_case(pkg, wl, c)
        row_case(pkg, wl, pkg.RmsnConfig.from_dict({**c.as_dict(), "grid": 3}))
    assert pkg.rmsnorm_read_status() == 0


@pytest.mark.parametrize("T,H", [(37, 2048), (300, 8192)])
def test_f32_residual_stream_writes_only_its_outputs(pkg, T, H):
    wl = synth.Workload(f"guard_r32_T{T}_H{H}", T, H, 96, "bf16", "bf16", 1e-6, has_bias=True,
                        res_dtype="f32")
    flags = pkg.make_flags("bf16", "bf16", True, True, True) | pkg.RMSN_RESIDUAL_F32
    for c in pkg.rmsnorm_list_configs(T, H, flags):
        row_case(pkg, wl, c)


@pytest.mark.parametrize("T,H,out_dt", [(33, 1000, "bf16"), (64, 4096, "fp8"), (5, 8192, "bf16")])
def test_host_memory_entry_writes_only_its_outputs(pkg, T, H, out_dt):
    wl = synth.Workload(f"guard_host_T{T}_H{H}", T, H, 97, "bf16", out_dt, 1e-6, has_bias=True)
    row_case(pkg, wl, None, host=True)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4", "nvfp4"])
@pytest.mark.parametrize("T,H", [(37, 2048), (1, 5120), (130, 7168)])
def test_block_formats_write_only_their_outputs(pkg, fmt, T, H):
    wl = synth.Workload(f"guard_{fmt}", T, H, 98, "bf16", "bf16", 1e-6, has_bias=True)
    inp = synth.make_inputs(wl)
    x, r, w, b = (inp[k].cuda() for k in ("x", "residual", "weight", "bias"))
    code, blk, per_byte = pkg.BLOCK_FORMATS[fmt]
    flags = pkg.make_flags("bf16", "f32", True, True, True)
    cfgs = pkg.block_format_configs(T, H, fmt)
    s = torch.cuda.current_stream().cuda_stream
    for c in [None] + cfgs:
        q = Guarded((T, H // per_byte), torch.uint8)
        bs = Guarded((T, H // blk), torch.uint8)
        ts = Guarded((T,), torch.float32) if fmt == "nvfp4" else None
        ro = Guarded((T, H), torch.bfloat16)
        st = pkg.rmsnorm_fwd_blockscaled(p(x), p(r), p(w), p(b), p(q.t), p(bs.t),
                                         None if ts is None else p(ts.t), p(ro.t), T, H, wl.eps,
                                         flags, code, 0.0, c, s)
        assert st == pkg.RMSN_OK
        for g in (q, bs, ts, ro):
            if g is not None:
                assert g.intact(), f"{fmt} {None if c is None else c.as_dict()}"
    assert pkg.rmsnorm_read_status() == 0
