"""Benchmark of the fused residual-add + RMSNorm on GB300.

One step = one rmsnorm_fwd call over the prefill workload (16384 tokens x
8192 hidden, bf16, residual + weight, eps 1e-5): reads x and residual, writes
residual_out and y.  Prints ONE JSON line on rank 0:

  value      algorithmic HBM GB/s of the whole job (all ranks), inputs resident
  e2e        the same metric through the public API with pinned HOST buffers:
             every step moves x and residual in and y and residual_out out
             (rmsnorm_fwd_host; explicit copies around rmsnorm_fwd as context)
  roofline   the kernel's average launch duration (CUDA events on its stream)
             against the measured HBM copy peak
  decode     us per call at decode sizes (T in {1,8,32,128,256}, H 4096):
             L2-hot back-to-back, CUDA-graph replay, and graph replay of
             programmatic-dependent launches, next to the measured empty-kernel
             launch time
  quantized  per-token FP8 and block-scaled MXFP8 / MXFP4 / NVFP4 outputs on
             4096 x {5120, 7168} with bias, algorithmic GB/s
  qk_norm    per-head QK norm (one launch, fused qkv, in place) against the
             row norm on the head views (two launches), us per call
  cpu_baseline  the CPU oracle on the host cores (rank 0, N = 1)

--out fp8 makes the timed step the quantised-output workload instead
(per-token FP8 E4M3 with bias; use --tokens 4096 --hidden 5120 or 7168).
A step whose bytes fit in L2 rotates over enough buffer sets to exceed it.

--impl reference times the CPU oracle instead (the only reference of this
method), on a bounded row sample per step.

Multi-GPU: rows are independent, so each rank runs its own full-size slice
of one seeded global batch (weak scaling, no collective on the data path); a
barrier and a MAX all-reduce of the elapsed time bracket the timed region.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused add+RMSNorm HBM GB/s (fraction of GB300 peak); us/call at decode sizes"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 10**6


def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# The measured selector table only picks launch shapes; a recorded capture is
# keyed by the full launch shape instead, so the table is not part of the hash.
SELECTION_DATA = ("rmsn_selector_table.inc",)


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "residual_add_rmsnorm_vec_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if fn in SELECTION_DATA:
            continue
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(variant_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources and the same launch shape."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    e = d.get(variant_key)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return int(e["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts + frac, float(parts[1]), float(parts[2]), parts[3], parts[5:9]))
            except Exception:
                continue
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[4]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use), "reasons": reasons,
                "samples": len(use), "in_region": bool(inside)}


def dist_setup(n_gpus: int):
    world = env_int("WORLD_SIZE", 1)
    rank = env_int("RANK", 0)
    local = env_int("LOCAL_RANK", 0)
    if n_gpus > 1 and world != n_gpus:
        raise SystemExit(f"--gpus {n_gpus} needs torchrun with {n_gpus} ranks (WORLD_SIZE={world})")
    pg = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=None)
        pg = dist
    return rank, local, world, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, v: float, device) -> float:
    if pg is None:
        return v
    import torch

    t = torch.tensor([v], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(pg, v: float, device) -> float:
    if pg is None:
        return v
    import torch

    t = torch.tensor([v], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.SUM)
    return float(t.item())


def aggregate(pg, elapsed_ms: float, bytes_rank: float, device):
    """Whole-job throughput: bytes of all ranks over the slowest rank's time.
    Returns (max elapsed ms, total bytes, GB/s)."""
    max_ms = max_over_ranks(pg, elapsed_ms, device)
    total = sum_over_ranks(pg, bytes_rank, device)
    return max_ms, total, total / (max_ms / 1e3) / 1e9


def rank_rows(rank: int, world: int, tokens_per_rank: int) -> range:
    """Rows of the global batch (world x tokens_per_rank tokens) owned by a rank."""
    return range(rank * tokens_per_rank, (rank + 1) * tokens_per_rank)


# ---------------------------------------------------------------------------- our arm


def step_workload(synth, args, n_tokens):
    """The timed step's workload: the bf16 prefill (default) or, with
    --out fp8, the per-token FP8 output with bias (4096 x 5120 / 7168)."""
    if args.out == "fp8":
        return synth.fp8_workload(args.hidden, n_tokens=n_tokens)
    return synth.prefill_workload(n_tokens, args.hidden)


NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal (the ~8 TB/s the prefill gate is stated against)


def step_config(wl, world: int) -> dict:
    """The `config` object of the JSON line: the workload only, with the same
    keys and values in both arms (timing details and the launch shape go in
    their own keys)."""
    return {"workload": workload_name(wl), "n_tokens": wl.n_tokens, "hidden": wl.hidden,
            "global_batch_tokens": wl.n_tokens * world,
            "parallelism": f"rows sharded, {world} independent replica(s)"}


def workload_name(wl) -> str:
    if wl.out_dtype == "fp8":
        return (f"fused residual-add + RMSNorm bf16 -> per-token FP8 E4M3 with bias "
                f"T={wl.n_tokens} H={wl.hidden} eps=1e-6")
    return f"prefill fused residual-add + RMSNorm bf16 T={wl.n_tokens} H={wl.hidden} eps=1e-5"


def run_ours(args):
    import torch

    import residual_add_rmsnorm_vec_gb300 as pkg
    from residual_add_rmsnorm_vec_gb300 import build, synth

    rank, local, world, pg = dist_setup(args.gpus)
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    build.build()

    # each rank owns a contiguous slice of one seeded global batch (weak scaling)
    wl = step_workload(synth, args, args.tokens)
    wl_global = step_workload(synth, args, args.tokens * world)
    T, H = wl.n_tokens, wl.hidden
    fp8 = wl.out_dtype == "fp8"
    flags = pkg.make_flags("bf16", wl.out_dtype, True, True, wl.has_bias)
    # consecutive steps are chained by programmatic dependent launch: a step's
    # grid is scheduled while the previous one drains and waits for it to
    # complete before its first read
    step_flags = flags if args.no_pdl else flags | pkg.RMSN_PDL
    host = synth.make_inputs(wl_global, rows=rank_rows(rank, world, T))
    w = host["weight"].to(dev)
    b = host["bias"].to(dev) if wl.has_bias else None
    # a step whose bytes fit in L2 rotates over enough copies of its buffers
    # that consecutive steps never find their inputs in L2
    bytes_step = wl.algorithmic_bytes()
    n_sets = max(1, -(-3 * L2_BYTES // bytes_step)) if bytes_step < 3 * L2_BYTES else 1
    sets = []
    for k in range(n_sets):
        x = host["x"].to(dev)
        r = host["residual"].to(dev)
        out = torch.empty((T, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
        res = torch.empty_like(x)
        scale = torch.empty((T,), dtype=torch.float32, device=dev) if fp8 else None
        sets.append((x.data_ptr(), r.data_ptr(), w.data_ptr(), None if b is None else b.data_ptr(),
                     out.data_ptr(), res.data_ptr(), None if scale is None else scale.data_ptr(),
                     (x, r, out, res, scale)))
    forced = None
    if args.config:
        forced = pkg.RmsnConfig.from_dict(json.loads(args.config))
    cfg = forced if forced is not None else pkg.rmsnorm_query_config(T, H, step_flags)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    def step(i):
        ptrs = sets[i % n_sets][:7]
        if forced is None:
            st = pkg.rmsnorm_fwd(*ptrs, T, H, wl.eps, step_flags, sptr)
        else:
            st = pkg.rmsnorm_fwd_ex(*ptrs, T, H, wl.eps, step_flags, 0.0, forced, sptr)
        if st != pkg.RMSN_OK:
            raise pkg.RmsnError(st, "rmsnorm_fwd")

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    K = args.steps
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    time.sleep(0.2)
    barrier(pg)
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    t_start.record(stream)
    for i in range(K):
        step(i)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    barrier(pg)
    clocks = sampler.stop(wall0, wall1)
    # the timed region holds only the K launches: its length / K is the
    # kernel's average launch duration, gaps between launches included
    kernel_ms = t_start.elapsed_time(t_end) / K
    elapsed_ms, total_bytes, value = aggregate(pg, t_start.elapsed_time(t_end),
                                               float(bytes_step * K), dev)

    # e2e: pinned host buffers, copies inside the timed region, every step
    e2e = run_e2e(pkg, wl, host, dev, stream, flags, max(3, min(K, args.e2e_steps)), pg)

    decode = None if args.skip_decode else run_decode(pkg, synth, dev, stream)
    qk = None if args.skip_decode else run_qk(pkg, synth, dev, stream)
    quant = None if args.skip_decode else run_quantized(pkg, synth, dev, stream)
    dtypes = None if args.skip_decode else run_dtype_paths(pkg, dev, stream, T, H)

    peak, peak_src = load_peaks()
    achieved = bytes_step / (kernel_ms / 1e3) / 1e9
    box_peak = copy_peak_same_box(dev)
    vkey = (f"{pkg.VARIANT_NAMES[cfg.variant]}_ch{cfg.chunks}_w{cfg.warps_per_block}"
            f"_st{cfg.stages}_g{cfg.grid}_T{T}_H{H}")
    if fp8:
        vkey += "_fp8"
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": ("synthetic, seeded: x, residual ~ N(0,1), weight = 1 + 0.1 N(0,1), "
                 "bias = 0.01 N(0,1)") if fp8 else
                ("synthetic, seeded: x ~ N(0,1) with 1% outlier channels x50, residual ~ N(0,4), "
                 "weight = 1 + 0.1 N(0,1)"),
        "config": step_config(wl, world),
        "l2": (f"inputs larger than L2 ({2 * T * H * 2 / 2**20:.0f} MiB read per step "
               f"vs {L2_BYTES / 1e6:.0f} MB L2), no flush") if n_sets == 1 else
              (f"{n_sets} rotating buffer sets of {bytes_step / 2**20:.0f} MiB per step "
               f"({n_sets * bytes_step / 2**20:.0f} MiB vs {L2_BYTES / 1e6:.0f} MB "
               f"L2), no flush"),
        "launch": dict(cfg.as_dict(), pdl=not args.no_pdl),
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": K,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "peak_nominal": NOMINAL_HBM_GBS,
                     "peak_same_box": round(box_peak, 1),
                     "frac_same_box": round(achieved / box_peak, 4),
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                     else "fallback 6.8 TB/s",
                     "traffic": recorded_traffic(vkey),
                     "algorithmic_bytes": bytes_step, "kernel": vkey,
                     "avg_launch_us": round(kernel_ms * 1e3, 3)},
    }
    if decode is not None:
        line["decode"] = decode
    if qk is not None:
        line["qk_norm"] = qk
    if quant is not None:
        line["quantized"] = quant
    if dtypes is not None:
        line["dtype_paths"] = dtypes
    if rank == 0 and world == 1 and not args.skip_cpu:
        line["cpu_baseline"] = run_cpu_baseline(wl, host, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def copy_peak_same_box(dev) -> float:
    """HBM copy bandwidth on this GPU, now: torch copy_ of 1 Gi bf16 elements,
    read + write bytes, best of 10 (the method of the measured-peaks record,
    repeated here so the kernel can also be put against its own box)."""
    import torch

    n = 1 << 30
    a = torch.empty(n, dtype=torch.bfloat16, device=dev)
    b = torch.empty_like(a)
    a.fill_(1.0)
    best = float("inf")
    for _ in range(12):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        b.copy_(a)
        e1.record()
        torch.cuda.synchronize(dev)
        best = min(best, e0.elapsed_time(e1))
    del a, b
    torch.cuda.empty_cache()
    return 2 * n * 2 / (best / 1e3) / 1e9


def run_e2e(pkg, wl, host, dev, stream, flags, steps, pg):
    """Host to host through the public API, every step: the rows start in
    page-locked host memory and the results end there.

    Headline: rmsnorm_fwd_host, where the kernel itself reads x, residual and
    weight across the CPU-GPU link and writes y and residual_out back (no
    staging copy).  For context, ``copies``: the same step as an explicit
    host-to-device copy, rmsnorm_fwd on device buffers, device-to-host copy,
    all on one stream.
    """
    import torch

    T, H = wl.n_tokens, wl.hidden
    fp8 = wl.out_dtype == "fp8"
    hx = host["x"].pin_memory()
    hr = host["residual"].pin_memory()
    hw = host["weight"].pin_memory()
    hb = host["bias"].pin_memory() if wl.has_bias else None
    hy = torch.empty((T, H), dtype=torch.uint8 if fp8 else torch.bfloat16).pin_memory()
    hres = torch.empty_like(hx).pin_memory()
    hsc = torch.empty((T,), dtype=torch.float32).pin_memory() if fp8 else None
    sptr = stream.cuda_stream

    def p(t):
        return None if t is None else t.data_ptr()

    hptrs = (hx.data_ptr(), hr.data_ptr(), hw.data_ptr(), p(hb), hy.data_ptr(), hres.data_ptr(),
             p(hsc))

    def step_host():
        st = pkg.rmsnorm_fwd_host(*hptrs, T, H, wl.eps, flags, 0.0, sptr)
        if st != pkg.RMSN_OK:
            raise pkg.RmsnError(st, "rmsnorm_fwd_host")

    dx = torch.empty_like(hx, device=dev)
    dr = torch.empty_like(hx, device=dev)
    dw = torch.empty_like(hw, device=dev)
    db = None if hb is None else torch.empty_like(hb, device=dev)
    dy = torch.empty_like(hy, device=dev)
    dres = torch.empty_like(dx)
    dsc = None if hsc is None else torch.empty_like(hsc, device=dev)

    def step_copies():
        dx.copy_(hx, non_blocking=True)
        dr.copy_(hr, non_blocking=True)
        dw.copy_(hw, non_blocking=True)
        if db is not None:
            db.copy_(hb, non_blocking=True)
        pkg.fused_add_rmsnorm(dx, dr, dw, db, eps=wl.eps, out_dtype=wl.out_dtype, out=dy,
                              residual_out=dres, out_scale=dsc)
        hy.copy_(dy, non_blocking=True)
        hres.copy_(dres, non_blocking=True)
        if dsc is not None:
            hsc.copy_(dsc, non_blocking=True)

    def timed(step):
        for _ in range(2):
            step()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        barrier(pg)
        a.record(stream)
        for _ in range(steps):
            step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return max_over_ranks(pg, a.elapsed_time(b), dev)

    world = 1 if pg is None else pg.get_world_size()
    h2d = sum(t.numel() * t.element_size() for t in (hx, hr, hw, hb) if t is not None)
    d2h = sum(t.numel() * t.element_size() for t in (hy, hres, hsc) if t is not None)
    ms = timed(step_host)
    ms_copies = timed(step_copies)
    gbs = wl.algorithmic_bytes() * steps * world / (ms / 1e3) / 1e9
    gbs_copies = wl.algorithmic_bytes() * steps * world / (ms_copies / 1e3) / 1e9
    return {"value": round(gbs, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": round(ms / steps, 4),
            "api": "rmsnorm_fwd_host on page-locked host buffers (the kernel moves the bytes "
                   "over the CPU-GPU link)",
            "copies": {"value": round(gbs_copies, 1), "ms_per_step": round(ms_copies / steps, 4),
                       "api": "cudaMemcpyAsync in, rmsnorm_fwd, cudaMemcpyAsync out"}}


def host_cost_c(T: int, H: int, n: int = 3000, extra_flags: int = 0) -> dict:
    """The library's host cost per rmsnorm_fwd call, and an empty kernel's,
    both timed in a C loop (the bench's harness library; no Python in the
    loop): host enqueue time and GPU time per call, back to back."""
    import ctypes

    from residual_add_rmsnorm_vec_gb300 import build

    lib = ctypes.CDLL(build.HOSTCOST_PATH)
    lib.rmsn_host_cost.restype = ctypes.c_int
    lib.rmsn_host_cost.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32,
                                   ctypes.POINTER(ctypes.c_double)]
    out = (ctypes.c_double * 4)()
    st = lib.rmsn_host_cost(T, H, n, extra_flags, out)
    if st != 0:
        raise RuntimeError(f"rmsn_host_cost failed with {st}")
    return {"empty_host_us": round(out[0], 3), "empty_gpu_us": round(out[1], 3),
            "lib_host_us": round(out[2], 3), "lib_gpu_us": round(out[3], 3)}


def run_decode(pkg, synth, dev, stream):
    """us per call at decode sizes (inputs L2-resident), back-to-back and in a
    CUDA graph, and the same for an empty kernel (torch.cuda._sleep(0)) and,
    in a graph, for torch's add of the same two inputs."""
    import torch

    res = {"hidden": 4096, "unit": "us/call"}
    n = 2000

    def timeit(fn, reps):
        for _ in range(20):
            fn()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) * 1e3 / reps

    def graph_time(fn, per_graph=100, replays=20):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(dev)
        s.wait_stream(stream)
        with torch.cuda.stream(s):
            fn()
            torch.cuda.synchronize(dev)
            with torch.cuda.graph(g, stream=s):
                for _ in range(per_graph):
                    fn()
        stream.wait_stream(s)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(replays):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) * 1e3 / (replays * per_graph)

    def empty():
        torch.cuda._sleep(0)

    res["empty_kernel_us"] = round(timeit(empty, n), 3)
    res["empty_kernel_graph_us"] = round(graph_time(empty), 3)
    flags = pkg.make_flags("bf16", "bf16", True, True, False)
    per_t = {}
    for T in synth.DECODE_TOKENS:
        wl = synth.decode_workload(T)
        inp = synth.make_inputs(wl)
        x = inp["x"].to(dev)
        r = inp["residual"].to(dev)
        w = inp["weight"].to(dev)
        out = torch.empty_like(x)
        ro = torch.empty_like(x)
        ptrs = (x.data_ptr(), r.data_ptr(), w.data_ptr(), None, out.data_ptr(), ro.data_ptr(),
                None)

        def call(fl=flags):
            st = pkg.rmsnorm_fwd(*ptrs, T, 4096, wl.eps, fl, torch.cuda.current_stream().cuda_stream)
            if st != pkg.RMSN_OK:
                raise pkg.RmsnError(st, "rmsnorm_fwd")

        def call_pdl():
            call(flags | pkg.RMSN_PDL | pkg.RMSN_PDL_EARLY_PARAMS)

        us = timeit(call, n)
        gus = graph_time(call)
        gus_pdl = graph_time(call_pdl)
        # the split-row cluster variant, each built cluster size, in graphs
        clusters = {}
        for c in pkg.rmsnorm_list_configs(T, 4096, flags):
            if c.variant != pkg.VARIANT_CLUSTER:
                continue

            def call_c(fl=flags, c=c):
                st = pkg.rmsnorm_fwd_ex(*ptrs, T, 4096, wl.eps, fl, 0.0, c,
                                        torch.cuda.current_stream().cuda_stream)
                if st != pkg.RMSN_OK:
                    raise pkg.RmsnError(st, "rmsnorm_fwd_ex")

            clusters[f"k{c.cluster}_ch{c.chunks}"] = {
                "graph_us": round(graph_time(call_c), 3),
                "graph_pdl_us": round(graph_time(
                    lambda c=c: call_c(flags | pkg.RMSN_PDL | pkg.RMSN_PDL_EARLY_PARAMS, c)), 3)}
        hc = host_cost_c(T, 4096)
        # floor for comparison: torch's elementwise add of the same x and r
        # (reads both, writes one tensor; no reduction), in a graph likewise
        gus_add = graph_time(lambda: torch.add(x, r, out=out))
        cfg = pkg.rmsnorm_query_config(T, 4096, flags)
        cfg_pdl = pkg.rmsnorm_query_config(T, 4096, flags | pkg.RMSN_PDL)
        per_t[str(T)] = {"us": round(us, 3), "graph_us": round(gus, 3),
                         "graph_pdl_us": round(gus_pdl, 3),
                         "torch_add_graph_us": round(gus_add, 3),
                         "host_us_c": hc["lib_host_us"], "gpu_us_c": hc["lib_gpu_us"],
                         "cluster": clusters,
                         "gbs_l2_hot": round(wl.algorithmic_bytes() / (us * 1e-6) / 1e9, 1),
                         "launch": f"{pkg.VARIANT_NAMES[cfg.variant]} ch{cfg.chunks} "
                                   f"w{cfg.warps_per_block} grid{cfg.grid}",
                         "launch_pdl": f"{pkg.VARIANT_NAMES[cfg_pdl.variant]} ch{cfg_pdl.chunks} "
                                       f"w{cfg_pdl.warps_per_block} st{cfg_pdl.stages} "
                                       f"grid{cfg_pdl.grid}"}
    res["tokens"] = per_t
    # an empty kernel launched from the same C loop (host cost, GPU time per launch)
    hc = host_cost_c(1, 4096)
    res["empty_kernel_host_us_c"] = hc["empty_host_us"]
    res["empty_kernel_gpu_us_c"] = hc["empty_gpu_us"]
    res["gate"] = "us/call <= 2x empty-kernel launch"
    res["within_2x_launch"] = all(v["us"] <= 2 * res["empty_kernel_us"] for v in per_t.values())
    res["within_2x_launch_graph"] = all(v["graph_us"] <= 2 * res["empty_kernel_graph_us"]
                                        for v in per_t.values())
    res["within_2x_launch_graph_pdl"] = all(v["graph_pdl_us"] <= 2 * res["empty_kernel_graph_us"]
                                            for v in per_t.values())
    return res


def run_qk(pkg, synth, dev, stream):
    """QK norm (per-head, in place) on Qwen3-8B-like heads (32 query, 8 key,
    head_dim 128, bf16): one rmsnorm_qk_fwd launch on a fused qkv buffer
    against the regular row norm applied to the query and key head views
    (two rmsnorm_fwd launches).  CUDA-graph replay, us per call.  From 16384
    tokens the launches alternate over two buffer sets (the q and k heads of
    one set alone exceed L2), so those figures are HBM-bound and are also
    given as a fraction of the measured copy peak."""
    import torch

    Hq, Hk, D = 32, 8, 128
    peak, _ = load_peaks()
    out = {"heads": f"{Hq} q + {Hk} k heads x {D}, bf16", "unit": "us/call"}
    for T in (1, 64, 512, 1024, 4096, 16384):
        inp = synth.qk_inputs(T, Hq, Hk, D, "bf16")
        n_sets = 2 if T >= 16384 else 1
        wq, wk = inp["q_weight"].to(dev), inp["k_weight"].to(dev)
        sets = []
        for _ in range(n_sets):
            qkv = inp["qkv"].to(dev)
            q = qkv[:, :Hq * D]
            k = qkv[:, Hq * D:(Hq + Hk) * D]
            sets.append((qkv, q, k, q.contiguous(), k.contiguous()))
        fl = pkg.make_flags("bf16", "bf16", False, True, False)

        def qk_call(i, variant=None, pdl=False):
            _, q, k, _, _ = sets[i % n_sets]
            pkg.qk_norm_(q, k, wq, wk, head_dim=D, eps=1e-6, variant=variant, pdl=pdl)

        def rows_call(i):
            _, _, _, qc, kc = sets[i % n_sets]
            s = torch.cuda.current_stream().cuda_stream
            for t, w, h in ((qc, wq, Hq), (kc, wk, Hk)):
                st = pkg.rmsnorm_fwd(t.data_ptr(), None, w.data_ptr(), None, t.data_ptr(), None,
                                     None, T * h, D, 1e-6, fl, s)
                if st != pkg.RMSN_OK:
                    raise pkg.RmsnError(st, "rmsnorm_fwd")

        def graph_us(fn, per_graph=50, replays=10):
            fn(0)
            torch.cuda.synchronize(dev)
            g = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream(dev)
            s.wait_stream(stream)
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    for i in range(per_graph):
                        fn(i)
            stream.wait_stream(s)
            g.replay()
            torch.cuda.synchronize(dev)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(replays):
                g.replay()
            b.record(stream)
            torch.cuda.synchronize(dev)
            return a.elapsed_time(b) * 1e3 / (replays * per_graph)

        nbytes = 2 * T * (Hq + Hk) * D * 2 + 2 * D * 2
        us_qk = graph_us(qk_call)
        us_rows = graph_us(rows_call)
        # both QK kernels forced: the ring variant and the one-pass register kernel
        us_ring = graph_us(lambda i: qk_call(i, "ring"))
        us_direct = graph_us(lambda i: qk_call(i, "direct"))
        # consecutive launches chained by programmatic dependent launch
        us_pdl = graph_us(lambda i: qk_call(i, pdl=True))
        res = {"qk_us": round(us_qk, 3), "qk_gbs": round(nbytes / us_qk / 1e3, 1),
               "row_norm_us": round(us_rows, 3),
               "row_norm_gbs": round(nbytes / us_rows / 1e3, 1),
               "speedup": round(us_rows / us_qk, 2),
               "ring_us": round(us_ring, 3), "direct_us": round(us_direct, 3),
               "pdl_us": round(us_pdl, 3)}
        if n_sets > 1:
            res["qk_frac_of_peak"] = round(nbytes / us_qk / 1e3 / peak, 4)
            res["qk_pdl_frac_of_peak"] = round(nbytes / us_pdl / 1e3 / peak, 4)
            res["buffer_sets"] = n_sets
            # torch's elementwise y = x * 1 over the same bytes (the q and k
            # heads' worth, read once and written once) in the same graph
            # method: the rate one launch of this size reaches, launch and
            # drain included
            n_el = T * (Hq + Hk) * D
            els = [(torch.empty(n_el, dtype=torch.bfloat16, device=dev).fill_(1.0),
                    torch.empty(n_el, dtype=torch.bfloat16, device=dev)) for _ in range(n_sets)]
            us_el = graph_us(lambda i: torch.mul(els[i % n_sets][0], 1.0, out=els[i % n_sets][1]))
            del els
            res["elementwise_same_bytes_us"] = round(us_el, 3)
            res["qk_vs_elementwise_same_bytes"] = round(us_el / us_qk, 4)
        out[f"T{T}"] = res
        del sets
    torch.cuda.empty_cache()
    return out


def run_quantized(pkg, synth, dev, stream):
    """Quantised outputs on the FP8 configuration's shapes (4096 tokens x
    hidden 5120 / 7168, bf16 x and residual, weight and bias): per-token FP8
    and the block-scaled MXFP8 / MXFP4 / NVFP4.  CUDA-graph replay of
    launches alternating over two input sets (above the L2 size), plain and
    chained by programmatic dependent launch; algorithmic GB/s."""
    import torch

    out = {"unit": "GB/s", "timing": "cuda graph, 2 rotating input sets; *_pdl: launches "
                                      "chained by programmatic dependent launch"}

    def graph_us(call, n=20, replays=5):
        for i in range(2):
            call(i)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(dev)
        s.wait_stream(stream)
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for i in range(n):
                    call(i)
        stream.wait_stream(s)
        g.replay()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(replays):
            g.replay()
        e.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(e) * 1e3 / (replays * n)

    # the workload's 4096 tokens, all four formats; 16384 tokens (per-token FP8
    # and NVFP4) shows the rate once a launch's fixed costs are spread thinner
    runs = [(4096, H, ("fp8", "mxfp8", "mxfp4", "nvfp4")) for H in synth.FP8_HIDDEN]
    runs += [(16384, H, ("fp8", "nvfp4")) for H in synth.FP8_HIDDEN]
    for T, H, fmts in runs:
        wl = synth.fp8_workload(H, n_tokens=T)
        inp = synth.make_inputs(wl)
        sets = []
        for k in range(2):
            x = inp["x"].to(dev) if k == 0 else inp["x"].to(dev).flip(0).contiguous()
            r = inp["residual"].to(dev) if k == 0 else inp["residual"].to(dev).flip(0).contiguous()
            sets.append((x, r, torch.empty_like(x)))
        w, b = inp["weight"].to(dev), inp["bias"].to(dev)
        res = {}
        for fmt in fmts:
            if fmt == "fp8":
                bufs = [(torch.empty((T, H), dtype=torch.uint8, device=dev),
                         torch.empty((T,), dtype=torch.float32, device=dev)) for _ in sets]
                nbytes = wl.algorithmic_bytes()

                def call(i, pdl=False, bufs=bufs):
                    x, r, ro = sets[i % 2]
                    q, sc = bufs[i % 2]
                    pkg.fused_add_rmsnorm(x, r, w, b, eps=wl.eps, out_dtype="fp8", out=q,
                                          residual_out=ro, out_scale=sc, pdl=pdl)
            else:
                code, blk, per_byte = pkg.BLOCK_FORMATS[fmt]
                nbytes = (T * H * 2 * 3 + T * H // per_byte + T * H // blk + 4 * H
                          + (4 * T if fmt == "nvfp4" else 0))
                flags = pkg.make_flags("bf16", "f32", True, True, True)
                bufs = [(torch.empty((T, H // per_byte), dtype=torch.uint8, device=dev),
                         torch.empty((T, H // blk), dtype=torch.uint8, device=dev),
                         torch.empty((T,), dtype=torch.float32, device=dev)) for _ in sets]

                def call(i, pdl=False, bufs=bufs, code=code, fmt=fmt, flags=flags):
                    x, r, ro = sets[i % 2]
                    q, bs, ts = bufs[i % 2]
                    st = pkg.rmsnorm_fwd_blockscaled(
                        x.data_ptr(), r.data_ptr(), w.data_ptr(), b.data_ptr(), q.data_ptr(),
                        bs.data_ptr(), ts.data_ptr() if fmt == "nvfp4" else None, ro.data_ptr(),
                        T, H, wl.eps, flags | (pkg.RMSN_PDL if pdl else 0), code, 0.0, None,
                        torch.cuda.current_stream().cuda_stream)
                    if st != pkg.RMSN_OK:
                        raise pkg.RmsnError(st, "rmsnorm_fwd_blockscaled")
            us = graph_us(call)
            us_pdl = graph_us(lambda i, call=call: call(i, pdl=True))
            res[fmt] = {"us": round(us, 2), "gbs": round(nbytes / us / 1e3, 1),
                        "us_pdl": round(us_pdl, 2), "gbs_pdl": round(nbytes / us_pdl / 1e3, 1)}
        # torch's elementwise y = x * 1 moving the per-token FP8 step's bytes
        # (half read, half written), two rotating sets, the same graph
        # method: the rate one launch of this size reaches, launch and drain
        # included
        nb = wl.algorithmic_bytes()
        els = [(torch.empty(nb // 4, dtype=torch.bfloat16, device=dev).fill_(1.0),
                torch.empty(nb // 4, dtype=torch.bfloat16, device=dev)) for _ in range(2)]
        us_el = graph_us(lambda i: torch.mul(els[i % 2][0], 1.0, out=els[i % 2][1]))
        res["elementwise_same_bytes"] = {"us": round(us_el, 2), "gbs": round(nb / us_el / 1e3, 1)}
        del els
        out[f"T{T}_H{H}"] = res
        del sets, inp
        torch.cuda.empty_cache()
    return out


def run_dtype_paths(pkg, dev, stream, T=16384, H=8192, n=200):
    """The other storage types of the prefill step at the bench shape: fp16
    in and out, and bf16 / fp16 activations over an fp32 residual stream.
    Seeded device inputs above the L2 size, the selector's launch, n eager
    launches back to back between two CUDA events; algorithmic GB/s."""
    import torch

    gen = torch.Generator(device=dev)
    gen.manual_seed(60)
    out = {"unit": "GB/s", "tokens": T, "hidden": H,
           "timing": f"{n} launches back to back, selector's launch, no PDL"}
    for name, act, res_dt in (("f16", torch.float16, torch.float16),
                              ("bf16_act_f32_stream", torch.bfloat16, torch.float32),
                              ("f16_act_f32_stream", torch.float16, torch.float32)):
        x = torch.randn((T, H), device=dev, generator=gen).to(act)
        r = (2 * torch.randn((T, H), device=dev, generator=gen)).to(res_dt)
        w = (1 + 0.1 * torch.randn((H,), device=dev, generator=gen)).to(act)
        y, ro = torch.empty_like(x), torch.empty_like(r)

        def call():
            pkg.fused_add_rmsnorm(x, r, w, None, eps=1e-5, out=y, residual_out=ro)

        for _ in range(5):
            call()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            call()
        e.record(stream)
        torch.cuda.synchronize(dev)
        us = a.elapsed_time(e) * 1e3 / n
        nbytes = T * H * (2 * x.element_size() + 2 * r.element_size()) + H * w.element_size()
        flags = pkg.make_flags("f16" if act == torch.float16 else "bf16",
                               "f16" if act == torch.float16 else "bf16", True, True, False)
        if res_dt == torch.float32:
            flags |= pkg.RMSN_RESIDUAL_F32
        cfg = pkg.rmsnorm_query_config(T, H, flags)
        out[name] = {"us": round(us, 2), "gbs": round(nbytes / us / 1e3, 1),
                     "algorithmic_bytes": nbytes,
                     "launch": f"{pkg.VARIANT_NAMES[cfg.variant]} ch{cfg.chunks} "
                               f"w{cfg.warps_per_block} st{cfg.stages} grid{cfg.grid}"}
        del x, r, w, y, ro
    torch.cuda.empty_cache()
    return out


def run_cpu_baseline(wl, host, seconds: float) -> dict:
    """The oracle as it stands, on every host core, over the whole workload
    (repeated until `seconds` have passed); and on one thread over the first
    1024 rows (repeated for a quarter of that time)."""
    import oracle

    cores = oracle.num_cpus()
    eps = float(np.float32(wl.eps))

    def timed(x, r, threads, budget):
        reps, t0 = 0, time.time()
        while True:
            oracle.rmsnorm(x, r, host["weight"], host["bias"], eps=eps, in_dtype="bf16",
                           out_dtype=wl.out_dtype, n_threads=threads)
            reps += 1
            if time.time() - t0 >= budget or reps >= 50:
                return reps, time.time() - t0

    reps, dt = timed(host["x"], host["residual"], cores, seconds)
    rows = min(1024, wl.n_tokens)
    reps1, dt1 = timed(host["x"][:rows], host["residual"][:rows], 1, seconds / 4)
    row_bytes = wl.algorithmic_bytes() / wl.n_tokens
    return {"value": round(wl.algorithmic_bytes() * reps / dt / 1e9, 3), "unit": UNIT,
            "cores": cores, "kind": "oracle",
            "sample": f"full {wl.n_tokens}x{wl.hidden} workload x {reps} passes ({dt:.1f} s), "
                      f"fp64 C oracle, {cores} threads",
            "single_thread": {"value": round(row_bytes * rows * reps1 / dt1 / 1e9, 3),
                              "unit": UNIT, "cores": 1,
                              "sample": f"first {rows} rows x {reps1} passes ({dt1:.1f} s)"}}


# ---------------------------------------------------------------------------- reference arm


def run_reference(args):
    rank = env_int("RANK", 0)
    if rank != 0:
        return
    import oracle
    from residual_add_rmsnorm_vec_gb300 import synth

    wl = step_workload(synth, args, args.tokens)
    T, H = wl.n_tokens, wl.hidden
    cores = oracle.num_cpus()
    eps = float(np.float32(wl.eps))
    # calibrate rows per step so that warmup + steps fit the time budget
    probe_rows = synth.sample_rows(T, 64)
    probe = synth.make_inputs(wl, rows=probe_rows)
    t0 = time.time()
    oracle.rmsnorm(probe["x"], probe["residual"], probe["weight"], probe["bias"], eps=eps,
                   in_dtype="bf16", out_dtype=wl.out_dtype, n_threads=cores)
    per_row = max((time.time() - t0) / len(probe_rows), 1e-7)
    n_steps = args.steps + args.warmup
    rows = int(max(1, min(T, args.ref_seconds / n_steps / per_row)))
    sample = synth.sample_rows(T, rows)
    inp = synth.make_inputs(wl, rows=sample)
    for _ in range(args.warmup):
        oracle.rmsnorm(inp["x"], inp["residual"], inp["weight"], inp["bias"], eps=eps,
                       in_dtype="bf16", out_dtype=wl.out_dtype, n_threads=cores)
    t0 = time.time()
    for _ in range(args.steps):
        oracle.rmsnorm(inp["x"], inp["residual"], inp["weight"], inp["bias"], eps=eps,
                       in_dtype="bf16", out_dtype=wl.out_dtype, n_threads=cores)
    dt = time.time() - t0
    bytes_step = wl.algorithmic_bytes() * len(sample) // T
    value = bytes_step * args.steps / dt / 1e9
    sample_txt = (f"{len(sample)} seeded rows of the {T}x{H} workload per step, fp64 C oracle, "
                  f"{cores} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic, seeded",
        "config": step_config(wl, args.gpus),
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores,
                         "kind": "oracle", "sample": sample_txt},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=6000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--tokens", type=int, default=16384)
    ap.add_argument("--hidden", type=int, default=8192)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--out", choices=["bf16", "fp8"], default="bf16",
                    help="output of the timed step: bf16 (the prefill workload) or per-token "
                         "FP8 with bias (use --tokens 4096 --hidden 5120 or 7168)")
    ap.add_argument("--skip-decode", action="store_true")
    ap.add_argument("--no-pdl", action="store_true",
                    help="launch the timed prefill steps without programmatic dependent launch")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--config", default="",
                    help='force a launch configuration, JSON such as '
                         '{"variant": 2, "chunks": 2, "max_warps": 32, "stages": 4}')
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
