"""Measure every built launch configuration over a tokens x hidden grid and
write the selector table (csrc/rmsn_selector_table.inc) from the fastest.

The blog "CuTeDSL at Perplexity" (section "Prefill and decode") picks the warp
count per block by benchmarking 8/16/32 warps until the bandwidth stops
improving; this does the same for every variant the library builds (one warp
per row, one block per row, bulk-copy ring depths, grid shapes) on the
current GPU.

Timing: `reps` back-to-back launches are captured in a CUDA graph and the
graph is replayed; the time per launch is the replay time (CUDA events on
the replay stream) over the launches, median of several replays, so host
launch overhead does not enter.  When one set of buffers is smaller than
3 x the L2 size the launches rotate over enough copies to exceed it, so the
figures are HBM (not L2) bandwidth; with --l2-hot one set is reused (the
decode situation, where the activations of a few tokens stay on chip).

    python -m residual_add_rmsnorm_vec_gb300.tune --out sweep.json --write-table
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import time

L2_BYTES = 129 * 10**6
TOKENS = (1, 4, 16, 64, 256, 1024, 4096, 16384, 65536)
HIDDEN = (2048, 4096, 8192, 16384)
# table keys; "+r32": bf16 / fp16 activations over an fp32 residual stream
DTYPE_CODES = {"f32": 0, "bf16": 1, "fp8": 2, "mxfp8": 3, "mxfp4": 4, "nvfp4": 5, "f16": 6,
               "bf16+r32": 7, "f16+r32": 8, "bf16+pdl": 9}
BLOCK_FMTS = ("mxfp8", "mxfp4", "nvfp4")


def _algorithmic_bytes(T, H, in_b, out_b, res, bias, fp8, fmt=None, res_b=None):
    if fmt in BLOCK_FMTS:
        blk, per_byte = (16, 2) if fmt == "nvfp4" else (32, 1 if fmt == "mxfp8" else 2)
        b = T * H * in_b + T * H // per_byte + T * H // blk + H * in_b
        b += 4 * T if fmt == "nvfp4" else 0
    else:
        b = T * H * in_b + T * H * out_b + H * in_b
        if fp8:
            b += 4 * T
    if res:
        b += 2 * T * H * (in_b if res_b is None else res_b)
    if bias:
        b += H * in_b
    return b


def measure(pkg, T, H, in_dt="bf16", out_dt="bf16", res=True, bias=False, reps=30,
            configs=None, l2_hot=False, replays=5):
    import torch

    dev = torch.device("cuda")
    r32 = in_dt.endswith("+r32")
    pdl = in_dt.endswith("+pdl")  # launches chained by programmatic dependent launch
    in_dt = in_dt.split("+")[0]
    tin = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[in_dt]
    tres = torch.float32 if r32 else tin
    in_b = 4 if in_dt == "f32" else 2
    res_b = 4 if r32 else in_b
    block = out_dt in BLOCK_FMTS
    out_b = {"bf16": 2, "f16": 2, "f32": 4, "fp8": 1}.get(out_dt, 1)
    tout = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}.get(
        out_dt, torch.uint8)
    # block formats share the launch shapes of the per-token FP8 output
    rflag = pkg.RMSN_RESIDUAL_F32 if r32 else 0
    rflag |= pkg.RMSN_PDL if pdl else 0
    flags = pkg.make_flags(in_dt, "fp8" if block else out_dt, res, True, bias) | rflag
    call_flags = pkg.make_flags(in_dt, "f32", res, True, bias) | rflag if block else flags
    set_bytes = T * H * (in_b + (2 * res_b if res else 0) + out_b)
    n_sets = 1 if l2_hot else max(1, min(64, -(-3 * L2_BYTES // max(1, set_bytes))))
    sets = []
    for _ in range(n_sets):
        x = torch.randn(T, H, device=dev).to(tin)
        r = torch.randn(T, H, device=dev).to(tres) if res else None
        if block:
            code, blk, per_byte = pkg.BLOCK_FORMATS[out_dt]
            q = torch.empty(T, H // per_byte, device=dev, dtype=torch.uint8)
            bsc = torch.empty(T, H // blk, device=dev, dtype=torch.uint8)
        else:
            q, bsc = torch.empty(T, H, device=dev, dtype=tout), None
        sets.append((x, r, q, torch.empty_like(r) if res else None,
                     torch.empty(T, device=dev, dtype=torch.float32)
                     if out_dt in ("fp8", "nvfp4") else None, bsc))
    w = (1 + 0.1 * torch.randn(H, device=dev)).to(tin)
    b = (0.01 * torch.randn(H, device=dev)).to(tin) if bias else None
    stream = torch.cuda.current_stream()
    if configs is None:
        configs = (pkg.block_format_configs(T, H, out_dt, res, bias) if block
                   else pkg.rmsnorm_list_configs(T, H, flags))
    algo = _algorithmic_bytes(T, H, in_b, out_b, res, bias, out_dt == "fp8", out_dt, res_b)
    results = []
    for cfg in configs:
        def launch_on(i, s):
            x, r, o, ro, sc, bsc = sets[i % n_sets]
            ptr = (lambda t: None if t is None else t.data_ptr())
            if block:
                st = pkg.rmsnorm_fwd_blockscaled(
                    x.data_ptr(), ptr(r), w.data_ptr(), ptr(b), o.data_ptr(), bsc.data_ptr(),
                    ptr(sc), ptr(ro), T, H, 1e-6, call_flags, pkg.BLOCK_FORMATS[out_dt][0], 0.0,
                    cfg, s.cuda_stream)
            else:
                st = pkg.rmsnorm_fwd_ex(x.data_ptr(), ptr(r), w.data_ptr(), ptr(b), o.data_ptr(),
                                        ptr(ro), ptr(sc), T, H, 1e-6, flags, 0.0, cfg,
                                        s.cuda_stream)
            if st != pkg.RMSN_OK:
                raise pkg.RmsnError(st, "launch")

        def launch(i):
            launch_on(i, stream)

        for i in range(3):
            launch(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for i in range(reps):
                    launch_on(i, cap)
        stream.wait_stream(cap)
        g.replay()
        torch.cuda.synchronize()
        times = []
        for _ in range(replays):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3 / reps)
        del g
        us = statistics.median(times)
        d = cfg.as_dict()
        d.update(us=round(us, 3), gbs=round(algo / (us * 1e-6) / 1e9, 1))
        results.append(d)
    del sets
    torch.cuda.empty_cache()
    return results


def sweep(pkg, shapes, in_dt, out_dt, res, bias, reps, l2_hot_below=0):
    """``l2_hot_below``: shapes with fewer tokens are timed L2-hot (decode)."""
    out = []
    for T, H in shapes:
        t0 = time.time()
        rs = measure(pkg, T, H, in_dt, out_dt, res, bias, reps, l2_hot=T < l2_hot_below)
        best = min(rs, key=lambda d: d["us"])
        out.append({"T": T, "H": H, "in": in_dt, "out": out_dt, "res": res, "bias": bias,
                    "best": best, "all": rs})
        print(f"T={T:6d} H={H:6d} {in_dt}->{out_dt}: best {best['variant_name']} "
              f"ch{best['chunks']} w{best['warps_per_block']}/{best['max_warps']} "
              f"st{best['stages']} grid{best['grid']}: {best['us']:.2f} us {best['gbs']:.0f} GB/s"
              f"  ({len(rs)} configs, {time.time() - t0:.1f} s)", flush=True)
    return out


ROW_RE = (r"\s*\{(-?\d+), (-?\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+)"
          r"(?:, (\d+), (\d+))?\},(?:\s*// ([\d.]+) us, ([\d.]+) GB/s)?")


def fixed_rule_shape(T, H, sms, in_bytes=2):
    """(variant, chunks, max_warps) of the selector's fixed rules for a
    shape without table rows (the blog's decode rule, else one block per row
    with two vectors per thread): the fallback the nearest-measured-hidden
    lookup sits in front of, for comparison."""
    nvec = H * in_bytes // 32
    if (T * nvec + 31) // 32 <= sms and nvec <= 256:
        ch = 1
        while 32 * ch < nvec:
            ch *= 2
        return (0, ch, 1)
    for ch, wm in ((2, 4), (2, 8), (2, 16), (2, 32), (4, 16)):
        if (nvec + 32 * ch - 1) // (32 * ch) <= wm:
            return (1, ch, wm)
    return (3, 0, 8)


def check_selector(pkg, shapes, reps=30, l2_hot_below=512):
    """For each (T, H) (bf16 with a residual and a weight): every built launch
    timed, against the selector's pick and the fixed rules' pick."""
    import torch

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    flags = pkg.make_flags("bf16", "bf16", True, True, False)
    key = lambda d: (d["variant"], d["chunks"], d["max_warps"], d["stages"])
    out = []
    for T, H in shapes:
        rs = measure(pkg, T, H, "bf16", "bf16", True, False, reps, l2_hot=T < l2_hot_below)
        best = min(rs, key=lambda d: d["us"])
        sel = pkg.rmsnorm_query_config(T, H, flags).as_dict()
        sel_us = min((d["us"] for d in rs if key(d) == key(sel)), default=None)
        rule = fixed_rule_shape(T, H, sms)
        rule_us = min((d["us"] for d in rs if (d["variant"], d["chunks"], d["max_warps"]) == rule),
                      default=None)
        name = lambda d: (f"{d['variant_name']} ch{d['chunks']} w{d['warps_per_block']}"
                          f"/{d['max_warps']} st{d['stages']}")
        row = {"T": T, "H": H, "best": name(best), "best_us": best["us"], "selector": name(sel),
               "selector_us": sel_us, "rule": f"{pkg.VARIANT_NAMES[rule[0]]} ch{rule[1]}/{rule[2]}",
               "rule_us": rule_us,
               "selector_over_best": round(sel_us / best["us"], 3) if sel_us else None,
               "rule_over_best": round(rule_us / best["us"], 3) if rule_us else None}
        print(json.dumps(row), flush=True)
        out.append(row)
    return out


def merge_table(entries, path):
    """Replace, in the table at `path`, the rows of each (input dtype, output
    dtype, hidden, residual setting) measured in `entries` and keep every
    other row, so a sweep of some hidden sizes (or of one residual setting)
    leaves the rows of the others in place.  Rows written before the table
    recorded the residual setting are read as measured with a residual, but
    the fp32 rows (measured without one)."""
    import re

    measured = {(DTYPE_CODES[e["in"]], DTYPE_CODES[e["out"]], e["H"], int(bool(e["res"])))
                for e in entries}
    kept = []
    for line in open(path):
        m = re.match(ROW_RE, line)
        if not m or int(m.group(1)) < 0:
            continue
        v = [int(m.group(i)) for i in range(1, 9)]
        res = int(m.group(9)) if m.group(9) is not None else int(v[0] != DTYPE_CODES["f32"])
        bias = int(m.group(10)) if m.group(10) is not None else int(v[1] != DTYPE_CODES["bf16"]
                                                                  and v[0] != DTYPE_CODES["f32"]
                                                                  and v[0] < 6)
        if (v[0], v[1], v[2], res) in measured:
            continue
        kept.append(tuple(v) + (res, bias, float(m.group(11) or 0), float(m.group(12) or 0)))
    write_table(entries, path, extra_rows=kept)


def write_table(entries, path, extra_rows=()):
    """Selector rows from the sweep: per (dtypes, hidden), the best shape from
    each measured token count upward.  Ties within 1 % prefer fewer warps,
    then the register kernel, then fewer ring stages."""
    rows = []
    for e in entries:
        best_us = e["best"]["us"]
        near = [d for d in e["all"] if d["us"] <= best_us * 1.01 and d["variant"] != 3]
        if not near:
            continue
        pick = min(near, key=lambda d: (d["warps_per_block"], d["variant"] != 1, d["stages"],
                                        d["us"]))
        rows.append((DTYPE_CODES[e["in"]], DTYPE_CODES[e["out"]], e["H"], e["T"], pick["variant"],
                     pick["chunks"], pick["max_warps"], pick["stages"], int(bool(e["res"])),
                     int(bool(e["bias"])), pick["us"], pick["gbs"]))
    rows.extend(extra_rows)
    rows.sort(key=lambda r: (r[0], r[1], r[2], -r[8], r[3]))
    lines = [
        "// Launch shapes chosen from measured bandwidth on a GB300 by",
        "// residual_add_rmsnorm_vec_gb300/tune.py (CUDA-graph replay of back-to-back",
        "// launches; inputs rotated past the L2 size from 512 tokens up, L2-hot below).",
        "// For one (input dtype, output dtype, hidden) the row with the largest",
        "// t_min <= n_tokens applies, among the rows measured with the caller's",
        "// residual setting where the table has any; hidden sizes without rows take",
        "// the rows of the nearest measured hidden size (within a factor of two),",
        "// else the fixed rule in the selector.  Input keys are DType codes, or 7 / 8",
        "// for bf16 / fp16 activations over an fp32 residual stream, or 9 for bf16",
        "// rows measured as launches chained by programmatic dependent launch (taken",
        "// first for calls with RMSN_PDL).  res / bias: the operands the row was",
        "// measured with.",
        "struct TableRow {",
        "    int in_dt, out_dt;",
        "    int64_t hidden, t_min;",
        "    int variant, chunks, max_warps, stages;",
        "    int res, bias;",
        "};",
        "",
        "static const TableRow kSelectorTable[] = {",
    ]
    seen = set()
    for r in rows:
        key = r[:4] + (r[8],)
        if key in seen:
            continue
        seen.add(key)
        lines.append(f"    {{{r[0]}, {r[1]}, {r[2]}, {r[3]}, {r[4]}, {r[5]}, {r[6]}, {r[7]}, "
                     f"{r[8]}, {r[9]}}},  // {r[10]:.2f} us, {r[11]:.0f} GB/s")
    if not seen:
        lines.append("    {-1, -1, 0, 0, 0, 0, 0, 0, 0, 0},")
    lines += LOOKUP_CPP
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")


LOOKUP_CPP = [
        "};",
        "",
        "// The row for (in_dt, out_dt, hidden) and n_tokens: among the rows measured",
        "// with the residual setting `res` if there are any, else among the others.",
        "bool table_lookup(int in_dt, int out_dt, int64_t hidden, int64_t n_tokens, int res,",
        "                  int* variant, int* chunks, int* max_warps, int* stages) {",
        "    bool same = false;",
        "    for (const TableRow& r : kSelectorTable)",
        "        same = same || (r.in_dt == in_dt && r.out_dt == out_dt && r.hidden == hidden &&",
        "                        r.res == res);",
        "    const TableRow* best = nullptr;",
        "    for (const TableRow& r : kSelectorTable) {",
        "        if (r.in_dt != in_dt || r.out_dt != out_dt || r.hidden != hidden) continue;",
        "        if (same && r.res != res) continue;",
        "        if (r.t_min <= n_tokens && (!best || r.t_min > best->t_min)) best = &r;",
        "    }",
        "    if (!best) return false;",
        "    *variant = best->variant;",
        "    *chunks = best->chunks;",
        "    *max_warps = best->max_warps;",
        "    *stages = best->stages;",
        "    return true;",
        "}",
        "",
        "// Measured hidden sizes of (in_dt, out_dt) other than `hidden` and within a",
        "// factor of two of it, nearest first by ratio (the smaller of two equally",
        "// near first); writes at most `cap`, returns how many.",
        "int table_neighbours(int in_dt, int out_dt, int64_t hidden, int64_t* out, int cap) {",
        "    int n = 0;",
        "    for (const TableRow& r : kSelectorTable) {",
        "        if (r.in_dt != in_dt || r.out_dt != out_dt || r.hidden == hidden) continue;",
        "        if (r.hidden > 2 * hidden || 2 * r.hidden < hidden) continue;",
        "        bool seen = false;",
        "        for (int i = 0; i < n; ++i) seen = seen || out[i] == r.hidden;",
        "        if (seen || n >= cap) continue;",
        "        // insert in order: a before b when max(a,h)/min(a,h) < max(b,h)/min(b,h)",
        "        const int64_t a = r.hidden;",
        "        int i = n++;",
        "        for (; i > 0; --i) {",
        "            const int64_t b = out[i - 1];",
        "            const int64_t lhs = (a > hidden ? a : hidden) * (b < hidden ? b : hidden);",
        "            const int64_t rhs = (b > hidden ? b : hidden) * (a < hidden ? a : hidden);",
        "            if (lhs > rhs || (lhs == rhs && a > b)) break;",
        "            out[i] = b;",
        "        }",
        "        out[i] = a;",
        "    }",
        "    return n;",
        "}",
]

def main():
    import torch

    import residual_add_rmsnorm_vec_gb300 as pkg
    from residual_add_rmsnorm_vec_gb300 import build

    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default="sweep.json")
    ap.add_argument("--reps", type=int, default=30)
    ap.add_argument("--write-table", action="store_true")
    ap.add_argument("--table-out", default=os.path.join(
        os.path.dirname(os.path.abspath(__file__)), "csrc", "rmsn_selector_table.inc"))
    ap.add_argument("--quick", action="store_true", help="a few shapes only")
    ap.add_argument("--l2-hot-below", type=int, default=512,
                    help="time shapes with fewer tokens L2-hot (decode sizes)")
    ap.add_argument("--block-formats", action="store_true",
                    help="sweep only the block-scaled outputs and merge their rows into the table")
    ap.add_argument("--shapes", default="",
                    help="comma list of TxH shapes (e.g. 16384x8190) to measure for --pairs (or "
                         "bf16:bf16) instead of the default grid; the table is left alone unless "
                         "--write-table")
    ap.add_argument("--pairs", default="",
                    help="comma list of input:output pairs (e.g. f16:f16,bf16+r32:bf16) to sweep "
                         "on the hidden sizes 2048..16384; rows merged into the table")
    ap.add_argument("--check-selector", default="",
                    help="comma list of TxH shapes (bf16, residual, weight): time every built "
                         "launch and report the selector's and the fixed rules' picks against "
                         "the fastest (e.g. for hidden sizes without table rows)")
    ap.add_argument("--outs", default="",
                    help="comma list of quantised outputs (fp8, mxfp8, mxfp4, nvfp4) to sweep on "
                         "the quantised shapes; rows merged into the table")
    ap.add_argument("--pdl", action="store_true",
                    help="with --outs / --block-formats: time launches chained by programmatic "
                         "dependent launch (the rows go to the PDL key)")
    args = ap.parse_args()
    build.build()
    torch.cuda.set_device(0)
    grid = [(T, H) for H in HIDDEN for T in TOKENS]
    if args.quick:
        grid = [(1, 4096), (256, 4096), (16384, 8192)]
    hot = args.l2_hot_below
    if args.check_selector:
        shapes = [tuple(int(v) for v in sh.split("x")) for sh in args.check_selector.split(",")]
        rows = check_selector(pkg, shapes, args.reps, hot)
        with open(args.out, "w") as f:
            json.dump({"meta": {"gpu": torch.cuda.get_device_name(0), "reps": args.reps,
                                "l2_hot_below": hot, "timing": "cuda graph replay"},
                       "rows": rows}, f, indent=1)
        return
    if args.pairs or args.shapes:
        shapes = [(T, H) for H in HIDDEN for T in (1, 16, 256, 1024, 4096, 16384)]
        if args.shapes:
            shapes = [tuple(int(v) for v in sh.split("x")) for sh in args.shapes.split(",")]
        entries = []
        for pair in (args.pairs or "bf16:bf16").split(","):
            i, o = pair.split(":")
            entries += sweep(pkg, shapes, i, o, True, False, args.reps, hot)
        with open(args.out, "w") as f:
            json.dump({"meta": {"gpu": torch.cuda.get_device_name(0), "reps": args.reps,
                                "l2_hot_below": hot, "timing": "cuda graph replay"},
                       "entries": entries}, f)
        if args.write_table:
            merge_table(entries, args.table_out)
        return
    if args.block_formats or args.outs:
        entries = []
        for fmt in (args.outs.split(",") if args.outs else BLOCK_FMTS):
            entries += sweep(pkg, [(T, H) for H in (4096, 5120, 7168, 8192)
                                   for T in (1, 64, 1024, 4096, 16384)],
                             "bf16+pdl" if args.pdl else "bf16", fmt, True, True, args.reps, hot)
        with open(args.out, "w") as f:
            json.dump({"meta": {"gpu": torch.cuda.get_device_name(0), "reps": args.reps,
                                "l2_hot_below": hot, "timing": "cuda graph replay"},
                       "entries": entries}, f)
        if args.write_table:
            merge_table(entries, args.table_out)
        return
    entries = sweep(pkg, grid, "bf16", "bf16", True, False, args.reps, hot)
    # the other dtype paths of the hot-path workloads
    entries += sweep(pkg, [(T, H) for H in (4096, 5120, 7168, 8192)
                           for T in (1, 64, 1024, 4096, 16384)],
                     "bf16", "fp8", True, True, args.reps, hot)
    entries += sweep(pkg, [(T, 1024) for T in (1, 64, 4096)], "f32", "f32", False, False,
                     args.reps, hot)
    meta = {"gpu": torch.cuda.get_device_name(0),
            "sms": torch.cuda.get_device_properties(0).multi_processor_count,
            "reps": args.reps, "l2_hot_below": args.l2_hot_below, "timing": "cuda graph replay"}
    with open(args.out, "w") as f:
        json.dump({"meta": meta, "entries": entries}, f)
    if args.write_table:
        # the rows of the other dtype pairs (block formats, fp16, fp32 stream) stay
        merge_table(entries, args.table_out)


if __name__ == "__main__":
    main()
