"""Run a few launches of named workloads through the C ABI, for profilers.

    python -m residual_add_rmsnorm_vec_gb300.profile_cases CASE [CASE ...] [--reps N]

Each case builds its seeded inputs, then launches the selector's (or the
named) configuration `reps` times on the current stream and synchronises, so
that an ncu capture can pick one launch (`-k regex:<kernel> -s <skip> -c 1`).
Cases:

  decode_T<T>        bf16 fused residual-add + RMSNorm, T tokens x 4096 (the
                     decode workload), the selector's launch
  cluster_T<T>_K<K>  the same rows on the split-row cluster variant, K blocks
  qk_T<T>            QK norm, 32 query + 8 key heads x 128 bf16 in a fused
                     qkv buffer (value heads skipped), one launch; qkring_T<T> /
                     qkdirect_T<T> force the ring / the register kernel
  ragged_T<T>_H<H>   bf16 rows off the 32-byte grid (ragged-row kernel), bias;
                     raggedfp8_T<T>_H<H>: the same with a per-token FP8 output
  fp8_T<T>_H<H>      bf16 in, per-token FP8 out, bias (the quantised workload)
  nvfp4_T<T>_H<H>    bf16 in, NVFP4 out, bias
  fp8pipe_T<T>_H<H>, nvfp4pipe_T<T>_H<H>
                     the same on the two-row pipelined ring (2 vectors a thread,
                     the 16-warp-bound instance)
  prefill_T<T>_H<H>  the prefill workload (outlier channels, eps 1e-5)
"""
from __future__ import annotations

import argparse
import re
import sys


def run_case(name: str, reps: int) -> str:
    import torch

    import residual_add_rmsnorm_vec_gb300 as pkg
    from residual_add_rmsnorm_vec_gb300 import synth

    dev = torch.device("cuda:0")
    m = re.fullmatch(r"(\w+?)_T(\d+)(?:_H(\d+))?(?:_K(\d+))?", name)
    if not m:
        raise SystemExit(f"unknown case {name}")
    kind, T = m.group(1), int(m.group(2))
    H = int(m.group(3)) if m.group(3) else 4096
    s = torch.cuda.current_stream(dev).cuda_stream
    if kind in ("qk", "qkring", "qkdirect"):
        Hq, Hk, D = 32, 8, 128
        inp = synth.qk_inputs(T, Hq, Hk, D, "bf16")
        qkv = inp["qkv"].to(dev)
        q, k = qkv[:, :Hq * D], qkv[:, Hq * D:(Hq + Hk) * D]
        wq, wk = inp["q_weight"].to(dev), inp["k_weight"].to(dev)
        variant = {"qk": None, "qkring": "ring", "qkdirect": "direct"}[kind]
        for _ in range(reps):
            pkg.qk_norm_(q, k, wq, wk, head_dim=D, eps=1e-6, variant=variant)
        torch.cuda.synchronize(dev)
        return f"{kind} T={T} heads {Hq}+{Hk} x {D}"
    if kind in ("decode", "cluster"):
        wl = synth.decode_workload(T) if H == 4096 else synth.Workload(
            f"decode_T{T}_H{H}", T, H, 10 + T, "bf16", "bf16", 1e-6)
    elif kind == "prefill":
        wl = synth.prefill_workload(T, H)
    elif kind in ("ragged", "raggedfp8"):
        wl = synth.Workload(f"{kind}_T{T}_H{H}", T, H, 80, "bf16",
                            "fp8" if kind == "raggedfp8" else "bf16", 1e-5, has_bias=True,
                            r_std=2.0)
    elif kind in ("fp8", "nvfp4", "fp8pipe", "nvfp4pipe"):
        wl = synth.fp8_workload(H, n_tokens=T)
    else:
        raise SystemExit(f"unknown case {name}")
    inp = synth.make_inputs(wl)
    g = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    cfg = None
    if kind == "cluster":
        K = int(m.group(4) or 8)
        flags = pkg.make_flags("bf16", "bf16", True, True, False)
        cands = [c for c in pkg.rmsnorm_list_configs(T, H, flags)
                 if c.variant == pkg.VARIANT_CLUSTER and c.cluster == K]
        if not cands:
            raise SystemExit(f"no cluster configuration with K={K} for {T}x{H}")
        cfg = cands[0]
    if kind.endswith("pipe"):
        flags = pkg.make_flags("bf16", "fp8", True, True, True)
        cands = [c for c in pkg.rmsnorm_list_configs(T, H, flags)
                 if c.variant == pkg.VARIANT_BULK_PIPE and c.chunks == 2]
        cands.sort(key=lambda c: -c.max_warps)  # the 16-warp-bound instance first
        if not cands:
            raise SystemExit(f"no pipelined ring configuration for {T}x{H}")
        cfg = cands[0]
    for _ in range(reps):
        if kind.startswith("nvfp4"):
            out = pkg.fused_add_rmsnorm_blockscaled(g["x"], g["residual"], g["weight"], g["bias"],
                                                    eps=wl.eps, fmt="nvfp4", config=cfg)
        else:
            out = pkg.fused_add_rmsnorm(g["x"], g["residual"], g["weight"], g["bias"], eps=wl.eps,
                                        out_dtype=wl.out_dtype, config=cfg)
    torch.cuda.synchronize(dev)
    del out
    if cfg is None:
        if kind.startswith("nvfp4"):
            # the block formats have their own table rows, which no query
            # exposes: the captured kernel's name and grid tell the launch
            return f"{name}: the selector's NVFP4 launch"
        flags = pkg.make_flags("bf16", wl.out_dtype, wl.has_residual, True, wl.has_bias)
        cfg = pkg.rmsnorm_query_config(T, H, flags)
    return f"{name}: {cfg.as_dict()}"


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("cases", nargs="+")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args(argv)
    import torch

    from residual_add_rmsnorm_vec_gb300 import build

    build.build()
    torch.cuda.set_device(0)
    for c in args.cases:
        print(run_case(c, args.reps), flush=True)


if __name__ == "__main__":
    main(sys.argv[1:])
