"""bench.py's contract on the CPU: the reference arm (the oracle timed on the
host cores) prints one JSON line with the keys the measurement needs, for
the prefill step and for the FP8 step; the recorded DRAM traffic is only
reported while the kernel sources still match the capture; the workload of
the timed step follows --out."""
import json
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def run_reference(*extra):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "3", "--warmup", "3", "--ref-seconds", "2", *extra],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("extra,workload", [
    ((), "prefill fused residual-add + RMSNorm bf16 T=16384 H=8192"),
    (("--out", "fp8", "--tokens", "4096", "--hidden", "5120"), "per-token FP8 E4M3 with bias"),
])
def test_reference_arm_line(extra, workload):
    d = run_reference(*extra)
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e", "gpu_launches"):
        assert k in d, k
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["gpu_launches"] == 0
    assert workload in d["config"]["workload"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    # the same config object as the repo's own arm prints (bench.step_config)
    from residual_add_rmsnorm_vec_gb300 import synth

    class A:
        out = "fp8" if "--out" in extra else "bf16"
        hidden = int(extra[extra.index("--hidden") + 1]) if "--hidden" in extra else 8192
    tokens = int(extra[extra.index("--tokens") + 1]) if "--tokens" in extra else 16384
    assert d["config"] == bench.step_config(bench.step_workload(synth, A, tokens), 1)


def test_reference_arm_other_ranks_print_nothing():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "3", "--warmup", "3"], capture_output=True, text=True,
                         timeout=300, cwd=ROOT, env=env)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_recorded_traffic_follows_the_sources(tmp_path, monkeypatch):
    rec = {"k_T1_H1": {"dram_bytes_per_launch": 123, "source_hash": bench.kernel_source_hash(),
                       "capture": "x"},
           "stale": {"dram_bytes_per_launch": 456, "source_hash": "0000", "capture": "y"}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the sources are hashed from the package, the record read from ROOT
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: rec["k_T1_H1"]["source_hash"])
    assert bench.recorded_traffic("k_T1_H1") == 123
    assert bench.recorded_traffic("stale") is None
    assert bench.recorded_traffic("absent") is None


def test_source_hash_leaves_out_only_the_selector_table(tmp_path, monkeypatch):
    # a recorded capture stays valid when only the measured selector table
    # changes (the record is keyed by the full launch shape), not when a
    # kernel source does
    csrc = tmp_path / "residual_add_rmsnorm_vec_gb300" / "csrc"
    shutil.copytree(os.path.join(ROOT, "residual_add_rmsnorm_vec_gb300", "csrc"), csrc)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    (csrc / "rmsn_selector_table.inc").write_text("// other rows\n")
    assert bench.kernel_source_hash() == h0
    k = csrc / "rmsn_kernels.cuh"
    k.write_text(k.read_text() + "\n// changed\n")
    assert bench.kernel_source_hash() != h0


def test_step_workload_follows_out():
    from residual_add_rmsnorm_vec_gb300 import synth

    class A:
        out, hidden = "bf16", 8192

    wl = bench.step_workload(synth, A, 16384)
    assert wl.out_dtype == "bf16" and not wl.has_bias and wl.algorithmic_bytes() == 1073758208
    A.out, A.hidden = "fp8", 5120
    wl = bench.step_workload(synth, A, 4096)
    assert wl.out_dtype == "fp8" and wl.has_bias
    assert wl.algorithmic_bytes() == 4096 * (7 * 5120 + 4) + 4 * 5120
