"""The bounds-checked debug build of the library (built with
-DRMSNORM_BOUNDS_CHECK): every global load and store and every ring copy of
its kernels is checked against the extent of its tensor, an access out of
range is skipped and sets bit 1 of the status word.  Here the guard-band
suite and the every-configuration parity suites run against that build in a
child process (the binding loads it through RMSNORM_GB300_LIB); those tests
assert that the status word stays 0, so no kernel shape at those sizes
indexes outside its tensors, reads included."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SUITES = [
    "tests/test_gpu_guard.py",
    "tests/test_gpu_parity.py::test_every_config",
    "tests/test_gpu_parity.py::test_ragged_kernel_every_config",
    "tests/test_gpu_parity.py::test_cluster_variant_decode",
    "tests/test_gpu_parity.py::test_deep_ring_wraps",
    "tests/test_gpu_blockscaled.py::test_block_formats_every_config",
    "tests/test_gpu_qk.py",
    "tests/test_gpu_parity.py::test_status_word_clear_after_all_runs",
]


def test_checked_build_keeps_every_access_in_bounds():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from residual_add_rmsnorm_vec_gb300 import build

    path = build.build(checked=True)
    env = dict(os.environ, RMSNORM_GB300_LIB=path)
    probe = subprocess.run(
        [sys.executable, "-c", "import residual_add_rmsnorm_vec_gb300 as p; p.load(); "
                               "print(p.library_path())"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert probe.returncode == 0, probe.stderr[-2000:]
    assert probe.stdout.strip() == path
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu",
                        "-p", "no:cacheprovider", *SUITES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=3600)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
