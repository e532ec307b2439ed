"""The tuner's selector-table writer, on the CPU: among launches within 1% of
the fastest it keeps the one with fewer warps, then the register kernel, then
fewer ring stages, and never the generic kernel; merging replaces only the
(dtype pair, hidden) rows it measured; and the C++ lookup it writes, compiled with the host
compiler, returns the row with the largest token threshold not above the
token count, and nothing for a hidden size or dtype pair it has no rows for."""
import re
import shutil
import subprocess

import pytest

from residual_add_rmsnorm_vec_gb300 import tune

ROW = re.compile(r"\s*\{(-?\d+), (-?\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), "
                 r"(\d+), (\d+)\},")


def cand(variant, warps, us, chunks=2, max_warps=16, stages=0):
    return {"variant": variant, "chunks": chunks, "warps_per_block": warps,
            "max_warps": max_warps, "stages": stages, "us": us, "gbs": 1e3 / us}


def entry(T, H, cands, i="bf16", o="bf16", res=True):
    return {"T": T, "H": H, "in": i, "out": o, "res": res, "bias": False,
            "best": min(cands, key=lambda d: d["us"]), "all": cands}


def rows_of(path):
    with open(path) as f:
        return [tuple(int(v) for v in m.groups()) for m in map(ROW.match, f) if m]


def test_tie_break_prefers_fewer_warps_then_register_kernel_then_fewer_stages(tmp_path):
    bf = tune.DTYPE_CODES["bf16"]
    entries = [
        # the ring at 8 warps is fastest; the register kernel at 8 warps is
        # within 1% and wins the tie; 4 warps is 1.2% slower and stays out;
        # the generic kernel is never taken
        entry(1, 4096, [cand(2, 8, 100.0, stages=4), cand(1, 8, 100.5), cand(1, 4, 101.2),
                        cand(3, 2, 100.2)]),
        # two rings within 1%: the one with fewer stages
        entry(16, 4096, [cand(2, 4, 50.0, stages=6), cand(2, 4, 50.3, stages=2)]),
        # fewer warps beat the fastest when within 1%
        entry(256, 4096, [cand(1, 16, 10.0, max_warps=16), cand(1, 8, 10.09, max_warps=8)]),
    ]
    path = tmp_path / "t.inc"
    tune.write_table(entries, str(path))
    got = {r[3]: r[4:8] for r in rows_of(path) if r[:3] == (bf, bf, 4096)}
    assert got[1] == (1, 2, 16, 0)
    assert got[16] == (2, 2, 16, 2)
    assert got[256] == (1, 2, 8, 0)


def test_merge_replaces_only_the_measured_hidden_sizes(tmp_path):
    c = tune.DTYPE_CODES
    path = tmp_path / "t.inc"
    tune.write_table([entry(1, 4096, [cand(1, 8, 3.0)]),
                      entry(1, 4096, [cand(1, 4, 4.0)], o="fp8"),
                      entry(4096, 4096, [cand(2, 8, 30.0, stages=4)], o="fp8"),
                      entry(1, 5120, [cand(1, 4, 4.5)], o="fp8")], str(path))
    before = rows_of(path)
    tune.merge_table([entry(1, 4096, [cand(1, 16, 3.5)], o="fp8")], str(path))
    after = rows_of(path)
    # another dtype pair, and another hidden size of the measured pair, stay
    assert [r for r in after if r[1] == c["bf16"]] == [r for r in before if r[1] == c["bf16"]]
    assert [r for r in after if r[2] == 5120] == [r for r in before if r[2] == 5120]
    # the measured (pair, hidden) is replaced whole: its 4096-token row goes
    fp8 = [r for r in after if r[1] == c["fp8"] and r[2] == 4096]
    assert fp8 == [(c["bf16"], c["fp8"], 4096, 1, 1, 2, 16, 0, 1, 0)]
    # a sweep without a residual adds its own rows and keeps those with one
    tune.merge_table([entry(1, 4096, [cand(1, 4, 2.0)], res=False)], str(path))
    bf = [r for r in rows_of(path) if r[:3] == (c["bf16"], c["bf16"], 4096)]
    assert sorted(r[8] for r in bf) == [0, 1] and (c["bf16"], c["bf16"], 4096, 1, 1, 2, 16, 0,
                                                   0, 0) in bf


HARNESS = r"""
#include <cstdint>
#include <cstdio>
#include "t.inc"
int main() {
    const long long q[][4] = {{1, 1, 4096, 1}, {1, 1, 4096, 15}, {1, 1, 4096, 16},
                              {1, 1, 4096, 255}, {1, 1, 4096, 1000000}, {1, 1, 5120, 64},
                              {1, 2, 4096, 64}};
    for (auto& x : q) {
        int v = -1, c = -1, w = -1, s = -1;
        const bool f = table_lookup((int)x[0], (int)x[1], x[2], x[3], 1, &v, &c, &w, &s);
        std::printf("%d %d %d %d %d\n", f ? 1 : 0, v, c, w, s);
    }
    return 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="no host C++ compiler")
def test_generated_lookup_takes_the_largest_threshold_not_above_the_tokens(tmp_path):
    tune.write_table([entry(1, 4096, [cand(1, 8, 2.0, max_warps=8)]),
                      entry(16, 4096, [cand(1, 16, 2.5, max_warps=16)]),
                      entry(256, 4096, [cand(2, 8, 9.0, stages=4, max_warps=32)])],
                     str(tmp_path / "t.inc"))
    (tmp_path / "h.cpp").write_text(HARNESS)
    subprocess.run(["g++", "-std=c++17", "-O1", "-o", str(tmp_path / "h"), str(tmp_path / "h.cpp")],
                   check=True, cwd=tmp_path)
    out = subprocess.run([str(tmp_path / "h")], check=True, capture_output=True,
                         text=True).stdout.split("\n")
    got = [tuple(int(v) for v in line.split()) for line in out if line.strip()]
    assert got == [
        (1, 1, 2, 8, 0),    # 1 token: the row from 1 up
        (1, 1, 2, 8, 0),    # 15 tokens: still the row from 1
        (1, 1, 2, 16, 0),   # 16 tokens: the row from 16
        (1, 1, 2, 16, 0),   # 255 tokens
        (1, 2, 2, 32, 4),   # far above the last threshold: its row
        (0, -1, -1, -1, -1),  # a hidden size without rows
        (0, -1, -1, -1, -1),  # a dtype pair without rows
    ]


NEIGHBOURS = r"""
#include <cstdint>
#include <cstdio>
#include "t.inc"
int main() {
    const long long q[] = {2560, 3584, 6656, 10240, 4096, 1024, 40000, 12288};
    for (long long h : q) {
        int64_t out[16];
        const int n = table_neighbours(1, 1, h, out, 16);
        std::printf("%lld:", h);
        for (int i = 0; i < n; ++i) std::printf(" %lld", (long long)out[i]);
        std::printf("\n");
    }
    // residual setting: rows measured without a residual win for res = 0 only
    int v, c, w, s;
    table_lookup(1, 1, 4096, 8, 0, &v, &c, &w, &s);
    std::printf("res0 %d %d\n", c, w);
    table_lookup(1, 1, 4096, 8, 1, &v, &c, &w, &s);
    std::printf("res1 %d %d\n", c, w);
    // only rows with a residual at 8192: a call without one takes them
    const bool f = table_lookup(1, 1, 8192, 8, 0, &v, &c, &w, &s);
    std::printf("fallback %d %d %d\n", f ? 1 : 0, c, w);
    return 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="no host C++ compiler")
def test_generated_neighbours_nearest_first_and_residual_rows(tmp_path):
    rows = [entry(1, h, [cand(1, 8, 2.0, max_warps=8)]) for h in (2048, 3072, 4096, 5120, 8192,
                                                                  16384)]
    rows.append(entry(1, 4096, [cand(1, 4, 1.0, chunks=1, max_warps=4)], res=False))
    tune.write_table(rows, str(tmp_path / "t.inc"))
    (tmp_path / "h.cpp").write_text(NEIGHBOURS)
    subprocess.run(["g++", "-std=c++17", "-O1", "-o", str(tmp_path / "h"), str(tmp_path / "h.cpp")],
                   check=True, cwd=tmp_path)
    out = subprocess.run([str(tmp_path / "h")], check=True, capture_output=True,
                         text=True).stdout.splitlines()
    assert out[:8] == [
        "2560: 3072 2048 4096 5120",  # ratios 1.2, 1.25, 1.6, 2.0
        "3584: 4096 3072 5120 2048",  # 1.143, 1.167, 1.429, 1.75 (8192 is beyond 2x)
        "6656: 8192 5120 4096",       # 1.231, 1.3, 1.625
        "10240: 8192 16384 5120",     # 1.25, 1.6, 2.0
        "4096: 5120 3072 2048 8192",  # not itself; 2048 and 8192 tie at 2.0: smaller first
        "1024: 2048",
        "40000:",
        "12288: 16384 8192",
    ]
    assert out[8:] == ["res0 1 4", "res1 2 8", "fallback 1 2 8"]


def test_fixed_rule_mirror_follows_the_documented_rules():
    # the tuner's copy of the selector's fixed rules (used to report how far
    # they were from the fastest launch): one warp per row while the problem
    # needs no more warps than SMs and a row fits 8 vectors a lane, else the
    # fewest of 4 / 8 / 16 / 32 warps with two vectors per thread
    assert tune.fixed_rule_shape(8, 2560, 152) == (0, 8, 1)     # 160 vectors: CH 8 covers
    assert tune.fixed_rule_shape(1, 4096, 152) == (0, 8, 1)
    assert tune.fixed_rule_shape(2, 512, 152) == (0, 1, 1)      # 32 vectors: one chunk
    assert tune.fixed_rule_shape(4096, 2560, 152) == (1, 2, 4)  # 4096 warps > 152 SMs
    assert tune.fixed_rule_shape(1, 10240, 152) == (1, 2, 16)   # 640 vectors > 8 per lane
    assert tune.fixed_rule_shape(16384, 6656, 152) == (1, 2, 8)
    assert tune.fixed_rule_shape(1, 65536, 152) == (3, 0, 8)    # nothing fits: generic
