"""The measured selector table (csrc/rmsn_selector_table.inc), checked on the
CPU against the sources it is read with: every row names a kernel that the
translation unit of its dtype pair instantiates, ring stages appear only on
ring rows and within the kernel's cap, each (input, output, hidden) runs
from one token up in increasing order, and the tuner writes the dtype codes
the library reads.  A row that fails any of these would be skipped by the
selector at run time and its shape would fall back to the fixed rule."""
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "residual_add_rmsnorm_vec_gb300", "csrc")


def read(name):
    with open(os.path.join(CSRC, name)) as f:
        return f.read()


def enum_values(text, name):
    body = re.search(r"enum %s : int32_t \{([^}]*)\}" % name, text).group(1)
    return {k: int(v) for k, v in re.findall(r"(\w+) = (\d+)", body)}


@pytest.fixture(scope="module")
def codes():
    reg = read("rmsn_registry.h")
    dtypes = enum_values(reg, "DType")
    variants = enum_values(reg, "Variant")
    api = read("rmsn_api.cu")
    r32 = {k: int(v) for k, v in re.findall(r"constexpr int (kTable\w+(?:R32|PDL)) = (\d+);",
                                             api)}
    stages = int(re.search(r"constexpr int kMaxStages = (\d+);", api).group(1))
    return dtypes, variants, r32, stages


@pytest.fixture(scope="module")
def rows():
    out = []
    for line in read("rmsn_selector_table.inc").splitlines():
        m = re.match(r"\s*\{(-?\d+), (-?\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), "
                     r"([01]), ([01])\},", line)
        if m:
            out.append(tuple(int(v) for v in m.groups()))
    assert out, "no rows parsed"
    return out


@pytest.fixture(scope="module")
def instantiated(codes):
    """(table input key, output code) -> set of (variant, CH, WMAX) built."""
    dtypes, variants, r32, _ = codes
    inst = read("rmsn_instances.cuh")
    body = inst[inst.index("static const KernelEntry kTable[]"):]
    vec = re.findall(r"RMSN_VEC4\((\d+), (\d+), (true|false)\)", body)
    bulk = re.findall(r"RMSN_BULK4\((\d+), (\d+)\)", body)
    pipe = re.findall(r"RMSN_PIPE4\((\d+), (\d+)\)", body)
    clu = re.findall(r"RMSN_CLU4\((\d+), (\d+)\)", body)
    assert vec and bulk and pipe and clu
    built = {}
    for tu in glob.glob(os.path.join(CSRC, "rmsn_k_*.cu")):
        with open(tu) as f:
            src = f.read()
        m_in = re.search(r"#define RMSN_DTI (k\w+)", src)
        m_out = re.search(r"#define RMSN_DTO (k\w+)", src)
        if not (m_in and m_out):
            continue
        tin = dtypes[m_in.group(1)]
        if re.search(r"#define RMSN_RF32 1", src):
            tin = r32["kTableF16R32"] if m_in.group(1) == "kF16" else r32["kTableBF16R32"]
        shapes = {(variants["kWarpRows"] if wr == "true" else variants["kBlockRow"], int(ch),
                   int(w)) for ch, w, wr in vec}
        if "#define RMSN_NO_BULK" not in src:
            shapes |= {(variants["kBulkRow"], int(ch), int(w)) for ch, w in bulk}
        if "#define RMSN_WITH_PIPE" in src:
            shapes |= {(variants["kBulkPipe"], int(ch), int(w)) for ch, w in pipe}
        if "#define RMSN_WITH_CLUSTER" in src:
            shapes |= {(variants["kCluster"], int(ch), int(k)) for ch, k in clu}
        built[(tin, dtypes[m_out.group(1)])] = shapes
        if tin == dtypes["kBF16"]:  # rows measured with PDL take the same kernels
            built[(r32["kTableBF16PDL"], dtypes[m_out.group(1)])] = shapes
    return built


def test_tuner_writes_the_library_codes(codes):
    from residual_add_rmsnorm_vec_gb300 import tune

    dtypes, _, r32, _ = codes
    names = {"f32": "kF32", "bf16": "kBF16", "fp8": "kFP8", "mxfp8": "kMXFP8",
             "mxfp4": "kMXFP4", "nvfp4": "kNVFP4", "f16": "kF16"}
    for name, enum in names.items():
        assert tune.DTYPE_CODES[name] == dtypes[enum], name
    assert tune.DTYPE_CODES["bf16+r32"] == r32["kTableBF16R32"]
    assert tune.DTYPE_CODES["f16+r32"] == r32["kTableF16R32"]
    assert tune.DTYPE_CODES["bf16+pdl"] == r32["kTableBF16PDL"]


def test_every_row_names_a_built_kernel(rows, instantiated, codes):
    _, variants, _, max_stages = codes
    for r in rows:
        tin, tout, hidden, t_min, variant, ch, wmax, stages, res, bias = r
        assert (tin, tout) in instantiated, f"no translation unit for {r}"
        assert (variant, ch, wmax) in instantiated[(tin, tout)], f"kernel not built: {r}"
        if variant in (variants["kBulkRow"], variants["kBulkPipe"]):
            assert 2 <= stages <= max_stages, r
        else:
            assert stages == 0, r
        assert hidden > 0 and t_min >= 1, r


def test_rows_cover_every_token_count_in_order(rows):
    groups = {}
    for r in rows:
        groups.setdefault(r[:3] + (r[8],), []).append(r[3])
    for key, t_mins in groups.items():
        assert t_mins[0] == 1, f"{key}: first row starts at {t_mins[0]} tokens"
        assert all(a < b for a, b in zip(t_mins, t_mins[1:])), f"{key}: {t_mins}"


def test_rows_are_whole_vector_shapes(rows, codes):
    """Table rows are measured on the 32-byte vector kernels, so each hidden
    size is a whole number of 32-byte vectors of the input type."""
    dtypes, _, r32, _ = codes
    elem = {dtypes["kF32"]: 4, dtypes["kBF16"]: 2, dtypes["kF16"]: 2,
            r32["kTableBF16R32"]: 4, r32["kTableF16R32"]: 4, r32["kTableBF16PDL"]: 2}
    for r in rows:
        assert (r[2] * elem[r[0]]) % 32 == 0, r


def test_rows_record_the_operands_they_were_measured_with(rows, codes):
    """Each row says whether its sweep had a residual and a bias: the 16-bit
    and fp32-stream rows were measured with a residual and no bias, the
    quantised outputs with both, the fp32 rows with neither."""
    dtypes, _, r32, _ = codes
    quant = {dtypes[k] for k in ("kFP8", "kMXFP8", "kMXFP4", "kNVFP4")}
    for r in rows:
        tin, tout, res, bias = r[0], r[1], r[8], r[9]
        if tin == dtypes["kF32"]:
            assert (res, bias) == (0, 0), r
        elif tout in quant:
            assert (res, bias) == (1, 1), r
        else:
            assert bias == 0, r
