"""CPU-only checks of the C ABI library and of the host-side logic (no GPU).

The library must build for sm_103a here (nvcc cross-compiles), load through
the binding and export every entry point include/qgemm.h declares.  No
compute entry point is called: there is no GPU in this container.
"""
import os
import re
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qgemm.h")
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))


def _declared_functions():
    names = []
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n.startswith(("qg", "qmoe"))))


@pytest.fixture(scope="module")
def built_lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from gemm_blockwise_dequant_gb300 import build

    return build.build()


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ["qgemm_nbits", "qgemm_nbits_uniform_zp", "qgemm_codebook4", "qmoe_decode_fused",
              "qgemm_workspace_bytes", "qmoe_decode_workspace_bytes", "qg_fp16_uniform_value",
              "qg_dequant_nbits", "qg_dequant_codebook4", "qg_status_string", "qg_test_bounded_wait"]:
        assert n in names


def test_library_exports_every_declared_symbol(built_lib):
    out = subprocess.run(["nm", "-D", "--defined-only", built_lib], capture_output=True, text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if " T " in line)
    missing = [n for n in _declared_functions() if n not in exported]
    assert not missing, missing


def test_binding_loads_and_names_statuses(built_lib):
    import gemm_blockwise_dequant_gb300 as qg

    L = qg.lib()
    for n in _declared_functions():
        assert hasattr(L, n)
    assert qg.qg_status_string(qg.QG_OK) == "QG_OK"
    assert qg.qg_status_string(qg.QG_ERR_UNSUPPORTED) == "QG_ERR_UNSUPPORTED"
    assert qg.qg_status_string(99) == "QG_ERR_UNKNOWN"


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import gemm_blockwise_dequant_gb300 as qg

    monkeypatch.setattr(qg, "_lib", None)
    monkeypatch.setattr(qg, "library_path", str(tmp_path / "missing.so"))
    with pytest.raises(qg.QGLibraryMissing):
        qg.lib()


def test_workload_generators_are_seeded_and_in_range():
    import workloads as W

    a, b = W.tiny_u4(0), W.tiny_u4(0)
    for k in ("W", "scales", "zero_points", "A"):
        assert np.array_equal(a[k], b[k])
    assert not np.array_equal(W.tiny_u4(1)["W"], a["W"])
    s = a["scales"].view(np.float16).astype(np.float64)
    assert s.min() >= 0.005 - 1e-5 and s.max() <= 0.02 + 1e-5
    z = a["zero_points"].view(np.float16).astype(np.float64)
    assert np.array_equal(z, np.round(z)) and z.min() >= 0 and z.max() <= 15
    cb = W.nf4_codebook()
    assert cb.dtype == np.float32 and cb.size == 16 and cb[0] == -1 and cb[-1] == 1 and (cb == 0).sum() == 1
    assert np.all(np.diff(cb) > 0)
    ids, w = W.routing(W.rng(0), 128, 8)
    assert len(set(ids.tolist())) == 8 and ids.min() >= 0 and ids.max() < 128
    assert abs(float(w.sum()) - 1.0) < 1e-6


def test_workload_phi4_shapes():
    import workloads as W

    assert W.PHI4_SHAPES["lm_head"] == (100352, 5120)
    d = W.phi4_u2("o", M=4)
    assert d["W"].shape == (5120, 5120 // 4) and d["scales"].shape == (5120, 80) and d["A"].shape == (4, 5120)


def test_workload_packed_zero_points_shapes():
    import workloads as W

    for bits, nb in ((2, 7), (3, 7), (4, 160), (8, 2)):
        d = W.packed_zp(5, nb * 32, M=2, bits=bits, block_size=32, seed=1)
        assert d["zp_packed"].shape == (5, (nb * bits + 7) // 8) and d["zp_packed"].dtype == np.uint8
        assert d["W"].shape == (5, nb * 32 * bits // 8) and d["scales"].shape == (5, nb) and d["A"].shape == (2, nb * 32)
    assert np.array_equal(W.packed_zp(4, 64, seed=3)["zp_packed"], W.packed_zp(4, 64, seed=3)["zp_packed"])


def _header_constants():
    """#define and enum integer constants of the header, evaluated (shifts and literals only)."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for name, expr in re.findall(r"^#define\s+(QG_[A-Z0-9_]+)\s+(.+)$", text, flags=re.M):
        expr = re.sub(r"(\d+)[uUlL]+", r"\1", expr.strip())
        if re.fullmatch(r"[\d\s()<>+*]+", expr):
            out[name] = eval(expr, {"__builtins__": {}})
    for body in re.findall(r"enum\s*\{([^}]*)\}", text):
        for name, val in re.findall(r"(QG_[A-Z0-9_]+)\s*=\s*(\d+)", body):
            out[name] = int(val)
    return out


def test_binding_constants_match_the_header():
    """The binding's copies of the header's constants (status codes, dtypes,
    table formats, the no-allocation scratch size) equal the header's values."""
    import gemm_blockwise_dequant_gb300 as qg

    consts = _header_constants()
    assert "QG_QMOE_NOALLOC_SCRATCH_BYTES" in consts
    for name, value in consts.items():
        if hasattr(qg, name):
            assert getattr(qg, name) == value, name
    for name in ("QG_QMOE_NOALLOC_SCRATCH_BYTES", "QG_OK", "QG_ERR_CUDA", "QG_BF16", "QG_WF_E4M3"):
        assert hasattr(qg, name) and name in consts, name
