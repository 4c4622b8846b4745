"""CPU-side checks of the C ABI: the library loads, exports every symbol the
header declares, validates arguments and plans groups without a GPU."""

import ctypes
import os
import re

import pytest

from oracle import muon_oracle as o

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from newton_schulz_03_gb300 import build_lib
    build_lib.build()
    import newton_schulz_03_gb300 as ns
    return ns


def header_symbols():
    src = open(os.path.join(ROOT, "include", "muon.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(muon_[a-z_0-9]+)\s*\(", src)))


def test_header_symbols_exported(lib):
    syms = header_symbols()
    assert "muon_step" in syms and "muon_newton_schulz_bf16" in syms
    so = ctypes.CDLL(lib.LIB_PATH)
    for s in syms:
        assert hasattr(so, s), f"{s} declared in muon.h but not exported"
    assert sorted(lib.EXPORTED) == syms


def test_status_strings(lib):
    assert lib.muon_status_string(0) == "MUON_OK"
    assert lib.muon_status_string(5) == "MUON_ERR_TIMEOUT"
    assert lib.muon_status_string(99) == "MUON_ERR_UNKNOWN"
    assert "sm_103a" in lib.muon_version()


def test_create_without_gpu_fails_cleanly(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(lib.MuonError) as ei:
        lib.muon_create()
    assert ei.value.status_name in ("MUON_ERR_NO_DEVICE", "MUON_ERR_UNSUPPORTED_ARCH")


def test_null_handle_rejected(lib):
    with pytest.raises(lib.MuonError) as ei:
        lib.muon_step(0, [(4, 4, 1)], [0], [0], [0], 0.02, 0.1, 0.95)
    assert ei.value.status_name == "MUON_ERR_INVALID_ARG"


def test_plan_groups_by_wide_shape(lib):
    # Expert up (1536x4096) and down (4096x1536) share one batch.
    info = lib.muon_plan_describe([(1536, 4096, 512), (4096, 1536, 512)], ns_steps=5)
    assert info["n_batches"] == 1 and info["matrices"] == 1024
    assert info["ns_algorithmic_flops"] == pytest.approx(1024 * o.ns_algorithmic_flops(1536, 4096))
    # The default 8 GiB cap cannot hold all 1024: chunks.
    assert info["n_chunks"] > 1
    assert info["workspace_bytes"] <= 8 << 30


def test_plan_chunks_respect_cap(lib):
    m, n = 2048, 2048
    per = 2 * m * n * 2 + 2 * m * m * 2
    info = lib.muon_plan_describe([(m, n, 96)], ns_steps=5, workspace_bytes_max=10 * per + 8192)
    assert info["max_chunk_matrices"] <= 10
    assert info["n_chunks"] == (96 + info["max_chunk_matrices"] - 1) // info["max_chunk_matrices"]
    assert info["workspace_bytes"] <= 10 * per + 8192


def test_plan_mixed_model_layer(lib):
    from newton_schulz_03_gb300.workloads import WORKLOADS
    w = WORKLOADS["l48_model"]
    groups = [(g.rows, g.cols, g.count) for g in w.groups]
    info = lib.muon_plan_describe(groups, ns_steps=5)
    assert info["n_batches"] == len(w.wide_batches()) == 4
    assert info["matrices"] == w.matrices_per_layer
    want = sum(c * o.ns_algorithmic_flops(mm, nn) for (mm, nn), c in w.wide_batches().items())
    assert info["ns_algorithmic_flops"] == pytest.approx(want)


def test_plan_launch_count(lib):
    info = lib.muon_plan_describe([(128, 64, 4)], ns_steps=5)
    # cast + norm + 5 x 3 products + apply
    assert info["launches_per_step"] == 1 + 1 + 15 + 1
    info0 = lib.muon_plan_describe([(128, 64, 4)], ns_steps=0)
    assert info0["launches_per_step"] == 1 + 1 + 1 + 1


@pytest.mark.parametrize("groups,steps", [
    ([(0, 4, 1)], 5), ([(4, -1, 1)], 5), ([(4, 4, -1)], 5), ([(4, 4, 1)], -1),
    ([(4, 4, 1)], 65), ([(4, 4, 1, float("nan"))], 5), ([(1 << 21, 4, 1)], 5),
])
def test_plan_rejects_bad_arguments(lib, groups, steps):
    with pytest.raises(lib.MuonError) as ei:
        lib.muon_plan_describe(groups, ns_steps=steps)
    assert ei.value.status_name == "MUON_ERR_INVALID_ARG"


def test_plan_empty_groups(lib):
    info = lib.muon_plan_describe([(64, 64, 0)], ns_steps=5)
    assert info["matrices"] == 0 and info["n_chunks"] == 0 and info["launches_per_step"] == 0


def test_missing_library_fails_loudly(tmp_path):
    """No fallback: with the shared library absent, the first call raises."""
    import subprocess
    import sys
    code = ("import newton_schulz_03_gb300 as ns\n"
            "try:\n"
            "    ns.muon_version()\n"
            "except ImportError as e:\n"
            "    print('raised', e)\n"
            "else:\n"
            "    print('no error')\n")
    env = dict(os.environ, MUON_LIB_PATH=str(tmp_path / "absent" / "libmuon_gb300.so"))
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.startswith("raised") and "is missing" in r.stdout
