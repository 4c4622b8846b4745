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


def test_plan_invariants_on_random_group_lists(lib):
    """Random group lists (shapes, counts, workspace caps, step counts): the
    planner counts every matrix once, batches exactly the distinct wide
    shapes, keeps chunks within the launch limits and the cap, and issues
    per chunk one cast and one apply per caller segment, one norm and the
    products."""
    import numpy as np
    rng = np.random.default_rng(2024)
    dims = [1, 7, 64, 100, 128, 129, 256, 513, 1536, 2048, 4096]
    for _ in range(300):
        groups = []
        for _ in range(int(rng.integers(1, 7))):
            r, c = int(rng.choice(dims)), int(rng.choice(dims))
            groups.append((r, c, int(rng.choice([0, 1, 2, 5, 40, 300]))))
        steps = int(rng.choice([0, 1, 5, 7]))
        cap = int(rng.choice([0, 1 << 20, 64 << 20, 1 << 30]))
        info = lib.muon_plan_describe(groups, ns_steps=steps, workspace_bytes_max=cap)
        live = [(min(r, c), max(r, c), k) for r, c, k in groups if k > 0]
        shapes = {(m, n) for m, n, _ in live}
        assert info["matrices"] == sum(k for _, _, k in live)
        assert info["n_batches"] == len(shapes)
        want = sum(k * o.ns_algorithmic_flops(m, n, steps) for m, n, k in live)
        assert info["ns_algorithmic_flops"] == pytest.approx(want, rel=1e-12)
        if not live:
            assert info["n_chunks"] == 0 and info["launches_per_step"] == 0
            continue
        C, G, B = info["n_chunks"], len(live), len(shapes)
        assert B <= C <= info["matrices"]
        assert 1 <= info["max_chunk_matrices"] <= 65535
        per_total = {}
        for m, n, k in live:
            per_total[(m, n)] = per_total.get((m, n), 0) + k
        # No batch is cut into more chunks than its matrices need at the
        # largest chunk size.
        assert C >= sum(-(-t // info["max_chunk_matrices"]) for t in per_total.values())
        products = 3 * steps if steps > 0 else 1
        segs_lo, segs_hi = max(C, G), G + C - B
        launches = info["launches_per_step"]
        assert C * (1 + products) + 2 * segs_lo <= launches <= C * (1 + products) + 2 * segs_hi
        # A cap that holds one matrix of each batch bounds the workspace
        # (X twice, A and B, per-tile partials, padding and alignment).
        one = max(4 * m * (n + 8) + 4 * m * (m + 8) + 4 * (-(-m // 64)) * (-(-n // 64)) + 4096
                  for m, n in shapes)
        if cap >= one:
            assert info["workspace_bytes"] <= cap
