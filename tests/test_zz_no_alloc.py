"""The allocation-free Newton-Schulz entry point.

Some callers cannot allocate device memory at the moment they
orthogonalise: code that runs while a CUDA graph is being built around it,
allocators and runtimes that must not re-enter the CUDA allocator, and
deployments whose device memory budget is fixed at start-up.  They call
muon_newton_schulz_bf16_static, whose scratch is a fixed static device
array of the library.

The static entry point launches the same kernels in the same order as the
handle-based muon_newton_schulz_bf16, so this test calls both through the C
ABI, twice in a row, and requires the two results to be identical bit for
bit; one matrix per case is also checked against the CPU oracle within the
Newton-Schulz tolerance of the parity tests.  It also checks that the calls
leave the device's free memory unchanged, that a batch of more than 65535
small matrices (more than one grid row limit) runs in passes, and that
shapes beyond the array or the dimension limit are rejected.

The file is named so that pytest collects it last.
"""

import numpy as np
import pytest

from oracle import muon_oracle as o
from tests.gpu_helpers import rel_fro, u16

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

NS_TOL = 2e-2          # m >= 64


@pytest.fixture(scope="module")
def ns():
    from newton_schulz_03_gb300 import build_lib
    build_lib.build()
    import newton_schulz_03_gb300 as pkg
    return pkg


def _inputs(m, n, count, seed):
    rng = np.random.default_rng(seed)
    Xb = o.bf16_rne_bits(rng.standard_normal((count, m, n), dtype=np.float32))
    Xf = o.bf16_bits_to_f64(Xb)
    inv = np.array([1.0 / (np.linalg.norm(Xf[i]) + o.NORM_EPS) for i in range(count)],
                   dtype=np.float32)
    return (torch.from_numpy(Xb.view(np.int16)).cuda(), torch.from_numpy(inv).cuda(), Xf, inv)


def _oracle_check(Xf, inv, got_bits, m, steps, idx):
    """Matrix `idx` of the static entry's output against the FP64 oracle
    (input X * inv, i.e. s = 1 / inv): within 2e-2 for m >= 64, and within
    the BF16 error model of the parity tests (1.15 x the error of the
    oracle's BF16 emulation + 5e-4) at every size, since a BF16 iteration
    on an 8 x 8 matrix can itself err by 5e-2."""
    s = 1.0 / float(inv[idx])
    ref = o.newton_schulz(Xf[idx], s, steps=steps)
    got = o.bf16_bits_to_f64(got_bits[idx])
    err = rel_fro(got, ref)
    if steps == 0:
        assert err <= 2.0 ** -8, f"{m}: matrix {idx}: {err:.3e}"   # one BF16 rounding of X / s
        return
    emu = o.newton_schulz(Xf[idx], s, steps=steps, emulate_bf16=True)
    bound = 1.15 * rel_fro(emu, ref) + 5e-4
    assert err <= bound, f"{m}: matrix {idx}: {err:.3e} vs error model {bound:.3e}"
    if m >= 64:
        assert err <= NS_TOL, f"{m}: matrix {idx} differs from the oracle by {err:.3e}"


@pytest.mark.parametrize("m,n,count,steps", [(256, 512, 5, 5), (2048, 2048, 3, 5),
                                             (64, 128, 4, 5), (256, 512, 5, 4),
                                             (128, 384, 3, 0)])
def test_static_entry_matches_handle_entry(ns, m, n, count, steps):
    with ns.Handle() as h:
        for call in range(2):                      # two calls in a row
            x, inv, Xf, invh = _inputs(m, n, count, seed=100 * call + m + n + steps)
            want = torch.zeros((count, m, n), dtype=torch.int16, device="cuda")
            got = torch.full((count, m, n), -1, dtype=torch.int16, device="cuda")
            flag = torch.zeros(1, dtype=torch.int32, device="cuda")
            ns.muon_newton_schulz_bf16(h.value, m, n, count, x, want, inv, steps)
            ns.muon_last_device_error(h.value)
            ns.muon_newton_schulz_bf16_static(m, n, count, x, got, inv, steps, None, flag)
            torch.cuda.synchronize()
            assert int(flag.item()) == 0
            assert torch.equal(got, want), f"call {call}: static and handle results differ"
            _oracle_check(Xf, invh, u16(got), m, steps, idx=call % count)


@pytest.mark.parametrize("steps", [0, 5])
def test_static_entry_more_matrices_than_one_grid_row_limit(ns, steps):
    # 70000 matrices of 8 x 8: the array holds 87381 of them, but one pass
    # covers at most 65535 (the scale kernel's grid.y), so two passes run.
    m, n, count = 8, 8, 70000
    x, inv, Xf, invh = _inputs(m, n, count, seed=31 + steps)
    with ns.Handle() as h:
        want = torch.zeros((count, m, n), dtype=torch.int16, device="cuda")
        ns.muon_newton_schulz_bf16(h.value, m, n, count, x, want, inv, steps)
        ns.muon_last_device_error(h.value)
    got = torch.full((count, m, n), -1, dtype=torch.int16, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    ns.muon_newton_schulz_bf16_static(m, n, count, x, got, inv, steps, None, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    assert torch.equal(got, want)
    bits = u16(got)
    for idx in (0, 65534, 65535, count - 1):       # both sides of the pass boundary
        _oracle_check(Xf, invh, bits, m, steps, idx)


def test_static_entry_allocates_nothing(ns):
    m, n, count = 512, 1024, 3
    x, inv, _, _ = _inputs(m, n, count, seed=7)
    out = torch.zeros((count, m, n), dtype=torch.int16, device="cuda")
    ns.muon_newton_schulz_bf16_static(m, n, count, x, out, inv, 5)   # set-up call
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        ns.muon_newton_schulz_bf16_static(m, n, count, x, out, inv, 5)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_static_entry_rejects_matrices_beyond_the_array(ns):
    # 2048 x 8704: 2*m*n + 4*m*m bytes = 52.4 MB fits; 4096 x 8192 does not.
    x = torch.zeros(8, dtype=torch.int16, device="cuda")
    inv = torch.ones(1, dtype=torch.float32, device="cuda")
    with pytest.raises(ns.MuonError) as ei:
        ns.muon_newton_schulz_bf16_static(4096, 8192, 1, x, x.clone(), inv, 5)
    assert ei.value.status_name == "MUON_ERR_INVALID_ARG"
    assert "static array" in str(ei.value)


def test_static_entry_rejects_the_shapes_the_handle_entry_rejects(ns):
    # The long side is limited to 2^20 for both entry points, although an
    # 8 x (2^20 + 8) matrix would fit the array.
    x = torch.zeros(8, dtype=torch.int16, device="cuda")
    inv = torch.ones(1, dtype=torch.float32, device="cuda")
    with pytest.raises(ns.MuonError) as ei:
        ns.muon_newton_schulz_bf16_static(8, (1 << 20) + 8, 1, x, x.clone(), inv)
    assert ei.value.status_name == "MUON_ERR_INVALID_ARG"
    with ns.Handle() as h:
        with pytest.raises(ns.MuonError) as ei:
            ns.muon_newton_schulz_bf16(h.value, 8, (1 << 20) + 8, 1, x, x.clone(), inv, 5)
        assert ei.value.status_name == "MUON_ERR_INVALID_ARG"
