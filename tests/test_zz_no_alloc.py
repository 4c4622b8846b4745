"""The allocation-free Newton-Schulz entry point.

Callers that cannot allocate device memory when they orthogonalise (code
inside CUDA graph construction, allocators or runtimes that must not
re-enter the CUDA allocator, fixed-budget deployments) use
muon_newton_schulz_bf16_static, whose scratch is a fixed static device
array of the library.  This test calls it through the C ABI twice in a
row and checks each result against the handle-based muon_newton_schulz_bf16
within the Newton-Schulz tolerance of the parity tests, and that the
calls leave the device's free memory unchanged.

The file is named so that pytest collects it last.
"""

import numpy as np
import pytest

from oracle import muon_oracle as o
from tests.gpu_helpers import rel_fro, u16

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

NS_TOL = 2e-2


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
    return (torch.from_numpy(Xb.view(np.int16)).cuda(), torch.from_numpy(inv).cuda())


@pytest.mark.parametrize("m,n,count", [(256, 512, 5), (2048, 2048, 3), (64, 128, 4)])
def test_static_entry_matches_handle_entry(ns, m, n, count):
    with ns.Handle() as h:
        results = []
        for call in range(2):                      # two calls in a row
            x, inv = _inputs(m, n, count, seed=100 * call + m + n)
            want = torch.zeros((count, m, n), dtype=torch.int16, device="cuda")
            got = torch.full((count, m, n), -1, dtype=torch.int16, device="cuda")
            flag = torch.zeros(1, dtype=torch.int32, device="cuda")
            ns.muon_newton_schulz_bf16(h.value, m, n, count, x, want, inv, 5)
            ns.muon_last_device_error(h.value)
            ns.muon_newton_schulz_bf16_static(m, n, count, x, got, inv, 5, None, flag)
            torch.cuda.synchronize()
            assert int(flag.item()) == 0
            results.append((o.bf16_bits_to_f64(u16(got)), o.bf16_bits_to_f64(u16(want))))
        for g, w in results:
            for i in range(count):
                assert rel_fro(g[i], w[i]) <= NS_TOL


def test_static_entry_allocates_nothing(ns):
    m, n, count = 512, 1024, 3
    x, inv = _inputs(m, n, count, seed=7)
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
