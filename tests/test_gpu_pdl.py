"""Programmatic dependent launch changes when a kernel's CTAs are scheduled,
never what they compute: a step run with it (the default) equals, bit for
bit, the same step in a process started with MUON_PDL=0 (plain serialised
launches).  The mixed shapes exercise both Newton-Schulz kernels (single CTA
for m <= 128, CTA pairs above) and the transposing elementwise kernels."""

import os
import subprocess
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GROUPS = [(384, 256, 3), (128, 64, 4), (512, 1536, 2)]

CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import newton_schulz_03_gb300 as ns
groups = [(384, 256, 3), (128, 64, 4), (512, 1536, 2)]
rng = np.random.default_rng(11)
st = [[torch.from_numpy(rng.standard_normal((k, r, c), dtype=np.float32)).cuda()
       for _ in range(3)] for r, c, k in groups]
with ns.Handle() as h:
    for _ in range(2):
        ns.muon_step(h.value, groups, [t[1] for t in st], [t[2] for t in st],
                     [t[0] for t in st], 0.02, 0.1, 0.95, 5)
    ns.muon_last_device_error(h.value)
torch.cuda.synchronize()
np.savez(sys.argv[2], *[t.cpu().numpy() for g in st for t in (g[0], g[1])])
"""


def run_child(tmp_path, name, pdl):
    env = dict(os.environ)
    env["MUON_PDL"] = "1" if pdl else "0"
    out = str(tmp_path / f"{name}.npz")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, out], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    with np.load(out) as z:
        return [z[k] for k in sorted(z.files, key=lambda s: int(s.split("_")[1]))]


def test_pdl_matches_serialised_launches(tmp_path):
    from newton_schulz_03_gb300 import build_lib
    build_lib.build()
    with_pdl = run_child(tmp_path, "pdl", True)
    without = run_child(tmp_path, "serial", False)
    assert len(with_pdl) == len(without) == 2 * len(GROUPS)
    for a, b in zip(with_pdl, without):
        assert a.shape == b.shape
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    # The step did something: weights moved from their initial values.
    rng = np.random.default_rng(11)
    W0 = rng.standard_normal((3, 384, 256), dtype=np.float32)
    assert not np.array_equal(with_pdl[0], W0)
