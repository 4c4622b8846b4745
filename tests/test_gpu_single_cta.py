"""The single-CTA Newton-Schulz kernels at every size (MUON_NS_PAIR=0).

By default matrices with more than 128 rows run on CTA pairs; the switch
keeps every product on single CTAs (128 x 256 tiles, symmetric results
stored in full with mirrored stores), for comparisons.  That path must
compute the same iteration: each matrix is checked against the FP64 oracle
("Frontier Pre-training at Microsoft AI", Method details §5, resharding
step 3: the quintic Newton-Schulz map on the BF16 momentum) within the
2e-2 bar, on shapes that span several tiles and end in ragged ones.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

from oracle import muon_oracle as o

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SHAPES = [(256, 512, 2), (200, 392, 2), (640, 1024, 1), (384, 384, 2)]
NS_TOL = 2e-2

CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import newton_schulz_03_gb300 as ns
data = np.load(sys.argv[2])
outs = []
with ns.Handle() as h:
    for i in range(int(data["n"])):
        x = torch.from_numpy(data[f"x{i}"]).cuda()
        inv = torch.from_numpy(data[f"inv{i}"]).cuda()
        count, m, n = x.shape
        out = torch.zeros_like(x)
        ns.muon_newton_schulz_bf16(h.value, m, n, count, x, out, inv, 5)
        ns.muon_last_device_error(h.value)
        outs.append(out.cpu().numpy())
np.savez(sys.argv[3], *outs)
"""


def test_single_cta_path_matches_the_oracle(tmp_path):
    from newton_schulz_03_gb300 import build_lib
    build_lib.build()
    rng = np.random.default_rng(31)
    inputs, arrays = {}, []
    for i, (m, n, count) in enumerate(SHAPES):
        xb = o.bf16_rne_bits(rng.standard_normal((count, m, n), dtype=np.float32))
        xf = o.bf16_bits_to_f64(xb)
        inv = np.array([1.0 / (np.linalg.norm(xf[k]) + o.NORM_EPS) for k in range(count)],
                       dtype=np.float32)
        inputs[f"x{i}"] = xb.view(np.int16)
        inputs[f"inv{i}"] = inv
        arrays.append((xf, inv))
    inputs["n"] = np.array(len(SHAPES))
    src, dst = str(tmp_path / "in.npz"), str(tmp_path / "out.npz")
    np.savez(src, **inputs)
    env = dict(os.environ)
    env["MUON_NS_PAIR"] = "0"
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, src, dst], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    with np.load(dst) as z:
        outs = [z[k] for k in sorted(z.files, key=lambda s: int(s.split("_")[1]))]
    for (m, n, count), (xf, inv), out in zip(SHAPES, arrays, outs):
        got = o.bf16_bits_to_f64(out.view(np.uint16))
        for k in range(count):
            ref = o.newton_schulz(xf[k], 1.0 / float(inv[k]))
            err = np.linalg.norm(got[k] - ref) / np.linalg.norm(ref)
            assert err <= NS_TOL, f"{m}x{n} matrix {k}: {err:.3e}"
