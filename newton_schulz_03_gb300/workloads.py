"""Synthetic workloads: shapes, hyper-parameters and seeded input generators.

This module holds no arithmetic of the method.  It only describes the
parameter shapes of the model family (MAI-Base-2 ladder rungs, "Frontier
Pre-training at Microsoft AI", Method details §2 and the model
architecture table) and draws seeded random inputs of those shapes.  Both
the tests (which feed the CPU oracle and the GPU path the same bytes) and
the benchmark use it.

Shapes follow PyTorch's (out_features, in_features) convention: an expert
up-projection is (intermediate x hidden), a down-projection is
(hidden x intermediate).  A tall matrix is orthogonalised as its
transpose, so an up/down pair shares one Newton-Schulz batch.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Optional, Tuple

import numpy as np


@dataclass(frozen=True)
class GroupSpec:
    """One caller group: ``count`` contiguous row-major FP32 matrices."""
    name: str
    rows: int
    cols: int
    count: int
    w_std: float = 0.02          # weights N(0, w_std)
    g_std: float = 1e-3          # gradient N(0, g_std)
    m_std: float = 1e-3          # momentum N(0, m_std)
    expert_scaled: bool = False  # multiply G and M of matrix e by exp(l_e)
    zero_index: Optional[int] = None  # matrix whose G and M are all zero

    @property
    def wide(self) -> Tuple[int, int]:
        return (min(self.rows, self.cols), max(self.rows, self.cols))

    @property
    def numel(self) -> int:
        return self.rows * self.cols * self.count


@dataclass(frozen=True)
class Workload:
    name: str
    description: str
    groups: Tuple[GroupSpec, ...]
    mu: float = 0.95
    lr: float = 0.02
    wd: float = 0.1
    ns_steps: int = 5
    layers: int = 1              # the step is repeated over this many layers
    seed_base: int = 0
    notes: str = ""

    @property
    def matrices_per_layer(self) -> int:
        return sum(g.count for g in self.groups)

    @property
    def matrices(self) -> int:
        return self.layers * self.matrices_per_layer

    def wide_batches(self) -> Dict[Tuple[int, int], int]:
        out: Dict[Tuple[int, int], int] = {}
        for g in self.groups:
            out[g.wide] = out.get(g.wide, 0) + g.count
        return out


def _experts(prefix: str, hidden: int, inter: int, n: int, **kw) -> List[GroupSpec]:
    return [GroupSpec(f"{prefix}.up", inter, hidden, n, expert_scaled=True, **kw),
            GroupSpec(f"{prefix}.down", hidden, inter, n, expert_scaled=True, **kw)]


WORKLOADS: Dict[str, Workload] = {
    # 4 tall 128x64 matrices, every input N(0, 1): exercises transpose to
    # wide and tiles larger than the matrix.
    "tiny": Workload(
        "tiny", "4 FP32 matrices of 128x64 (tall), N(0,1) inputs",
        (GroupSpec("tiny", 128, 64, 4, w_std=1.0, g_std=1.0, m_std=1.0),),
        seed_base=0),
    # Dense ladder rung L=24, hidden 2048: Q, K, V, O of 24 layers.
    "l24_attention": Workload(
        "l24_attention", "rung L=24: 96 square 2048x2048 attention projections",
        (GroupSpec("attn", 2048, 2048, 96),),
        seed_base=1000),
    # MoE rung L=48, hidden 4096: 512 routed experts, up and down.
    "l48_experts": Workload(
        "l48_experts", "rung L=48: 512 experts x (up 1536x4096, down 4096x1536)",
        tuple(_experts("expert", 4096, 1536, 512, zero_index=7)),
        seed_base=2000),
    # One full-scale layer (L=102, hidden 8704).
    "l102_layer": Workload(
        "l102_layer", "rung L=102 layer: 512 experts x (2048x8704, 8704x2048), "
        "shared expert 8704x13056 + 13056x8704, 4 attention 8704x8704",
        tuple(_experts("expert", 8704, 2048, 512, zero_index=7)) + (
            GroupSpec("shared.up", 13056, 8704, 1),
            GroupSpec("shared.down", 8704, 13056, 1),
            GroupSpec("attn", 8704, 8704, 4)),
        seed_base=3000),
    # Whole-model step of rung L=48: one layer's state, stepped 48 times.
    "l48_model": Workload(
        "l48_model", "rung L=48 whole model: 48 layers x (4 attention 4096x4096, "
        "shared 4096x6144 + 6144x4096, 512 experts x (1536x4096, 4096x1536), "
        "router 512x4096); one layer resident, stepped 48 times",
        (GroupSpec("attn", 4096, 4096, 4),
         GroupSpec("shared.up", 6144, 4096, 1),
         GroupSpec("shared.down", 4096, 6144, 1))
        + tuple(_experts("expert", 4096, 1536, 512, zero_index=7))
        + (GroupSpec("router", 512, 4096, 1),),
        layers=48, seed_base=4000),
}


def group_seed(workload: Workload, group_index: int) -> int:
    return workload.seed_base + group_index


def expert_log_scales(workload: Workload, count: int) -> np.ndarray:
    """l_e ~ Laplace(0, 1) per expert, shared by an expert's up and down
    matrices (one draw per workload)."""
    rng = np.random.default_rng(workload.seed_base + 999)
    return rng.laplace(0.0, 1.0, size=count)


def make_group_numpy(workload: Workload, group_index: int):
    """(W, M, G) as FP32 numpy arrays of shape [count, rows, cols]."""
    g = workload.groups[group_index]
    rng = np.random.default_rng(group_seed(workload, group_index))
    shape = (g.count, g.rows, g.cols)
    W = (rng.standard_normal(shape, dtype=np.float32) * np.float32(g.w_std))
    M = (rng.standard_normal(shape, dtype=np.float32) * np.float32(g.m_std))
    G = (rng.standard_normal(shape, dtype=np.float32) * np.float32(g.g_std))
    if g.expert_scaled:
        sc = np.exp(expert_log_scales(workload, g.count)).astype(np.float32)
        M *= sc[:, None, None]
        G *= sc[:, None, None]
    if g.zero_index is not None and g.zero_index < g.count:
        M[g.zero_index] = 0.0
        G[g.zero_index] = 0.0
    return W, M, G


def make_group_torch(workload: Workload, group_index: int, device: str = "cuda",
                     first: int = 0, count: Optional[int] = None):
    """(W, M, G) as FP32 torch tensors [count, rows, cols] for matrices
    first .. first+count-1 of a group (default: the whole group), drawn on
    ``device`` (used where the host cannot hold a whole workload).  Matrix
    i is drawn by its own seeded generator, so a slice of a group has the
    same values whether it is made alone (one rank's share) or as part of
    the whole group."""
    import torch
    g = workload.groups[group_index]
    if count is None:
        count = g.count - first
    shape = (count, g.rows, g.cols)
    W = torch.empty(shape, device=device, dtype=torch.float32)
    M = torch.empty(shape, device=device, dtype=torch.float32)
    G = torch.empty(shape, device=device, dtype=torch.float32)
    gen = torch.Generator(device=device)
    for j in range(count):
        gen.manual_seed((group_seed(workload, group_index) << 20) + first + j)
        W[j].normal_(0.0, g.w_std, generator=gen)
        M[j].normal_(0.0, g.m_std, generator=gen)
        G[j].normal_(0.0, g.g_std, generator=gen)
    if g.expert_scaled:
        sc = np.exp(expert_log_scales(workload, g.count)[first:first + count]).astype(np.float32)
        sc = torch.from_numpy(sc).to(device)
        M.mul_(sc[:, None, None])
        G.mul_(sc[:, None, None])
    if g.zero_index is not None and first <= g.zero_index < first + count:
        M[g.zero_index - first].zero_()
        G[g.zero_index - first].zero_()
    return W, M, G


def random_wide_bf16_like(m: int, n: int, count: int, seed: int, std: float = 1.0):
    """Seeded FP32 matrices [count, m, n] for Newton-Schulz-only tests."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal((count, m, n), dtype=np.float32) * np.float32(std)
