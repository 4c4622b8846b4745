"""The Muon step under ZeRO data parallelism: resharding around the
Newton-Schulz products.

"Frontier Pre-training at Microsoft AI", Method details §5, resharding
pipeline, and "Microsoft Reveals MAI-Base-2 Training Recipe", section "How
to Make Parameter Updates Faster and More Stable?": the optimizer state is
sharded over the data-parallel ranks, but the Newton-Schulz iteration needs
whole matrices, so one step is

  1. every rank updates its FP32 momentum shard and casts it to BF16;
  2. an all-to-all per group of same-shape parameters gives every rank the
     complete matrices it owns;
  3. the owners orthogonalise them locally;
  4. a second all-to-all returns each rank the update of its shard;
  5. every rank applies the update to its FP32 weight shard.

Router weights are replicated instead of sharded (the pages' tuning
bullets): every rank updates the whole momentum, so the first exchange is
skipped, each router matrix is orthogonalised by one owner, and a single
all-gather hands every rank every router's update.  The exchange layout of
a group list is computed once and reused ("resharding metadata caching").

Layout.  Group g (``count`` matrices of rows x cols, E = rows * cols
elements each) is one flat buffer of count * E elements split into
``world`` contiguous shards of S = ceil(count * E / world) elements: rank q
holds [q S, min((q + 1) S, count * E)).  The owners of whole matrices come
from ``muon_partition`` (one contiguous slice of each group per rank, ranks
in order), so the piece rank q sends rank p is the intersection of q's
shard with p's slice, the pieces a shard sends are consecutive in rank
order, and the pieces an owner receives tile its slice in rank order: each
exchange is one ``all_to_all_single`` per group on the buffers as they lie,
with no packing.  BF16 payloads travel as bytes.

The local compute goes through an ``ops`` object: ``LibraryOps`` runs it in
this package's kernels on the GPU (``muon_shard_momentum_cast``,
``muon_norm_from_sumsq``, ``muon_transpose_bf16``,
``muon_newton_schulz_bf16``, ``muon_shard_apply``); the exchanges go
through a ``comm`` object, ``TorchDistComm`` for ``torch.distributed``
(NCCL on GPUs, gloo on CPUs), started asynchronously so that one group's
exchanges overlap another group's Newton-Schulz products (the pages'
cross-batch prefetch).  Newton-Schulz on the owner needs both sides
of the matrix to be multiples of 8 (the products' 16-byte TMA pitch).
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Sequence, Tuple

from . import _native as nat


@dataclass
class GroupLayout:
    """Exchange layout of one group (all counts in elements)."""
    rows: int
    cols: int
    count: int
    scale: float
    replicated: bool
    shard: List[Tuple[int, int]] = field(default_factory=list)   # [rank] -> [begin, end)
    own: List[Tuple[int, int]] = field(default_factory=list)     # [rank] -> (first, count)
    send: List[List[int]] = field(default_factory=list)          # [q][p] elements q -> p
    touched: List[Tuple[int, int]] = field(default_factory=list)  # [rank] -> matrices [k0, k1)

    @property
    def elems(self) -> int:
        return self.rows * self.cols

    @property
    def total(self) -> int:
        return self.count * self.elems

    def sums_range(self, q: int, p: int) -> Tuple[int, int]:
        """Matrices of p's slice that q's shard touches: [lo, hi), global."""
        f, c = self.own[p]
        k0, k1 = self.touched[q]
        lo, hi = max(k0, f), min(k1, f + c)
        return (lo, hi) if hi > lo else (lo, lo)


class ReshardPlan:
    """Shards, owners and exchange sizes of a group list over `world`
    ranks.  `groups` are (rows, cols, count[, update_scale]); groups whose
    index is in `replicated` are held whole by every rank."""

    def __init__(self, groups: Sequence, world: int, replicated: Sequence[int] = (),
                 ns_steps: int = 5):
        if world < 1:
            raise ValueError("world must be >= 1")
        self.world = world
        self.ns_steps = ns_steps
        slices, self.rank_seconds = nat.muon_partition(groups, world, ns_steps)
        rep = set(int(i) for i in replicated)
        self.groups: List[GroupLayout] = []
        for g, spec in enumerate(groups):
            rows, cols, count = int(spec[0]), int(spec[1]), int(spec[2])
            scale = float(spec[3]) if len(spec) > 3 else 1.0
            gl = GroupLayout(rows, cols, count, scale, g in rep)
            own = [(0, 0)] * world
            for r in range(world):
                for gg, first, c in slices[r]:
                    if gg == g:
                        own[r] = (first, c)
            gl.own = own
            E, total = gl.elems, gl.total
            if gl.replicated:
                gl.shard = [(0, total)] * world
            else:
                S = -(-total // world)
                gl.shard = [(min(q * S, total), min((q + 1) * S, total)) for q in range(world)]
            gl.touched = [((b // E, (e - 1) // E + 1) if e > b else (b // E, b // E))
                          for b, e in gl.shard]
            gl.send = [[0] * world for _ in range(world)]
            if not gl.replicated:
                for q, (b, e) in enumerate(gl.shard):
                    for p, (f, c) in enumerate(own):
                        lo, hi = max(b, f * E), min(e, (f + c) * E)
                        gl.send[q][p] = max(0, hi - lo)
            self.groups.append(gl)

    def shard_elems(self, g: int, rank: int) -> int:
        b, e = self.groups[g].shard[rank]
        return e - b


class _Done:
    """Handle of an exchange that already completed."""

    def wait(self) -> None:
        return None


class TorchDistComm:
    """The exchanges over torch.distributed (default process group).  With
    `async_op` the collective is only started and a handle with wait() is
    returned (NCCL runs it on its own stream, ordered after the work
    already queued on the caller's stream; wait() orders the caller's stream
    after it)."""

    def all_to_all(self, out, inp, out_splits, in_splits, async_op: bool = False):
        import torch.distributed as dist
        work = dist.all_to_all_single(out, inp, output_split_sizes=list(out_splits),
                                      input_split_sizes=list(in_splits), async_op=async_op)
        return work if async_op else _Done()

    def all_gather(self, out_list, inp, async_op: bool = False):
        import torch.distributed as dist
        work = dist.all_gather(out_list, inp, async_op=async_op)
        return work if async_op else _Done()


def _bytes(t):
    """A contiguous tensor as a flat uint8 view (BF16 payloads travel as bytes)."""
    import torch
    return t.contiguous().view(-1).view(torch.uint8)


class LibraryOps:
    """The local compute of the resharded step in this package's kernels
    (CUDA tensors; BF16 payloads held as int16 bit patterns)."""

    def __init__(self, handle: int, stream=None):
        self.h = handle
        self.stream = stream

    def empty(self, n, dtype, like):
        import torch
        return torch.empty(n, dtype=dtype, device=like.device)

    def zeros(self, shape, dtype, like):
        import torch
        return torch.zeros(shape, dtype=dtype, device=like.device)

    def shard_cast(self, M, G, mu, begin, end, E):
        """Step 1 on a shard: (X bits, per-piece sums of squares)."""
        import torch
        X = torch.empty(end - begin, dtype=torch.int16, device=M.device)
        k0, k1 = begin // E, ((end - 1) // E + 1 if end > begin else begin // E)
        sums = torch.empty(max(0, k1 - k0), dtype=torch.float32, device=M.device)
        nat.muon_shard_momentum_cast(self.h, begin, end, E, M, G, mu, X, sums, self.stream)
        return X, sums

    def orthogonalise(self, X, sums, rows, cols, steps):
        """Step 3 on the owner: X (count, rows, cols) BF16 bits, sums (count,
        parts) -> the update O (count, rows, cols) BF16 bits."""
        import torch
        count = X.shape[0]
        if count == 0:
            return X
        m, n = min(rows, cols), max(rows, cols)
        if rows > cols:
            Xw = torch.empty((count, m, n), dtype=torch.int16, device=X.device)
            nat.muon_transpose_bf16(self.h, rows, cols, count, X, Xw, self.stream)
        else:
            Xw = X.contiguous()
        inv = torch.empty(count, dtype=torch.float32, device=X.device)
        nat.muon_norm_from_sumsq(self.h, m, n, count, sums.shape[1], sums.contiguous(), Xw, inv,
                                 self.stream)
        Ow = torch.empty_like(Xw)
        nat.muon_newton_schulz_bf16(self.h, m, n, count, Xw, Ow, inv, steps, None, self.stream)
        if rows > cols:
            O = torch.empty((count, rows, cols), dtype=torch.int16, device=X.device)
            nat.muon_transpose_bf16(self.h, m, n, count, Ow, O, self.stream)
            return O
        return Ow

    def apply(self, W, O, lr, wd, scale):
        nat.muon_shard_apply(self.h, W.numel(), W, O, lr, wd, scale, self.stream)


def resharded_step(plan: ReshardPlan, rank: int, state: Sequence, lr: float, wd: float,
                   mu: float, ops, comm=None, overlap: bool = True) -> None:
    """One Muon step of rank `rank`.  state[g] = (M, G, W) of this rank: 1-D
    FP32 tensors of the rank's shard of group g (its whole buffer for a
    replicated group); M and W are updated in place.

    With `overlap` (the pages' cross-batch prefetch) the exchanges are
    started asynchronously: every group's first exchange is under way
    before the first group is orthogonalised, and each group's return
    exchange runs while the next groups are orthogonalised, so the
    collectives of one group overlap the Newton-Schulz products of
    another.  Every rank issues the collectives in the same order (group
    by group), as the collectives require."""
    comm = comm or TorchDistComm()
    world = plan.world
    steps = plan.ns_steps
    # Phase 1: shard-side update and cast; exchange 1 of every group started.
    inbound = []
    for g, gl in enumerate(plan.groups):
        M, G, W = state[g]
        E = gl.elems
        if gl.replicated:
            # The whole momentum is here (no first exchange).
            X, sums = ops.shard_cast(M, G, mu, 0, gl.total, E)
            inbound.append((X, sums, None, []))
            continue
        b, e = gl.shard[rank]
        X, sums = ops.shard_cast(M, G, mu, b, e, E)
        first, own = gl.own[rank]
        # Pieces of X to the owners of their matrices.
        Xown = ops.empty(own * E, X.dtype, X)
        isz = X.element_size()
        w1 = comm.all_to_all(_bytes(Xown), _bytes(X),
                             [gl.send[q][rank] * isz for q in range(world)],
                             [gl.send[rank][p] * isz for p in range(world)], async_op=overlap)
        # The pieces' sums of squares go with them: rank q sends p the sums
        # of the matrices of p's slice that q's shard touches.
        k0 = gl.touched[rank][0]
        out_n = [gl.sums_range(q, rank)[1] - gl.sums_range(q, rank)[0] for q in range(world)]
        in_n = [gl.sums_range(rank, p)[1] - gl.sums_range(rank, p)[0] for p in range(world)]
        send_sums = ops.empty(sum(in_n), sums.dtype, X)
        at = 0
        for p in range(world):
            lo, hi = gl.sums_range(rank, p)
            send_sums[at:at + hi - lo] = sums[lo - k0:hi - k0]
            at += hi - lo
        recv_sums = ops.empty(sum(out_n), sums.dtype, X)
        ssz = sums.element_size()
        w2 = comm.all_to_all(_bytes(recv_sums), _bytes(send_sums), [n * ssz for n in out_n],
                             [n * ssz for n in in_n], async_op=overlap)
        inbound.append((X, send_sums, (Xown, recv_sums), [w1, w2]))
    # Phase 2: orthogonalise each group as its pieces arrive; start its return.
    outbound = []
    for g, gl in enumerate(plan.groups):
        E, r, c = gl.elems, gl.rows, gl.cols
        first, own = gl.own[rank]
        X, _, recv, works = inbound[g]
        for w in works:
            w.wait()
        if gl.replicated:
            sums = inbound[g][1]
            Xo = X[first * E:(first + own) * E].view(own, r, c)
            So = sums[first:first + own].view(own, 1)
            Oo = ops.orthogonalise(Xo, So, r, c, steps)
            # One all-gather of the owners' updates (padded to the largest slice).
            most = max(cnt for _, cnt in gl.own) * E
            buf = ops.zeros(most, Oo.dtype, X)
            if own:
                buf[:own * E] = Oo.reshape(-1)
            parts = [ops.empty(most, Oo.dtype, X) for _ in range(world)]
            w = comm.all_gather([_bytes(p) for p in parts], _bytes(buf), async_op=overlap)
            outbound.append((parts, buf, w))
            continue
        Xown, recv_sums = recv
        S = ops.zeros((own, world), recv_sums.dtype, X)
        at = 0
        for q in range(world):
            lo, hi = gl.sums_range(q, rank)
            if hi > lo:
                S[lo - first:hi - first, q] = recv_sums[at:at + hi - lo]
            at += hi - lo
        O = ops.orthogonalise(Xown.view(own, r, c), S, r, c, steps)
        b, e = gl.shard[rank]
        Oshard = ops.empty(e - b, O.dtype, X)
        isz = O.element_size()
        w = comm.all_to_all(_bytes(Oshard), _bytes(O),
                            [gl.send[rank][p] * isz for p in range(world)],
                            [gl.send[q][rank] * isz for q in range(world)], async_op=overlap)
        outbound.append((Oshard, O, w))
    # Phase 3: apply each shard's update once it is back.
    for g, gl in enumerate(plan.groups):
        M, G, W = state[g]
        E = gl.elems
        if gl.replicated:
            parts, _, w = outbound[g]
            w.wait()
            O = ops.empty(gl.total, parts[0].dtype, parts[0])
            for p, (f, cnt) in enumerate(gl.own):
                O[f * E:(f + cnt) * E] = parts[p][:cnt * E]
            ops.apply(W, O, lr, wd, gl.scale)
            continue
        Oshard, _, w = outbound[g]
        w.wait()
        ops.apply(W, Oshard, lr, wd, gl.scale)
