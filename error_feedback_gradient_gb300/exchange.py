"""Packet exchange between data-parallel ranks, around the receive side.

"梯度稀疏化：只传输重要的梯度元素", §详细算法流程 step 5 (each worker packs its
non-zero values and their indices; the packets are exchanged with
Allgather and every receiver sums them locally) and §与Allreduce的融合 (the
sparse packets go directly through the collective library's Allgather).
One rank is one worker; rank order is worker order, so the receive side
sums the packets in rank order exactly as ``sparse_aggregate_apply`` does
for W local workers.  Two schemes:

``allgather_apply``
    Every rank all-gathers the fixed-size packets of all ranks (values, and
    int32 indices or bitmaps) and runs ``sparse_aggregate_apply`` on the
    ``world`` packets: every rank gets the dense G and updates its whole
    replica of w.  Traffic per rank: (world - 1) packets.
``range_apply``
    Index-range reduce-scatter.  Rank q owns the indices
    [q * s, (q + 1) * s) (s = ``shard_length(n, world)``).  Each rank splits
    its ascending packet at the range bounds (``packet_split``, a binary
    search on the device), the slices go to their owners with one
    all-to-all each for values and indices, every owner rebases the slices
    it received to its range (``index_rebase``) and runs the receive side on
    its range alone, and the ranks all-gather the updated ranges of w.
    Traffic per rank: about one packet plus n / world weights.  int32
    packets only (a bitmap slice would need a population-count prefix).

The collectives are plain ``torch.distributed`` calls (NCCL on GPUs); every
arithmetic step runs in the library's kernels through ``binding``.  ``ops``
is the object whose methods run those steps; the default is ``binding``
itself, and it raises when the library is missing (there is no fallback).

Every rank must pass the same n, k and format (the packets are fixed-size)
and the same w (data-parallel replicas).  The host reads the split sizes of
``range_apply`` back (one small device-to-host copy per call), since the
all-to-all needs them.
"""

from __future__ import annotations

from typing import Optional

import torch
import torch.distributed as dist

from . import binding

IDX_INT32 = binding.IDX_INT32
IDX_BITMAP = binding.IDX_BITMAP
_ALIGN = 1024   # shard lengths are multiples of the receive side's tile


def _world(group) -> tuple:
    if group is None and not (dist.is_available() and dist.is_initialized()):
        raise RuntimeError("torch.distributed is not initialised")
    return dist.get_rank(group), dist.get_world_size(group)


def shard_length(n: int, world: int) -> int:
    """Length s of each rank's index range in ``range_apply``: ceil(n / world)
    rounded up to a multiple of 1024."""
    s = -(-int(n) // int(world))
    return -(-s // _ALIGN) * _ALIGN


def padded_length(n: int, world: int) -> int:
    """Elements w must hold for ``range_apply``: world * shard_length."""
    return int(world) * shard_length(n, world)


class Exchange:
    """Buffers of one exchange configuration (n, k, format, world), reused
    across steps.  ``allgather_apply`` and ``range_apply`` are the two
    schemes described in the module docstring."""

    def __init__(self, n: int, k: int, idx_format: int = IDX_INT32, group=None,
                 device=None, ops=binding):
        self.rank, self.world = _world(group)
        self.group, self.ops = group, ops
        self.n, self.k, self.fmt = int(n), int(k), int(idx_format)
        if self.fmt not in (IDX_INT32, IDX_BITMAP):
            raise ValueError("idx_format must be IDX_INT32 or IDX_BITMAP")
        if not 0 <= self.k <= self.n:
            raise ValueError("need 0 <= k <= n")
        dev = torch.device(device) if device is not None else (
            torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available()
            else torch.device("cpu"))
        self.device = dev
        W, k = self.world, self.k
        self.values_all = torch.empty(W * k, dtype=torch.float32, device=dev)
        if self.fmt == IDX_INT32:
            self.index_all = torch.empty(W * k, dtype=torch.int32, device=dev)
        else:
            self.nwords = (self.n + 31) // 32
            self.index_all = torch.empty(W * self.nwords, dtype=torch.int32, device=dev)
        self.ws_all = torch.empty(max(1, ops.aggregate_workspace_size(W, self.fmt, self.n)),
                                  dtype=torch.uint8, device=dev)
        self.s = shard_length(self.n, W)
        if self.fmt == IDX_INT32:
            # a range receives at most W * k entries (all of every packet)
            self.recv_values = torch.empty(max(1, W * k), dtype=torch.float32, device=dev)
            self.recv_index = torch.empty(max(1, W * k), dtype=torch.int32, device=dev)
            self.ws_range = torch.empty(
                max(1, ops.aggregate_workspace_size(W, IDX_INT32, self.s)), dtype=torch.uint8,
                device=dev)
            self.bounds = [min(q * self.s, self.n) for q in range(W)] + [self.n]
            self.starts = torch.empty(W + 1, dtype=torch.int64, device=dev)
            self.starts_all = torch.empty(W * (W + 1), dtype=torch.int64, device=dev)

    # -- scheme 1 ---------------------------------------------------------
    def allgather_apply(self, values: torch.Tensor, index: torch.Tensor, eta: float,
                        G: Optional[torch.Tensor], w: torch.Tensor) -> None:
        """All-gather every rank's packet (values[k], and indices[k] or
        bitmap[ceil(n/32)] as int32), then G = the rank-order sum of the
        world packets and w -= eta * G where some packet touches it."""
        W, k = self.world, self.k
        dist.all_gather_into_tensor(self.values_all, values[:k].contiguous(), group=self.group)
        idx = index[:k] if self.fmt == IDX_INT32 else index[:self.nwords]
        dist.all_gather_into_tensor(self.index_all, idx.contiguous(), group=self.group)
        vals = [self.values_all[r * k:(r + 1) * k] for r in range(W)]
        if self.fmt == IDX_INT32:
            inds = [self.index_all[r * k:(r + 1) * k] for r in range(W)]
            self.ops.sparse_aggregate_apply(vals, inds, None, [k] * W, self.n, eta, G, w,
                                            self.ws_all, IDX_INT32)
        else:
            bms = [self.index_all[r * self.nwords:(r + 1) * self.nwords] for r in range(W)]
            self.ops.sparse_aggregate_apply(vals, None, bms, [k] * W, self.n, eta, G, w,
                                            self.ws_all, IDX_BITMAP)

    # -- scheme 2 ---------------------------------------------------------
    def range_apply(self, values: torch.Tensor, indices: torch.Tensor, eta: float,
                    w: torch.Tensor, G_shard: Optional[torch.Tensor] = None) -> None:
        """Index-range reduce-scatter of int32 packets.  w holds at least
        ``padded_length(n, world)`` elements (the tail past n is never
        touched by the update and is gathered as it is); on return every
        rank holds the whole updated w.  G_shard, if given, receives the
        dense G of this rank's range (its first min(s, n - rank * s)
        elements)."""
        if self.fmt != IDX_INT32:
            raise ValueError("range_apply takes int32 packets")
        W, k, s, r = self.world, self.k, self.s, self.rank
        if w.numel() < W * s:
            raise ValueError(f"w must hold padded_length(n, world) = {W * s} elements")
        # 1. this rank's slice for every range
        self.ops.packet_split(indices, k, self.bounds, self.starts)
        dist.all_gather_into_tensor(self.starts_all, self.starts, group=self.group)
        st = self.starts_all.view(W, W + 1).cpu().tolist()   # st[src][q]
        send = [st[r][q + 1] - st[r][q] for q in range(W)]
        recv = [st[src][r + 1] - st[src][r] for src in range(W)]
        lo, total = st[r][0], sum(recv)
        # 2. slices to their owners (source-rank order on arrival)
        rv, ri = self.recv_values[:total], self.recv_index[:total]
        dist.all_to_all_single(rv, values[lo:lo + sum(send)].contiguous(), recv, send,
                               group=self.group)
        dist.all_to_all_single(ri, indices[lo:lo + sum(send)].contiguous(), recv, send,
                               group=self.group)
        # 3. receive side on this rank's range
        a = min(r * s, self.n)
        n_r = max(0, min(self.n, a + s) - a)
        self.ops.index_rebase(ri, total, a)
        offs = [0]
        for c in recv:
            offs.append(offs[-1] + c)
        vals = [rv[offs[q]:offs[q + 1]] for q in range(W)]
        inds = [ri[offs[q]:offs[q + 1]] for q in range(W)]
        w_own = w[r * s:(r + 1) * s]
        if n_r > 0:
            self.ops.sparse_aggregate_apply(vals, inds, None, recv, n_r, eta,
                                            None if G_shard is None else G_shard[:n_r],
                                            w_own[:n_r], self.ws_range, IDX_INT32)
        # 4. every rank gets every updated range
        dist.all_gather_into_tensor(w[:W * s], w_own, group=self.group)
