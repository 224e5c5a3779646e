"""The packet exchange's rank logic on CPU: two, three and four gloo ranks run
``Exchange.allgather_apply`` (int32 and bitmap packets) and
``Exchange.range_apply`` ("梯度稀疏化：只传输重要的梯度元素", §详细算法流程
step 5 and §与Allreduce的融合).

With no GPU here, the device steps (packet split, index rebase, receive
side) are computed by the oracle through a test-only ``ops`` object; what
is under test is what the exchange itself decides: which collectives carry
which slices, the rank order of the packets, the range bounds and padding,
and the gathering of the updated ranges.  Every rank's result must equal
the oracle's receive side over all ranks' packets in rank order."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle

F32 = np.float32


class OracleOps:
    """The exchange's device steps, computed by the oracle on CPU tensors."""

    @staticmethod
    def aggregate_workspace_size(W, idx_format, n):
        return 1

    @staticmethod
    def packet_split(indices, k, bounds, starts):
        starts.copy_(torch.from_numpy(oracle.packet_split(indices[:k].numpy(), bounds)))
        return starts

    @staticmethod
    def index_rebase(indices, count, base):
        indices[:count] = torch.from_numpy(
            (indices[:count].numpy().astype(np.int64) - int(base)).astype(np.int32))

    @staticmethod
    def sparse_aggregate_apply(values, indices, bitmaps, ks, n, eta, G, w, workspace,
                               idx_format):
        packets = []
        for r, v in enumerate(values):
            p = {"values": v[:ks[r]].numpy()}
            if indices is not None:
                p["indices"] = indices[r][:ks[r]].numpy()
            else:
                p["bitmap"] = bitmaps[r].numpy().view(np.uint32)
            packets.append(p)
        Gn = oracle.sparse_aggregate(packets, n)
        if G is not None:
            G.copy_(torch.from_numpy(Gn))
        w.copy_(torch.from_numpy(oracle.sgd_apply(w.numpy(), Gn, eta)))


def _packet(rank, n, k):
    """Rank r's packet: k ascending distinct indices (ranks overlap, so the
    rank order of the sum matters) and values of mixed scale."""
    rng = np.random.default_rng(100 + rank)
    idx = np.sort(rng.choice(n, k, replace=False)).astype(np.int32)
    vals = (rng.standard_normal(k) * 10.0 ** rng.integers(-6, 0, k)).astype(F32)
    return idx, vals


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, n, k, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    from error_feedback_gradient_gb300 import exchange as ex
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        idx, vals = _packet(rank, n, k)
        w0 = (np.random.default_rng(7).standard_normal(ex.padded_length(n, world))
              * 0.02).astype(F32)
        res = {}
        # all-gather, int32 packets
        x = ex.Exchange(n, k, ex.IDX_INT32, device="cpu", ops=OracleOps)
        w = torch.from_numpy(w0[:n].copy())
        G = torch.empty(n)
        x.allgather_apply(torch.from_numpy(vals), torch.from_numpy(idx), 0.1, G, w)
        res["ag_int32"] = (G.numpy().copy(), w.numpy().copy())
        # all-gather, bitmap packets
        xb = ex.Exchange(n, k, ex.IDX_BITMAP, device="cpu", ops=OracleOps)
        flags = np.zeros(n, bool)
        flags[idx] = True
        bm = torch.from_numpy(oracle.pack_bits(flags).view(np.int32))
        w = torch.from_numpy(w0[:n].copy())
        G = torch.empty(n)
        xb.allgather_apply(torch.from_numpy(vals), bm, 0.1, G, w)
        res["ag_bitmap"] = (G.numpy().copy(), w.numpy().copy())
        # index-range reduce-scatter, twice in a row (the buffers are reused)
        w = torch.from_numpy(w0.copy())
        Gs = torch.empty(x.s)
        for _ in range(2):
            x.range_apply(torch.from_numpy(vals), torch.from_numpy(idx), 0.1, w, Gs)
        res["range"] = (Gs.numpy().copy(), w.numpy().copy(), x.s)
        out.put((rank, res))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def _run(world, n, k):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, n, k, q))
             for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return res


def _expect(world, n, k, w0, steps=1):
    packets = []
    for r in range(world):
        idx, vals = _packet(r, n, k)
        packets.append({"indices": idx, "values": vals})
    G = oracle.sparse_aggregate(packets, n)
    w = w0
    for _ in range(steps):
        w = oracle.sgd_apply(w, G, 0.1)
    return G, w


@pytest.mark.parametrize("world,n,k", [
    (2, 10_007, 400), (3, 5_000, 300), (4, 7_001, 250),
    (3, 1_500, 50),     # rank 2's range lies wholly past n
    (2, 1_000, 0),      # empty packets
    (2, 1_000, 1_000),  # every element in every packet
])
def test_gloo_ranks_exchange_packets(world, n, k):
    from error_feedback_gradient_gb300 import exchange as ex
    res = _run(world, n, k)
    w0 = (np.random.default_rng(7).standard_normal(ex.padded_length(n, world)) * 0.02).astype(F32)
    G, w1 = _expect(world, n, k, w0[:n])
    _, w2 = _expect(world, n, k, w0[:n], steps=2)
    for r in range(world):
        for key in ("ag_int32", "ag_bitmap"):
            g_got, w_got = res[r][key]
            assert np.array_equal(g_got.view(np.uint32), G.view(np.uint32)), (r, key)
            assert np.array_equal(w_got.view(np.uint32), w1.view(np.uint32)), (r, key)
        g_sh, w_got, s = res[r]["range"]
        a = min(r * s, n)
        n_r = max(0, min(n, a + s) - a)    # 0 for a range wholly past n
        assert np.array_equal(g_sh[:n_r].view(np.uint32), G[a:a + n_r].view(np.uint32)), r
        assert np.array_equal(w_got[:n].view(np.uint32), w2.view(np.uint32)), r
        assert np.array_equal(w_got[n:].view(np.uint32), w0[n:].view(np.uint32)), r


def test_shard_lengths():
    from error_feedback_gradient_gb300 import exchange as ex
    assert ex.shard_length(10_007, 2) == 5120 and ex.padded_length(10_007, 2) == 10_240
    assert ex.shard_length(1 << 31, 8) == 1 << 28
    assert ex.shard_length(1, 4) == 1024
    for n in (1, 1023, 1024, 1025, 5_000_001):
        for world in (1, 2, 3, 8):
            s = ex.shard_length(n, world)
            assert s % 1024 == 0 and world * s >= n and (world * (s - 1024) < n or s == 1024)
