"""GPU parity of the packet exchange's device steps and of the exchange on
one GPU ("梯度稀疏化：只传输重要的梯度元素", §详细算法流程 step 5 and
§与Allreduce的融合): ef_packet_split and ef_index_rebase bit for bit against
the oracle, both exchange schemes in a world-size-1 NCCL group, and the
index-range scheme's compute for four ranks simulated on one GPU."""

import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

import error_feedback_gradient_gb300 as efg
from error_feedback_gradient_gb300 import exchange as ex
import oracle
from efcheck import assert_bits_equal, host

pytestmark = pytest.mark.gpu
DEV = "cuda"
F32 = np.float32


def _sorted_packet(n, k, seed):
    rng = np.random.default_rng(seed)
    if k > n // 2:
        idx = np.sort(rng.permutation(n)[:k])
    else:
        idx = np.unique(rng.integers(0, n, int(k * 1.2) + 8))[:k]
        while idx.size < k:
            idx = np.unique(np.concatenate([idx, rng.integers(0, n, k)]))[:k]
    return idx.astype(np.int32)


@pytest.mark.parametrize("n,k,nparts", [(100, 0, 3), (1000, 1, 1), (1000, 999, 7),
                                        (1_000_003, 5000, 8), (1 << 31, 1 << 22, 64),
                                        (1 << 20, 3000, 1024)])
def test_packet_split_matches_oracle(n, k, nparts):
    idx = _sorted_packet(n, k, n % 1000 + k)
    rng = np.random.default_rng(k + 5)
    bounds = np.sort(rng.integers(0, n + 1, nparts + 1))
    bounds[0], bounds[-1] = 0, n
    bounds[nparts // 2] = bounds[max(0, nparts // 2 - 1)]          # an empty range
    if k:
        bounds[min(nparts, 1)] = max(bounds[min(nparts, 1) - 1], int(idx[k // 2]))  # on an entry
    bounds = np.maximum.accumulate(bounds)
    d_idx = torch.from_numpy(idx).to(DEV)
    got = efg.binding.packet_split(d_idx, k, bounds.tolist())
    want = oracle.packet_split(idx, bounds)
    assert host(got).tolist() == want.tolist()


def test_packet_split_bounds_outside_and_refusals():
    idx = torch.tensor([3, 9, 40, 41], dtype=torch.int32, device=DEV)
    got = efg.binding.packet_split(idx, 4, [-5, 0, 41, 42, 1 << 40])
    assert host(got).tolist() == oracle.packet_split([3, 9, 40, 41], [-5, 0, 41, 42, 1 << 40]).tolist()
    with pytest.raises(efg.EFError):
        efg.binding.packet_split(idx, 4, [5, 3])       # bounds must not decrease
    with pytest.raises(efg.EFError):
        efg.binding.packet_split(idx, 4, [0])          # at least one range


def test_index_rebase_exact():
    idx = _sorted_packet(1 << 30, 100_003, 3)
    d = torch.from_numpy(idx).to(DEV)
    efg.binding.index_rebase(d, 100_000, 12345)
    want = idx.copy()
    want[:100_000] = (idx[:100_000].astype(np.int64) - 12345).astype(np.int32)
    assert np.array_equal(host(d), want)
    efg.binding.index_rebase(d, 0, 7)                  # empty: nothing happens
    assert np.array_equal(host(d), want)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.fixture
def nccl_world1():
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0,
                            world_size=1)
    try:
        yield
    finally:
        dist.destroy_process_group()


def test_exchange_world1_nccl(nccl_world1):
    n, k = 1_000_003, 1000
    idx = _sorted_packet(n, k, 11)
    vals = (np.random.default_rng(12).standard_normal(k) * 1e-3).astype(F32)
    w0 = (np.random.default_rng(13).standard_normal(ex.padded_length(n, 1)) * 0.02).astype(F32)
    G_want = oracle.sparse_aggregate([{"indices": idx, "values": vals}], n)
    w_want = oracle.sgd_apply(w0[:n], G_want, 0.1)
    d_idx, d_val = torch.from_numpy(idx).to(DEV), torch.from_numpy(vals).to(DEV)
    for fmt in (ex.IDX_INT32, ex.IDX_BITMAP):
        x = ex.Exchange(n, k, fmt)
        w = torch.from_numpy(w0[:n].copy()).to(DEV)
        G = torch.empty(n, device=DEV)
        if fmt == ex.IDX_INT32:
            x.allgather_apply(d_val, d_idx, 0.1, G, w)
        else:
            flags = np.zeros(n, bool)
            flags[idx] = True
            bm = torch.from_numpy(oracle.pack_bits(flags).view(np.int32)).to(DEV)
            x.allgather_apply(d_val, bm, 0.1, G, w)
        assert efg.workspace_status(x.ws_all) == 0
        assert_bits_equal(G, G_want, f"G ({fmt})")
        assert_bits_equal(w, w_want, f"w ({fmt})")
    x = ex.Exchange(n, k, ex.IDX_INT32)
    w = torch.from_numpy(w0.copy()).to(DEV)
    Gs = torch.empty(x.s, device=DEV)
    x.range_apply(d_val, d_idx, 0.1, w, Gs)
    assert efg.workspace_status(x.ws_range) == 0
    assert_bits_equal(Gs[:n], G_want, "G range")
    assert_bits_equal(w[:n], w_want, "w range")
    assert_bits_equal(w[n:], w0[n:], "w padding")


def test_range_exchange_four_ranks_simulated():
    """The index-range scheme's device steps for four ranks on one GPU: each
    rank's packet is split at the range bounds, the slices of every range
    are concatenated in source-rank order (what the all-to-all delivers),
    rebased and aggregated on the range; the ranges put together must equal
    the receive side over all packets."""
    W, n, k = 4, 3_000_017, 3000
    s = ex.shard_length(n, W)
    bounds = [min(q * s, n) for q in range(W)] + [n]
    pk = [(_sorted_packet(n, k, 40 + r),
           (np.random.default_rng(50 + r).standard_normal(k) * 1e-3).astype(F32))
          for r in range(W)]
    w0 = (np.random.default_rng(60).standard_normal(W * s) * 0.02).astype(F32)
    d = [(torch.from_numpy(i).to(DEV), torch.from_numpy(v).to(DEV)) for i, v in pk]
    starts = [host(efg.binding.packet_split(i, k, bounds)).tolist() for i, _ in d]
    w = torch.from_numpy(w0.copy()).to(DEV)
    G = torch.empty(W * s, device=DEV)
    for q in range(W):
        sl = [(i[starts[r][q]:starts[r][q + 1]], v[starts[r][q]:starts[r][q + 1]])
              for r, (i, v) in enumerate(d)]
        ri = torch.cat([a for a, _ in sl]).contiguous()
        rv = torch.cat([b for _, b in sl]).contiguous()
        cnt = [a.numel() for a, _ in sl]
        efg.binding.index_rebase(ri, ri.numel(), q * s)
        offs = np.concatenate([[0], np.cumsum(cnt)]).tolist()
        n_q = min(n, (q + 1) * s) - q * s
        wsq = torch.empty(efg.aggregate_workspace_size(W, efg.IDX_INT32, n_q), dtype=torch.uint8,
                          device=DEV)
        efg.sparse_aggregate_apply([rv[offs[r]:offs[r + 1]] for r in range(W)],
                                   [ri[offs[r]:offs[r + 1]] for r in range(W)], None, cnt, n_q,
                                   0.1, G[q * s:q * s + n_q], w[q * s:q * s + n_q], wsq)
        assert efg.workspace_status(wsq) == 0
    G_want = oracle.sparse_aggregate([{"indices": i, "values": v} for i, v in pk], n)
    w_want = oracle.sgd_apply(w0[:n], G_want, 0.1)
    assert_bits_equal(G[:n], G_want, "G")
    assert_bits_equal(w[:n], w_want, "w")
