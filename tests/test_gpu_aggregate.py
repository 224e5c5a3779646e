"""GPU parity of sparse_aggregate_apply against the oracle."""

import json
import os

import numpy as np
import pytest
import torch

import error_feedback_gradient_gb300 as efg
from efcheck import assert_bits_equal, assert_close, host
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _packets(n, W, density, seed, overlap=True):
    rng = np.random.default_rng(seed)
    shared = np.sort(rng.choice(n, max(1, int(n * density / 2)), replace=False))
    pk = []
    for w in range(W):
        k = int(n * density)
        own = rng.choice(n, k, replace=False)
        idx = np.unique(np.concatenate([own, shared]) if overlap else own)
        vals = (rng.standard_t(3, idx.size) * 1e-3).astype(np.float32)
        pk.append({"indices": idx.astype(np.int32), "values": vals})
    return pk


def _run(pk, n, eta, fmt, with_G=True, w0=None):
    W = len(pk)
    vals = [torch.from_numpy(p["values"]).to(DEV) for p in pk]
    ks = [p["values"].size for p in pk]
    if fmt == efg.IDX_INT32:
        inds = [torch.from_numpy(p["indices"]).to(DEV) for p in pk]
        bms = None
    else:
        inds = None
        bms = []
        for p in pk:
            flags = np.zeros(n, bool)
            flags[p["indices"]] = True
            bms.append(torch.from_numpy(oracle.pack_bits(flags).view(np.int32)).to(DEV))
    if w0 is None:
        w0 = (np.random.default_rng(1).standard_normal(n) * 0.02).astype(np.float32)
    w = torch.from_numpy(w0.copy()).to(DEV)
    G = torch.empty(n, device=DEV) if with_G else None
    ws = torch.empty(efg.aggregate_workspace_size(W, fmt, n), dtype=torch.uint8, device=DEV)
    efg.sparse_aggregate_apply(vals, inds, bms, ks, n, eta, G, w, ws, fmt)
    torch.cuda.synchronize()
    return G, w, w0, ws


@pytest.mark.parametrize("fmt", [efg.IDX_INT32, efg.IDX_BITMAP])
@pytest.mark.parametrize("W", [1, 2, 3, 8])
@pytest.mark.parametrize("n", [1, 100, 8192, 8193, 1_000_003])
def test_aggregate_random(fmt, W, n):
    pk = _packets(n, W, 0.01 if n > 100 else 0.3, seed=n + W)
    G, w, w0, ws = _run(pk, n, 0.1, fmt)
    G_want = oracle.sparse_aggregate(pk, n)
    w_want = oracle.sgd_apply(w0, G_want, 0.1)
    assert efg.workspace_status(ws) == 0
    assert_close(G, G_want, "G")
    assert_bits_equal(G, G_want, "G (bitwise)")
    assert_close(w, w_want, "w")
    assert_bits_equal(w, w_want, "w (bitwise)")
    _, w2, _, _ = _run(pk, n, 0.1, fmt, with_G=False)
    assert_bits_equal(w2, w_want, "w with G = NULL")


@pytest.mark.parametrize("fmt", [efg.IDX_INT32, efg.IDX_BITMAP])
def test_aggregate_sparse_and_dense_tiles_mixed(fmt):
    """Warp tiles of several 1024-element sub-tiles (n > 2^25): most hold a
    few entries and are summed from a shared list; a region where worker 2
    sends every index is summed sub-tile by sub-tile; the ragged tail ends
    mid-tile."""
    n = (1 << 25) + 12_345
    pk = _packets(n, 4, 0.001, seed=77)
    rng = np.random.default_rng(78)
    idx = np.unique(np.concatenate([pk[2]["indices"], np.arange(5_000_000, 5_100_000)]))
    pk[2] = {"indices": idx.astype(np.int32),
             "values": (rng.standard_t(3, idx.size) * 1e-3).astype(np.float32)}
    G, w, w0, ws = _run(pk, n, 0.05, fmt)
    G_want = oracle.sparse_aggregate(pk, n)
    assert efg.workspace_status(ws) == 0
    assert_bits_equal(G, G_want, "G")
    assert_bits_equal(w, oracle.sgd_apply(w0, G_want, 0.05), "w")


@pytest.mark.parametrize("fmt", [efg.IDX_INT32, efg.IDX_BITMAP])
@pytest.mark.parametrize("density", [0.0005, 0.01])
def test_aggregate_sixty_four_workers(fmt, density):
    """The largest worker count, with overlapping packets: sparse tiles go
    through the list (owner lane + binary search in 63 other runs), denser
    ones through the shared dense copy."""
    n = 300_001
    pk = _packets(n, 64, density, seed=int(density * 1e5))
    G, w, w0, ws = _run(pk, n, 0.1, fmt)
    G_want = oracle.sparse_aggregate(pk, n)
    assert efg.workspace_status(ws) == 0
    assert_bits_equal(G, G_want, "G")
    assert_bits_equal(w, oracle.sgd_apply(w0, G_want, 0.1), "w")


def test_aggregate_golden_examples():
    fx = json.load(open(os.path.join(GOLDEN, "aggregate_examples.json")))
    for ex in fx["examples"]:
        pk = [{"indices": np.array(p["indices"], np.int32),
               "values": np.array([float(v) for v in p["values"]], np.float32)}
              for p in ex["packets"]]
        w0 = np.array([float(v) for v in ex["w0"]], np.float32)
        for fmt in (efg.IDX_INT32, efg.IDX_BITMAP):
            G, w, _, _ = _run(pk, ex["n"], ex["eta"], fmt, w0=w0)
            assert host(G).tolist() == [float(x) for x in ex["G"]]
            if "G_signbit" in ex:
                assert np.signbit(host(G)).tolist() == ex["G_signbit"]
            w_want = oracle.sgd_apply(w0, oracle.sparse_aggregate(pk, ex["n"]), ex["eta"])
            assert_bits_equal(w, w_want, ex["name"])


def test_aggregate_full_packets_and_empty_workers():
    n = 20_000
    pk = [{"indices": np.arange(n, dtype=np.int32), "values": np.ones(n, np.float32)},
          {"indices": np.zeros(0, np.int32), "values": np.zeros(0, np.float32)},
          {"indices": np.array([0, n - 1], np.int32), "values": np.array([2, 3], np.float32)}]
    for fmt in (efg.IDX_INT32, efg.IDX_BITMAP):
        G, w, w0, _ = _run(pk, n, 0.5, fmt)
        G_want = oracle.sparse_aggregate(pk, n)
        assert_bits_equal(G, G_want, "G")
        assert_bits_equal(w, oracle.sgd_apply(w0, G_want, 0.5), "w")


def test_malformed_packets_are_reported():
    n = 50_000
    bad = [{"indices": np.array([10, 5, 20000], np.int32), "values": np.ones(3, np.float32)}]
    _, _, _, ws = _run(bad, n, 0.1, efg.IDX_INT32)
    assert efg.workspace_status(ws) == 13          # EF_ERR_PACKET
    oob = [{"indices": np.array([1, 2, n + 5], np.int32), "values": np.ones(3, np.float32)}]
    _, _, _, ws = _run(oob, n, 0.1, efg.IDX_INT32)
    assert efg.workspace_status(ws) == 13
    # bitmap whose population count disagrees with k
    flags = np.zeros(n, bool)
    flags[[3, 4, 5]] = True
    bm = torch.from_numpy(oracle.pack_bits(flags).view(np.int32)).to(DEV)
    w = torch.zeros(n, device=DEV)
    ws = torch.empty(efg.aggregate_workspace_size(1, efg.IDX_BITMAP, n), dtype=torch.uint8,
                     device=DEV)
    efg.sparse_aggregate_apply([torch.ones(2, device=DEV)], None, [bm], [2], n, 0.1, None, w,
                               ws, efg.IDX_BITMAP)
    assert efg.workspace_status(ws) == 13
