"""GPU parity of the 8-bit packet path (ef_topk_compress_q8, ef_q8_dequantize)
against the oracle: codes, scales, indices or bitmap and the residual bit
for bit."""

import numpy as np
import pytest
import torch

import error_feedback_gradient_gb300 as efg
from error_feedback_gradient_gb300 import workloads as wl
from efcheck import assert_bits_equal, host
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"
FMTS = [efg.IDX_INT32, efg.IDX_BITMAP]


def _t(n, seed, scale=1e-3):
    return wl.student_t3(n, scale, seed, DEV)


def gpu_q8(g_raw, e, offs, ks, fmt=efg.IDX_INT32):
    n = g_raw.numel()
    K = int(sum(ks))
    q = torch.empty(K, dtype=torch.int8, device=DEV)
    sc = torch.empty(len(ks), dtype=torch.float32, device=DEV)
    idx = torch.empty(K, dtype=torch.int32, device=DEV) if fmt == efg.IDX_INT32 else None
    bm = torch.empty((n + 31) // 32, dtype=torch.int32, device=DEV) if fmt == efg.IDX_BITMAP else None
    ws = torch.empty(efg.topk_q8_workspace_size(n, offs, ks, fmt), dtype=torch.uint8, device=DEV)
    efg.topk_compress_q8(g_raw, e, offs, ks, q, sc, idx, bm, ws, fmt)
    return {"q": q, "scales": sc, "indices": idx, "bitmap": bm, "ws": ws}


def check_q8_step(g_raw, e, offs, ks, fmt=efg.IDX_INT32):
    g_np, e_np = host(g_raw), host(e)
    out = gpu_q8(g_raw, e, offs, ks, fmt)
    want = oracle.topk_q8_ef_step(g_np, e_np, offs, ks,
                                  "int32" if fmt == efg.IDX_INT32 else "bitmap")
    torch.cuda.synchronize()
    assert efg.workspace_status(out["ws"]) == 0
    if fmt == efg.IDX_INT32:
        assert_bits_equal(out["indices"], want["indices"], "indices")
    else:
        assert_bits_equal(out["bitmap"], want["bitmap"], "bitmap")
    assert np.array_equal(host(out["q"]), want["q"]), "codes"
    assert_bits_equal(out["scales"], want["scales"], "scales")
    assert_bits_equal(e, want["e"], "residual")
    return want, out


@pytest.mark.parametrize("fmt", FMTS)
def test_q8_small_and_streaming_segments(fmt):
    sizes = [1, 3, 100, 4096, 32768, 32769, 100_003, 0, 7, 250_000]
    ks = [1, 0, 10, 41, 327, 33, 1000, 0, 7, 2500]
    offs = wl.segments_from_sizes(sizes)
    n = offs[-1]
    check_q8_step(_t(n, 1), _t(n, 2, 1e-4), offs, ks, fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_q8_large_segment_several_chunks(fmt):
    n, k = 3_000_017, 30_000            # 8 chunks of 4096 entries, ragged
    check_q8_step(_t(n, 3), _t(n, 4, 1e-4), [0, n], [k], fmt)


def test_q8_special_values():
    n = 150_001
    g = _t(n, 7)
    g[::1000] = float("inf")
    g[5::1003] = float("-inf")
    g[7::2000] = float("nan")
    g[9::97] = 1e-40
    g[11::89] = -0.0
    check_q8_step(g, torch.zeros(n, device=DEV), [0, 1000, 40_000, n], [3, 500, 900])


def test_q8_zero_and_tied_segments():
    n = 200_000
    g = torch.zeros(n, device=DEV)
    g[100_000:] = 0.5                       # one tensor all zero, one all tied
    check_q8_step(g, torch.zeros(n, device=DEV), [0, 100_000, n], [50, 777])


def test_q8_multistep_carries_quantisation_error():
    n, k = 400_000, 400
    e = torch.zeros(n, device=DEV)
    for step in range(3):
        want, _ = check_q8_step(_t(n, 60 + step), e, [0, n], [k])
        e.copy_(torch.from_numpy(want["e"]))


def test_q8_many_segments_several_launches():
    rng = np.random.default_rng(5)
    sizes = [int(x) for x in rng.integers(1, 5000, 300)]
    ks = [int(rng.integers(0, s + 1)) // 10 for s in sizes]
    offs = wl.segments_from_sizes(sizes)
    n = offs[-1]
    check_q8_step(_t(n, 8), _t(n, 9, 1e-4), offs, ks)


def test_q8_dequantize_and_receive():
    """Receiver: codes times the segment scale, then the usual aggregate of
    two workers; equal to the oracle on the dequantised values."""
    n = 300_000
    offs, ks = [0, 50_000, n], [500, 2000]
    pk, want_pk = [], []
    for w in range(2):
        g = _t(n, 80 + w)
        want, out = check_q8_step(g, torch.zeros(n, device=DEV), offs, ks)
        vals = torch.empty(sum(ks), device=DEV)
        efg.q8_dequantize(out["q"], out["scales"], ks, vals)
        dq_want = np.concatenate([
            oracle.q8_dequantize(want["q"][a:a + k], want["scales"][i])
            for i, (a, k) in enumerate(zip([0, ks[0]], ks))])
        torch.cuda.synchronize()
        assert_bits_equal(vals, dq_want, "dequantised values")
        pk.append((vals, out["indices"]))
        want_pk.append({"indices": want["indices"], "values": dq_want})
    w0 = (np.random.default_rng(3).standard_normal(n) * 0.02).astype(np.float32)
    wt = torch.from_numpy(w0.copy()).to(DEV)
    G = torch.empty(n, device=DEV)
    efg.sparse_aggregate_apply([p[0] for p in pk], [p[1] for p in pk], None, [sum(ks)] * 2, n,
                               0.1, G, wt)
    G_want = oracle.sparse_aggregate(want_pk, n)
    torch.cuda.synchronize()
    assert_bits_equal(G, G_want, "G")
    assert_bits_equal(wt, oracle.sgd_apply(w0, G_want, 0.1), "w")


def test_q8_argument_errors():
    n = 1000
    g = _t(n, 1)
    e = torch.zeros(n, device=DEV)
    q = torch.empty(10, dtype=torch.int8, device=DEV)
    sc = torch.empty(1, device=DEV)
    idx = torch.empty(10, dtype=torch.int32, device=DEV)
    with pytest.raises(efg.EFError):           # scale output missing
        efg.topk_compress_q8(g, e, [0, n], [10], q, None, idx)
    with pytest.raises(efg.EFError):           # codes overlap the scale
        efg.topk_compress_q8(g, e, [0, n], [10], q, q, idx)
    with pytest.raises(efg.EFError):           # k above the segment length
        efg.topk_compress_q8(g, e, [0, n], [n + 1], q, sc, idx)
    with pytest.raises(efg.EFError):
        efg.q8_dequantize(q, sc, [-1], torch.empty(10, device=DEV))
