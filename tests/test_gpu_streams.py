"""Calls in flight on several streams at once: the W workers' compress calls
run on a stream each, interleaved, with workspaces of their own, and the
receive side waits for them on the caller's stream.  The library keeps no
state between calls, so every output equals the oracle's, step after step."""

import numpy as np
import pytest
import torch

import error_feedback_gradient_gb300 as efg
from error_feedback_gradient_gb300 import workloads as wl
from efcheck import assert_bits_equal, host
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_workers_on_their_own_streams():
    n, W, eta, beta1 = 3_000_017, 4, 0.1, 0.9
    offs, ks = [0, 1_000_000, 2_500_000, n], [1000, 1500, 500]
    K, nw = sum(ks), (n + 31) // 32
    e_int = [wl.normal(n, 1e-4, 20 + w, DEV) for w in range(W)]
    e_bm = [wl.normal(n, 1e-4, 30 + w, DEV) for w in range(W)]
    eps = [wl.normal(n, 1e-4, 40 + w, DEV) for w in range(W)]
    w_int, w_bm, w_sign = (wl.normal(n, 0.02, s, DEV) for s in (50, 51, 52))
    G_int, G_bm, G_sign = (torch.empty(n, device=DEV) for _ in range(3))
    v_int = [torch.empty(K, device=DEV) for _ in range(W)]
    i_int = [torch.empty(K, dtype=torch.int32, device=DEV) for _ in range(W)]
    v_bm = [torch.empty(K, device=DEV) for _ in range(W)]
    bm = [torch.empty(nw, dtype=torch.int32, device=DEV) for _ in range(W)]
    bits = [torch.empty(nw, dtype=torch.int32, device=DEV) for _ in range(W)]
    u8 = torch.uint8
    ws_i = [torch.empty(efg.topk_workspace_size(n, offs, ks, efg.IDX_INT32), dtype=u8,
                        device=DEV) for _ in range(W)]
    ws_b = [torch.empty(efg.topk_workspace_size(n, offs, ks, efg.IDX_BITMAP), dtype=u8,
                        device=DEV) for _ in range(W)]
    wa_i = torch.empty(efg.aggregate_workspace_size(W, efg.IDX_INT32, n), dtype=u8, device=DEV)
    wa_b = torch.empty(efg.aggregate_workspace_size(W, efg.IDX_BITMAP, n), dtype=u8, device=DEV)
    streams = [torch.cuda.Stream() for _ in range(W)]
    main = torch.cuda.current_stream()
    fork = torch.cuda.Event()
    done = [[torch.cuda.Event() for _ in range(W)] for _ in range(3)]
    for step in range(2):
        g = [wl.student_t3(n, 1e-3, 100 * step + w, DEV) for w in range(W)]
        before = {name: [host(t) for t in ts] for name, ts in
                  (("e_int", e_int), ("e_bm", e_bm), ("eps", eps))}
        w0 = [host(t) for t in (w_int, w_bm, w_sign)]
        fork.record(main)
        for w, st in enumerate(streams):
            st.wait_event(fork)
            with torch.cuda.stream(st):
                efg.topk_compress(g[w], e_int[w], offs, ks, v_int[w], i_int[w], None, ws_i[w])
                done[0][w].record(st)
                efg.topk_compress(g[w], e_bm[w], offs, ks, v_bm[w], None, bm[w], ws_b[w],
                                  efg.IDX_BITMAP)
                done[1][w].record(st)
                efg.sign_compress(g[w], eps[w], beta1, bits[w])
                done[2][w].record(st)
        for ev in done[0]:
            main.wait_event(ev)
        efg.sparse_aggregate_apply(v_int, i_int, None, [K] * W, n, eta, G_int, w_int, wa_i)
        for ev in done[1]:
            main.wait_event(ev)
        efg.sparse_aggregate_apply(v_bm, None, bm, [K] * W, n, eta, G_bm, w_bm, wa_b,
                                   efg.IDX_BITMAP)
        for ev in done[2]:
            main.wait_event(ev)
        efg.sign_aggregate_apply(bits, n, efg.APPLY_SGD, eta, beta1, G_sign, w_sign)

        gh = [host(t) for t in g]
        pk_i = [oracle.topk_ef_step(gh[w], before["e_int"][w], offs, ks) for w in range(W)]
        pk_b = [oracle.topk_ef_step(gh[w], before["e_bm"][w], offs, ks, "bitmap")
                for w in range(W)]
        sg = [oracle.sign_ef_step(gh[w], before["eps"][w], beta1) for w in range(W)]
        torch.cuda.synchronize()
        for ws in ws_i + ws_b + [wa_i, wa_b]:
            assert efg.workspace_status(ws) == 0
        for w in range(W):
            tag = f"worker {w}, step {step}"
            assert_bits_equal(i_int[w], pk_i[w]["indices"], f"indices, {tag}")
            assert_bits_equal(v_int[w], pk_i[w]["values"], f"values, {tag}")
            assert_bits_equal(e_int[w], pk_i[w]["e"], f"residual, {tag}")
            assert_bits_equal(bm[w], pk_b[w]["bitmap"], f"bitmap, {tag}")
            assert_bits_equal(v_bm[w], pk_b[w]["values"], f"bitmap values, {tag}")
            assert_bits_equal(e_bm[w], pk_b[w]["e"], f"bitmap residual, {tag}")
            assert np.array_equal(host(bits[w]).view(np.uint32), sg[w][0]), f"bits, {tag}"
            assert_bits_equal(eps[w], sg[w][1], f"eps, {tag}")
        Gi = oracle.sparse_aggregate(pk_i, n)
        Gb = oracle.sparse_aggregate(pk_b, n)
        Gs = oracle.sign_aggregate([s[0] for s in sg], n)
        assert_bits_equal(G_int, Gi, f"G int32, step {step}")
        assert_bits_equal(G_bm, Gb, f"G bitmap, step {step}")
        assert_bits_equal(G_sign, Gs, f"G sign, step {step}")
        assert_bits_equal(w_int, oracle.sgd_apply(w0[0], Gi, eta), f"w int32, step {step}")
        assert_bits_equal(w_bm, oracle.sgd_apply(w0[1], Gb, eta), f"w bitmap, step {step}")
        assert_bits_equal(w_sign, oracle.sgd_apply(w0[2], Gs, eta), f"w sign, step {step}")
