"""The regular entry points can be captured in a CUDA graph: their launch
plan travels in kernel parameters and workspaces, nothing synchronises the
host and nothing allocates.  One top-k + receive step of the 2^20 workload is
captured once and replayed on fresh inputs; every replay matches the oracle."""

import numpy as np
import pytest
import torch

import error_feedback_gradient_gb300 as efg
from error_feedback_gradient_gb300 import workloads as wl
from efcheck import assert_bits_equal, host
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_topk_step_replays_from_a_cuda_graph():
    w = wl.workload("topk_2p20")
    n, K = w.n, w.total_k
    g = torch.empty(n, device=DEV)
    e = torch.zeros(n, device=DEV)
    wt = w.weights(DEV)
    v = torch.empty(K, device=DEV)
    i = torch.empty(K, dtype=torch.int32, device=DEV)
    G = torch.empty(n, device=DEV)
    ws = torch.empty(efg.topk_workspace_size(n, w.seg_offsets, w.seg_k), dtype=torch.uint8,
                     device=DEV)
    wa = torch.empty(efg.aggregate_workspace_size(1, efg.IDX_INT32, n), dtype=torch.uint8,
                     device=DEV)

    def step():
        efg.topk_compress(g, e, w.seg_offsets, w.seg_k, v, i, None, ws)
        efg.sparse_aggregate_apply([v], [i], None, [K], n, w.eta, G, wt, wa)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        g.copy_(w.gradient(0, 9, DEV))
        step()                                  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for s in range(1, 4):
        g.copy_(w.gradient(0, s, DEV))
        e_before, w_before = host(e), host(wt)
        graph.replay()
        want = oracle.topk_ef_step(host(g), e_before, w.seg_offsets, w.seg_k)
        G_want = oracle.sparse_aggregate([want], n)
        torch.cuda.synchronize()
        assert_bits_equal(i, want["indices"], f"indices, replay {s}")
        assert_bits_equal(v, want["values"], f"values, replay {s}")
        assert_bits_equal(e, want["e"], f"residual, replay {s}")
        assert_bits_equal(G, G_want, f"G, replay {s}")
        assert_bits_equal(wt, oracle.sgd_apply(w_before, G_want, w.eta), f"w, replay {s}")
