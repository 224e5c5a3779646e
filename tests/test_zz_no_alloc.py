"""The allocation-free top-k entry point gives what the regular one gives.

ef_topk_compress_noalloc exists for callers that cannot call cudaMalloc at
compression time (for example a hook running while a framework's memory
pool owns all free device memory, or a latency-critical host section that
must not risk an allocation that synchronises the device).  It runs the same
computation with one library-owned scratch array instead of a caller-owned
workspace.  This file checks, through the C ABI, that two consecutive steps
(the second carrying the first one's residual, so the shared scratch is
reused with the previous call's contents still in it) match the regular
entry point bit for bit, and that requests larger than the array are
refused before any work.  It is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

import error_feedback_gradient_gb300 as efg
from error_feedback_gradient_gb300 import workloads as wl
from efcheck import assert_bits_equal

pytestmark = pytest.mark.gpu
DEV = "cuda"
EF_OK, EF_ERR_WORKSPACE = 0, 6


def _i64(xs):
    return (ctypes.c_int64 * len(xs))(*[int(x) for x in xs])


def _noalloc(g, e, offs, ks, vals, idx):
    lib = efg.library()
    return lib.ef_topk_compress_noalloc(
        g.data_ptr(), e.data_ptr(), g.numel(), len(ks), _i64(offs), _i64(ks), efg.IDX_INT32,
        vals.data_ptr(), idx.data_ptr(), None, torch.cuda.current_stream().cuda_stream)


def _regular(g, e, offs, ks, vals, idx):
    lib = efg.library()
    nbytes = efg.topk_workspace_size(g.numel(), offs, ks)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    return lib.ef_topk_compress(
        g.data_ptr(), e.data_ptr(), g.numel(), len(ks), _i64(offs), _i64(ks), efg.IDX_INT32,
        vals.data_ptr(), idx.data_ptr(), None, ws.data_ptr(), nbytes,
        torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_regular_on_two_calls_in_a_row():
    sizes = [20_000, 980_000, 2_000_017]          # one small tensor, two streaming ones
    offs = wl.segments_from_sizes(sizes)
    ks = [200, 980, 2000]
    n, K = offs[-1], sum(ks)
    e_reg = wl.student_t3(n, 1e-4, 71, DEV)
    e_na = e_reg.clone()
    assert efg.topk_workspace_size(n, offs, ks) <= 33554432
    for step in range(2):
        g = wl.student_t3(n, 1e-3, 72 + step, DEV)
        v_reg = torch.empty(K, device=DEV)
        i_reg = torch.empty(K, dtype=torch.int32, device=DEV)
        v_na = torch.full((K,), -1.0, device=DEV)
        i_na = torch.full((K,), -1, dtype=torch.int32, device=DEV)
        assert _regular(g, e_reg, offs, ks, v_reg, i_reg) == EF_OK
        assert _noalloc(g, e_na, offs, ks, v_na, i_na) == EF_OK
        torch.cuda.synchronize()
        assert_bits_equal(i_na, i_reg, f"indices, call {step + 1}")
        assert_bits_equal(v_na, v_reg, f"values, call {step + 1}")
        assert_bits_equal(e_na, e_reg, f"residual, call {step + 1}")


def test_noalloc_refuses_requests_beyond_its_scratch():
    n = 1 << 24
    ks = [n // 4]                                 # a candidate list far beyond 32 MiB
    assert efg.topk_workspace_size(n, [0, n], ks) > 33554432
    fake = ctypes.c_void_p(1 << 20)
    st = efg.library().ef_topk_compress_noalloc(fake, ctypes.c_void_p(2 << 30), n, 1,
                                                _i64([0, n]), _i64(ks), efg.IDX_INT32,
                                                ctypes.c_void_p(4 << 30), ctypes.c_void_p(5 << 30),
                                                None, None)
    assert st == EF_ERR_WORKSPACE
