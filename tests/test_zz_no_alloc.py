"""The allocation-free top-k entry point gives what the regular one gives.

ef_topk_compress_noalloc exists for callers that cannot call cudaMalloc at
compression time (for example a hook running while a framework's memory
pool owns all free device memory, or a latency-critical host section that
must not risk an allocation that synchronises the device).  It runs the same
computation with one library-owned scratch array instead of a caller-owned
workspace.  This file checks, through the C ABI, that two consecutive steps
(the second carrying the first one's residual, so the shared scratch is
reused with the previous call's contents still in it) match the regular
entry point bit for bit -- with int32 indices on a mix of small and
streaming tensors, with a bitmap on the same mix, and on small tensors
only -- that the device-side status of each call reads back as clean, and
that requests larger than the array are refused before any work.  It is
collected last on purpose.
"""

import ctypes

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


def _p(t):
    return None if t is None else t.data_ptr()


def _noalloc(g, e, offs, ks, vals, idx, bm, fmt):
    lib = efg.library()
    return lib.ef_topk_compress_noalloc(
        g.data_ptr(), e.data_ptr(), g.numel(), len(ks), _i64(offs), _i64(ks), fmt,
        vals.data_ptr(), _p(idx), _p(bm), torch.cuda.current_stream().cuda_stream)


def _regular(g, e, offs, ks, vals, idx, bm, fmt):
    lib = efg.library()
    nbytes = efg.topk_workspace_size(g.numel(), offs, ks, fmt)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    return lib.ef_topk_compress(
        g.data_ptr(), e.data_ptr(), g.numel(), len(ks), _i64(offs), _i64(ks), fmt,
        vals.data_ptr(), _p(idx), _p(bm), ws.data_ptr(), nbytes,
        torch.cuda.current_stream().cuda_stream)


def _two_calls(sizes, ks, fmt, seed):
    offs = wl.segments_from_sizes(sizes)
    n, K = offs[-1], sum(ks)
    e_reg = wl.student_t3(n, 1e-4, seed, DEV)
    e_na = e_reg.clone()
    assert efg.topk_workspace_size(n, offs, ks, fmt) <= 33554432
    bitmap = fmt == efg.IDX_BITMAP
    for step in range(2):
        g = wl.student_t3(n, 1e-3, seed + 1 + step, DEV)
        v_reg = torch.empty(K, device=DEV)
        v_na = torch.full((K,), -1.0, device=DEV)
        if bitmap:
            i_reg = i_na = None
            b_reg = torch.empty((n + 31) // 32, dtype=torch.int32, device=DEV)
            b_na = torch.full(((n + 31) // 32,), -1, dtype=torch.int32, device=DEV)
        else:
            b_reg = b_na = None
            i_reg = torch.empty(K, dtype=torch.int32, device=DEV)
            i_na = torch.full((K,), -1, dtype=torch.int32, device=DEV)
        assert _regular(g, e_reg, offs, ks, v_reg, i_reg, b_reg, fmt) == EF_OK
        assert _noalloc(g, e_na, offs, ks, v_na, i_na, b_na, fmt) == EF_OK
        assert efg.binding.topk_noalloc_status() == EF_OK
        torch.cuda.synchronize()
        if bitmap:
            assert_bits_equal(b_na, b_reg, f"bitmap, call {step + 1}")
        else:
            assert_bits_equal(i_na, i_reg, f"indices, call {step + 1}")
        assert_bits_equal(v_na, v_reg, f"values, call {step + 1}")
        assert_bits_equal(e_na, e_reg, f"residual, call {step + 1}")


def test_noalloc_matches_regular_on_two_calls_in_a_row():
    # one small tensor, two streaming ones
    _two_calls([20_000, 980_000, 2_000_017], [200, 980, 2000], efg.IDX_INT32, 71)


def test_noalloc_bitmap_matches_regular_on_two_calls_in_a_row():
    _two_calls([20_000, 980_000, 2_000_017], [200, 980, 2000], efg.IDX_BITMAP, 81)


def test_noalloc_small_segments_only():
    _two_calls([1, 64, 1000, 32_768, 7, 20_001], [1, 3, 10, 327, 0, 200], efg.IDX_INT32, 91)


def test_noalloc_refuses_requests_beyond_its_scratch():
    # real device buffers, so that a refusal that failed to happen would give
    # a wrong status or result rather than touch memory that is not there
    n = 1 << 24
    ks = [n // 4]                                 # a candidate list far beyond 32 MiB
    assert efg.topk_workspace_size(n, [0, n], ks) > 33554432
    g = torch.zeros(n, device=DEV)
    e = torch.zeros(n, device=DEV)
    vals = torch.full((ks[0],), 7.0, device=DEV)
    idx = torch.full((ks[0],), 7, dtype=torch.int32, device=DEV)
    st = _noalloc(g, e, [0, n], ks, vals, idx, None, efg.IDX_INT32)
    assert st == EF_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((vals == 7.0).all()) and bool((idx == 7).all())      # nothing was written
