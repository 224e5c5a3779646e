"""Helpers shared by the GPU parity tests: run one step through the C ABI and
compare it with the CPU oracle on the same inputs.

Exactness: indices, packed values, residuals and sign bitmaps must be
identical bit for bit; the EMA error buffer, the momentum, the aggregated
gradient and the updated weights must satisfy
max|gpu - oracle| <= 1e-6 * max|oracle| per array (with the explicit
round-to-nearest sequences both sides use they are in fact bit-identical,
which the tests also record).  NaN payload bits are not part of any result:
every NaN compares equal to every NaN.
"""

from __future__ import annotations

import numpy as np
import torch

import error_feedback_gradient_gb300 as efg
import oracle

F32 = np.float32
REL_TOL = 1e-6


def u32(x) -> np.ndarray:
    """Bit patterns of an array.  For float arrays every NaN maps to
    0x7FFFFFFF (the GPU's arithmetic returns one canonical NaN, numpy
    propagates the input's payload)."""
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().numpy()
    x = np.ascontiguousarray(x)
    bits = x.view(np.uint32).copy()
    if x.dtype == np.float32:
        bits[np.isnan(x)] = np.uint32(0x7FFFFFFF)
    return bits


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def assert_bits_equal(got, want, what: str) -> None:
    g, w = u32(got), u32(want)
    assert g.shape == w.shape, f"{what}: shape {g.shape} vs {w.shape}"
    if not np.array_equal(g, w):
        bad = np.flatnonzero(g != w)
        raise AssertionError(f"{what}: {bad.size} of {g.size} differ, first at {bad[:5].tolist()} "
                             f"got {g[bad[:5]].tolist()} want {w[bad[:5]].tolist()}")


def assert_close(got, want, what: str, rel: float = REL_TOL) -> None:
    g = np.asarray(host(got) if isinstance(got, torch.Tensor) else got, np.float64)
    w = np.asarray(want, np.float64)
    assert g.shape == w.shape, what
    # non-finite entries must agree exactly (NaN where NaN, same infinity)
    assert np.array_equal(np.isnan(g), np.isnan(w)), f"{what}: NaN positions differ"
    inf = np.isinf(w)
    assert np.array_equal(g[inf], w[inf]) and not np.isinf(g[~inf]).any(), f"{what}: inf differs"
    fin = np.isfinite(w)
    if not fin.any():
        return
    scale = np.max(np.abs(w[fin]))
    err = np.max(np.abs(g[fin] - w[fin]))
    assert err <= rel * scale, f"{what}: max|diff| {err} > {rel} * {scale}"


def gpu_topk(g_raw: torch.Tensor, e: torch.Tensor, offs, ks, fmt=efg.IDX_INT32):
    """Run ef_topk_compress (e updated in place); returns the packet tensors."""
    n = g_raw.numel()
    K = int(sum(ks))
    dev = g_raw.device
    vals = torch.empty(K, dtype=torch.float32, device=dev)
    idx = torch.empty(K, dtype=torch.int32, device=dev) if fmt == efg.IDX_INT32 else None
    bm = (torch.empty((n + 31) // 32, dtype=torch.int32, device=dev)
          if fmt == efg.IDX_BITMAP else None)
    nbytes = efg.topk_workspace_size(n, offs, ks, fmt)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    efg.topk_compress(g_raw, e, offs, ks, vals, idx, bm, ws, fmt)
    return {"values": vals, "indices": idx, "bitmap": bm, "ws": ws}


def check_topk_step(g_raw: torch.Tensor, e: torch.Tensor, offs, ks, fmt=efg.IDX_INT32):
    """One lockstep top-k step: the oracle and the GPU get the same g_raw and
    e; every output is compared bit for bit.  Returns the oracle's result."""
    g_np, e_np = host(g_raw), host(e)
    out = gpu_topk(g_raw, e, offs, ks, fmt)
    want = oracle.topk_ef_step(g_np, e_np, offs, ks,
                               "int32" if fmt == efg.IDX_INT32 else "bitmap")
    torch.cuda.synchronize()
    assert efg.workspace_status(out["ws"]) == 0
    if fmt == efg.IDX_INT32:
        assert_bits_equal(out["indices"], want["indices"], "indices")
    else:
        assert_bits_equal(out["bitmap"], want["bitmap"], "bitmap")
    assert_bits_equal(out["values"], want["values"], "values")
    assert_bits_equal(e, want["e"], "residual")
    return want, out
