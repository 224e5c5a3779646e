"""Oracle work for the full-size GPU parity tests, spread over host cores.

The oracle is elementwise for the 1-bit path and the sign receive side, and
independent per worker for the top-k steps, so its results are the same
whether computed whole or in pieces; this module runs the pieces in a pool
of processes started with ``spawn`` (never forked from a process holding a
CUDA context).  It imports only numpy and the oracle.
"""

from __future__ import annotations

import contextlib
import multiprocessing as mp
import os

import numpy as np

import oracle

CHUNK = 1 << 27   # elements per piece of elementwise work (a multiple of 32)


@contextlib.contextmanager
def pool(processes: int = 0):
    n = processes or max(1, min(16, os.cpu_count() or 1))
    p = mp.get_context("spawn").Pool(n)
    try:
        yield p
    finally:
        p.terminate()
        p.join()


def _sign_piece(args):
    g, eps, beta1 = args
    return oracle.sign_ef_step(g, eps, beta1)


def sign_ef_step(p, g: np.ndarray, eps: np.ndarray, beta1: float):
    """oracle.sign_ef_step over the whole arrays, in pieces of CHUNK elements."""
    n = g.size
    parts = p.map(_sign_piece, [(g[a:a + CHUNK], eps[a:a + CHUNK], beta1)
                                for a in range(0, n, CHUNK)], chunksize=1)
    return np.concatenate([b for b, _ in parts]), np.concatenate([e for _, e in parts])


def _sign_apply_piece(args):
    words, m, w, eta = args
    G = oracle.sign_aggregate(words, m)
    return G, oracle.sgd_apply(w, G, eta)


def sign_aggregate_sgd(p, bit_vectors, n: int, w: np.ndarray, eta: float):
    """G = oracle.sign_aggregate(bit_vectors, n) and oracle.sgd_apply(w, G),
    in pieces of CHUNK elements (bit word a // 32 starts piece a)."""
    tasks = []
    for a in range(0, n, CHUNK):
        m = min(CHUNK, n - a)
        words = [np.asarray(b)[a // 32:(a + m + 31) // 32] for b in bit_vectors]
        tasks.append((words, m, w[a:a + m], eta))
    parts = p.map(_sign_apply_piece, tasks, chunksize=1)
    return np.concatenate([G for G, _ in parts]), np.concatenate([x for _, x in parts])


def _topk_worker(args):
    g, e, offs, ks, fmt = args
    out = oracle.topk_ef_step(g, e, offs, ks, fmt)
    return {key: out[key] for key in ("indices", "values", "e", "bitmap") if key in out}


def topk_ef_steps(p, gs, es, offs, ks, fmt: str = "int32"):
    """oracle.topk_ef_step for several workers at once (one process each)."""
    return p.map(_topk_worker, [(g, e, offs, ks, fmt) for g, e in zip(gs, es)], chunksize=1)
