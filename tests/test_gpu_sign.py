"""GPU parity of ef_sign_compress and sign_aggregate_apply against the oracle."""

import numpy as np
import pytest
import torch

import error_feedback_gradient_gb300 as efg
from error_feedback_gradient_gb300 import workloads as wl
from efcheck import assert_bits_equal, assert_close, host
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _sign_step(g, eps, beta1=0.9):
    n = g.numel()
    g_np, eps_np = host(g), host(eps)
    bits = torch.empty((n + 31) // 32, dtype=torch.int32, device=DEV)
    efg.sign_compress(g, eps, beta1, bits)
    bits_want, eps_want = oracle.sign_ef_step(g_np, eps_np, beta1)
    torch.cuda.synchronize()
    assert_bits_equal(bits, bits_want, "sign bits")
    assert_close(eps, eps_want, "eps")
    assert_bits_equal(eps, eps_want, "eps (bitwise)")
    return bits, bits_want, eps_want


@pytest.mark.parametrize("n", [1, 5, 31, 32, 33, 127, 128, 129, 1000, (1 << 20) + 7])
def test_sign_sizes(n):
    _sign_step(wl.normal(n, 1e-3, n, DEV), wl.normal(n, 1e-3, n + 1, DEV))


def test_sign_long_spans_with_ragged_tail():
    """Above about 80 M elements each warp streams contiguous 4096-element
    spans; 2^27 + 37 elements end in a partial span, a partial 128-element
    group and a partial bit word."""
    n = (1 << 27) + 37
    _sign_step(wl.normal(n, 1e-3, 71, DEV), wl.normal(n, 1e-3, 72, DEV))


def test_sign_unaligned_and_special():
    n = 100_003
    gb = wl.normal(n + 4, 1e-3, 1, DEV)
    eb = wl.normal(n + 4, 1e-3, 2, DEV)
    gb[3::101] = 0.0
    gb[5::103] = -0.0
    gb[7::1001] = float("nan")
    gb[9::999] = float("-inf")
    gb[11::77] = 1e-40
    _sign_step(gb[1:n + 1], eb[1:n + 1])          # same phase: scalar words path
    _sign_step(gb[2:n + 2], eb[3:n + 3])          # mixed phases
    _sign_step(gb[:n], eb[:n], beta1=0.5)


def test_sign_zero_is_plus_one():
    g = torch.tensor([0.0, -0.0, 1.0, -1.0] * 40, device=DEV)
    bits, _, _ = _sign_step(g, torch.zeros_like(g))
    assert host(bits).view(np.uint32)[0] == 0b0111_0111_0111_0111_0111_0111_0111_0111


@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 6, 7, 8, 9, 64])
@pytest.mark.parametrize("mode", [efg.APPLY_SGD, efg.APPLY_MOMENTUM])
@pytest.mark.parametrize("n", [33, 4097, 1_000_003])
def test_sign_aggregate(W, mode, n):
    """Worker counts 1 to 9 and the maximum 64, sizes below one float4
    chunk's word and with ragged tails."""
    bits, wants = [], []
    for w in range(W):
        g = wl.normal(n, 1e-3, 50 + w, DEV)
        b = torch.empty((n + 31) // 32, dtype=torch.int32, device=DEV)
        efg.sign_compress(g, torch.zeros_like(g), 0.9, b)
        bits.append(b)
        wants.append(host(b).view(np.uint32))
    x0 = wl.normal(n, 0.02, 77, DEV)
    x = x0.clone()
    G = torch.empty(n, device=DEV)
    efg.sign_aggregate_apply(bits, n, mode, 0.1, 0.9, G, x)
    G_want = oracle.sign_aggregate(wants, n)
    if mode == efg.APPLY_SGD:
        x_want = oracle.sgd_apply(host(x0), G_want, 0.1)
    else:
        x_want = oracle.onebit_momentum(host(x0), G_want, 0.9)
    torch.cuda.synchronize()
    assert_bits_equal(G, G_want, "G")
    assert_close(x, x_want, "update")
    assert_bits_equal(x, x_want, "update (bitwise)")
    # without the dense output
    x2 = x0.clone()
    efg.sign_aggregate_apply(bits, n, mode, 0.1, 0.9, None, x2)
    assert_bits_equal(x2, x_want, "update, G = NULL")


def test_sign_aggregate_unaligned():
    n = 10_001
    b = torch.empty((n + 31) // 32, dtype=torch.int32, device=DEV)
    g = wl.normal(n, 1e-3, 5, DEV)
    efg.sign_compress(g, torch.zeros_like(g), 0.9, b)
    xb = wl.normal(n + 1, 0.02, 6, DEV)
    x0 = host(xb[1:])
    Gb = torch.empty(n + 1, device=DEV)
    efg.sign_aggregate_apply([b], n, efg.APPLY_SGD, 0.25, 0.9, Gb[1:], xb[1:])
    G_want = oracle.sign_aggregate([host(b).view(np.uint32)], n)
    torch.cuda.synchronize()
    assert_bits_equal(Gb[1:], G_want, "G")
    assert_bits_equal(xb[1:], oracle.sgd_apply(x0, G_want, 0.25), "w")
