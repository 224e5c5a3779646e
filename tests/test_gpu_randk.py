"""GPU parity of ef_randk_compress (random magnitude-proportional
sparsification) against the oracle: kept indices, values, residual and
per-segment counts bit for bit on the same seeded inputs and generator
key."""

import numpy as np
import pytest
import torch

import error_feedback_gradient_gb300 as efg
from error_feedback_gradient_gb300 import workloads as wl
from efcheck import assert_bits_equal, host
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _t(n, seed, scale=1e-3):
    return wl.student_t3(n, scale, seed, DEV)


def gpu_randk(g_raw, e, offs, ks, seed, step, capacity):
    vals = torch.empty(max(capacity, 1), device=DEV)
    idx = torch.empty(max(capacity, 1), dtype=torch.int32, device=DEV)
    counts = torch.empty(len(ks) + 1, dtype=torch.int64, device=DEV)
    ws = torch.empty(efg.randk_workspace_size(g_raw.numel(), offs, ks), dtype=torch.uint8,
                     device=DEV)
    efg.randk_compress(g_raw, e, offs, ks, seed, step, vals[:capacity] if capacity else vals[:0],
                       idx[:capacity] if capacity else idx[:0], counts, ws)
    return vals, idx, counts, ws


def check_randk(g_raw, e, offs, ks, seed, step, capacity=None):
    if capacity is None:
        capacity = int(sum(ks) * 2 + 1000)
    g_np, e_np = host(g_raw), host(e)
    vals, idx, counts, ws = gpu_randk(g_raw, e, offs, ks, seed, step, capacity)
    want = oracle.randk_ef_step(g_np, e_np, offs, ks, seed, step, capacity)
    torch.cuda.synchronize()
    c = host(counts)
    total = int(c[-1])
    status = efg.workspace_status(ws)
    assert status == (15 if want["kept"] > capacity else 0)
    assert total == want["indices"].size
    assert c[:-1].tolist() == want["counts"].tolist()
    assert_bits_equal(idx[:total], want["indices"], "indices")
    assert_bits_equal(vals[:total], want["values"], "values")
    assert_bits_equal(e, want["e"], "residual")
    return want


def test_randk_single_tensor_several_tiles():
    n = 100_003
    check_randk(_t(n, 1), _t(n, 2, 1e-4), [0, n], [1000], seed=12345, step=0)


def test_randk_segments_mixed_sizes_and_k():
    sizes = [1, 7, 100, 8191, 8192, 8193, 0, 50_000, 3, 200_000]
    ks = [1, 0, 10, 81, 82, 0, 0, 500, 3, 2000]
    offs = wl.segments_from_sizes(sizes)
    n = offs[-1]
    check_randk(_t(n, 3), _t(n, 4, 1e-4), offs, ks, seed=7, step=3)


def test_randk_many_segments_several_launches():
    rng = np.random.default_rng(9)
    sizes = [int(x) for x in rng.integers(1, 3000, 300)]
    ks = [max(0, s // 20) for s in sizes]
    offs = wl.segments_from_sizes(sizes)
    n = offs[-1]
    check_randk(_t(n, 5), torch.zeros(n, device=DEV), offs, ks, seed=2**63 + 5, step=2**40 + 1)


def test_randk_special_values_and_clipping():
    n = 60_000
    g = _t(n, 6)
    g[::997] = 50.0                  # c |g| > 1: kept surely
    g[3::5003] = float("inf")
    g[7::7001] = float("nan")
    g[1000:2000] = 0.0
    check_randk(g, torch.zeros(n, device=DEV), [0, 30_000, n], [300, 300], seed=1, step=1)


def test_randk_zero_segment_and_capacity_cut():
    n = 40_000
    g = _t(n, 8)
    g[:20_000] = 0.0                 # S = 0: keeps nothing
    check_randk(g, torch.zeros(n, device=DEV), [0, 20_000, n], [100, 400], seed=3, step=9)
    # capacity below the kept count: the packet stops, the rest stays in e
    check_randk(_t(n, 9), torch.zeros(n, device=DEV), [0, n], [2000], seed=4, step=4,
                capacity=500)
    check_randk(_t(n, 9), torch.zeros(n, device=DEV), [0, n], [2000], seed=4, step=4,
                capacity=0)


def test_randk_multistep_with_residual():
    n, k = 300_000, 3000
    e = torch.zeros(n, device=DEV)
    for step in range(3):
        want = check_randk(_t(n, 20 + step), e, [0, n], [k], seed=99, step=step)
        e.copy_(torch.from_numpy(want["e"]))


def test_randk_exact_sum_at_2p24():
    """A 2^24-element tensor with a wide spread of magnitudes: the exact
    sum, the coefficient and every draw agree with the oracle."""
    n = 1 << 24
    g = _t(n, 10) * torch.exp(torch.linspace(-20, 20, n, device=DEV))
    check_randk(g, torch.zeros(n, device=DEV), [0, n], [16_777], seed=2024, step=1)


def test_randk_count_statistics():
    """Over 40 steps the mean kept count is within a few standard errors
    of the expectation sum(p)."""
    n, k = 1_000_000, 1000
    g = _t(n, 11)
    cnts = []
    for step in range(40):
        e = torch.zeros(n, device=DEV)
        _, _, counts, _ = gpu_randk(g, e, [0, n], [k], 5, step, 10_000)
        cnts.append(int(host(counts)[-1]))
    gn = host(g)
    c = float(oracle.randk_coefficient(gn, k))
    p = np.minimum(1.0, c * np.abs(gn).astype(np.float64))
    mean, var = p.sum(), np.sum(p * (1 - p))
    assert abs(np.mean(cnts) - mean) < 5 * np.sqrt(var / 40)


def test_randk_block_edges_and_unaligned_residual():
    """Segments that start inside a quad of four elements and straddle the
    aligned 32768-element blocks, segments shorter than a quad, dense keep
    fractions, and a residual buffer that is only 4-byte aligned (the
    element-wise load path)."""
    sizes = [3, 5, 32_765, 32_768, 32_771, 1, 2, 65_549, 4, 100_000, 6]
    ks = [3, 2, 16_000, 300, 30_000, 1, 0, 650, 4, 99_000, 3]
    offs = wl.segments_from_sizes(sizes)
    n = offs[-1]
    for shift in (0, 1, 3):
        g_big = _t(n + 4, 30 + shift)
        e_big = _t(n + 4, 40 + shift, 1e-4)
        g, e = g_big[shift:shift + n], e_big[shift:shift + n]
        check_randk(g, e, offs, ks, seed=77 + shift, step=shift)


def test_randk_launch_without_draws_carries_the_packet_offset():
    """Segments go to the device in groups of 128; a group whose segments
    all have k = 0 draws nothing, and the packet positions of the groups
    after it still follow on from the groups before it."""
    rng = np.random.default_rng(12)
    sizes = [int(x) for x in rng.integers(1, 4000, 400)]
    ks = [0 if 128 <= i < 256 else max(1, s // 25) for i, s in enumerate(sizes)]
    offs = wl.segments_from_sizes(sizes)
    n = offs[-1]
    check_randk(_t(n, 13), _t(n, 14, 1e-4), offs, ks, seed=8, step=5)


def test_randk_sampled_bound_too_low_and_empty_sample():
    """Long tensors are sampled in blocks of 64 elements at the start of
    each of up to 2048 equal strides.  One large value inside the first
    sampled block makes the sample overstate the sum of |g| several times,
    so the bound taken from it falls below the true coefficient; a tensor
    whose nonzero elements all lie outside the sampled blocks gives an
    empty sample.  Both must still match the oracle."""
    n = 1 << 20
    g = _t(n, 31)
    g[5] = 1000.0
    check_randk(g, torch.zeros(n, device=DEV), [0, n], [1000], seed=21, step=2)
    stride = n // 1024                       # 1024 sampled blocks of 64
    pos = torch.arange(n, device=DEV)
    g2 = torch.where(pos % stride >= 64, _t(n, 32), torch.zeros(n, device=DEV))
    check_randk(g2, torch.zeros(n, device=DEV), [0, n], [1000], seed=22, step=3)
    # both in one call, beside a segment whose sample is representative
    g3 = torch.cat([g, g2, _t(n, 33)])
    check_randk(g3, torch.zeros(3 * n, device=DEV), [0, n, 2 * n, 3 * n], [1000, 500, 2000],
                seed=23, step=4)


def test_randk_sampled_segments_across_launch_groups():
    """More than 128 segments, with segments long enough to be sampled in
    both launch groups, dense and sparse keep fractions among them, and a
    capacity that cuts the packet inside the second group."""
    rng = np.random.default_rng(17)
    sizes = [int(x) for x in rng.integers(1, 2000, 140)]
    for i, s in ((3, 70_000), (60, 300_000), (131, 150_001), (139, 65_536)):
        sizes[i] = s
    ks = [max(0, s // 50) for s in sizes]
    ks[60] = 250_000                         # dense: c |g| > 1 for many elements
    ks[131] = 150
    offs = wl.segments_from_sizes(sizes)
    n = offs[-1]
    g, e = _t(n, 40), _t(n, 41, 1e-4)
    want = check_randk(g, e, offs, ks, seed=5, step=11)
    # the same inputs with a capacity below the kept count
    g2, e2 = _t(n, 40), _t(n, 41, 1e-4)
    check_randk(g2, e2, offs, ks, seed=5, step=11, capacity=int(want["kept"]) - 1000)
