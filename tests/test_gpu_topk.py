"""GPU parity of ef_topk_compress against the oracle (bit-exact)."""

import numpy as np
import pytest
import torch

import error_feedback_gradient_gb300 as efg
from error_feedback_gradient_gb300 import workloads as wl
from efcheck import check_topk_step, gpu_topk, host, assert_bits_equal

pytestmark = pytest.mark.gpu
DEV = "cuda"
FMTS = [efg.IDX_INT32, efg.IDX_BITMAP]


def _t(n, seed, scale=1e-3):
    return wl.student_t3(n, scale, seed, DEV)


@pytest.mark.parametrize("fmt", FMTS)
def test_small_segments(fmt):
    sizes = [1, 2, 3, 31, 32, 33, 100, 1000, 4096, 20000, 32767, 32768]
    ks = [1, 0, 3, 5, 32, 1, 10, 17, 41, 200, 327, 1]
    offs = wl.segments_from_sizes(sizes)
    n = offs[-1]
    check_topk_step(_t(n, 1), _t(n, 2, 1e-4), offs, ks, fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_small_segments_both_select_paths(fmt):
    """Tensors of at most 4096 elements, finished by one CTA each: with a
    small k the few keys at or above the k-th key's first-digit bin are
    ranked directly; with a large k, an all-equal tensor or mostly zeros
    (more than 256 such keys) the three-pass radix select runs."""
    rng = np.random.default_rng(44)
    parts, ks = [], []
    parts.append(rng.standard_t(3, 4096) * 1e-3); ks.append(41)        # direct
    parts.append(rng.standard_t(3, 4096) * 1e-3); ks.append(2000)      # radix
    parts.append(np.full(3000, 0.25)); ks.append(7)                    # all equal: radix
    z = np.zeros(4000); z[rng.choice(4000, 20, replace=False)] = 1e-3
    parts.append(z); ks.append(50)                                     # zeros at the cut: radix
    parts.append(rng.standard_t(3, 300) * 1e-3); ks.append(300)        # k = len, 300 keys: radix
    parts.append(rng.standard_t(3, 200) * 1e-3); ks.append(200)        # k = len, 200 keys: direct
    # residuals: zero on the all-equal and mostly-zero tensors, so that g
    # keeps their ties and zeros
    es = [rng.standard_t(3, p.size) * 1e-4 if i not in (2, 3) else np.zeros(p.size)
          for i, p in enumerate(parts)]
    g = torch.from_numpy(np.concatenate(parts).astype(np.float32)).to(DEV)
    e = torch.from_numpy(np.concatenate(es).astype(np.float32)).to(DEV)
    offs = wl.segments_from_sizes([p.size for p in parts])
    check_topk_step(g, e, offs, ks, fmt)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n,k", [(32769, 328), (100_003, 1000), (1 << 20, 10486),
                                 (3_000_017, 3000), (200_000, 1), (40_000, 40_000),
                                 (50_000, 0)])
def test_single_streaming_segment(n, k, fmt):
    check_topk_step(_t(n, 10 + n % 97), _t(n, 20 + n % 89, 1e-4), [0, n], [k], fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_mixed_segments_and_empty(fmt):
    sizes = [0, 64, 40000, 0, 1, 250_000, 7, 65_537, 32768, 32769]
    ks = [0, 1, 400, 0, 1, 250, 7, 0, 16, 33]
    offs = wl.segments_from_sizes(sizes)
    n = offs[-1]
    check_topk_step(_t(n, 3), _t(n, 4, 1e-4), offs, ks, fmt)


def test_ties_everywhere():
    # one value everywhere: every candidate list overflows, the whole-segment
    # select runs, and the lowest indices win
    n = 300_000
    g = torch.full((n,), 0.5, device=DEV)
    check_topk_step(g, torch.zeros(n, device=DEV), [0, 100_000, n], [777, 5000])
    # a few levels with +-0 and sign flips, many equal keys at the threshold
    rng = np.random.default_rng(5)
    lv = np.array([0.0, -0.0, 1e-3, -1e-3, 2e-3, -2e-3, 4e-3], np.float32)
    g = torch.from_numpy(lv[rng.integers(0, lv.size, n)]).to(DEV)
    check_topk_step(g, torch.zeros(n, device=DEV), [0, n], [60_000])
    check_topk_step(g, torch.zeros(n, device=DEV), [0, 20_000, n], [3000, 200_000])


def test_special_values():
    n = 150_001
    g = _t(n, 7)
    g[::1000] = float("inf")
    g[5::1003] = float("-inf")
    g[7::2000] = float("nan")
    g[9::97] = 1e-40          # denormal
    g[11::89] = -0.0
    # NaNs with different payloads and signs: all tie above +Inf
    raw = g.view(torch.int32)
    raw[13::3001] = 0x7FC00001
    raw[17::3007] = -4194304          # 0xFFC00000
    e = torch.zeros(n, device=DEV)
    check_topk_step(g, e, [0, 1000, n], [3, 500])


def test_unaligned_addresses():
    n = 120_001
    base_g = _t(n + 8, 8)
    base_e = _t(n + 8, 9, 1e-4)
    # same misalignment (16-byte path with a phase) ...
    check_topk_step(base_g[1:n + 1], base_e[1:n + 1], [0, 5, 50_007, n], [1, 400, 700])
    # ... and different misalignments (scalar path)
    check_topk_step(base_g[2:n + 2], base_e[3:n + 3], [0, 5, 50_007, n], [1, 400, 700])


@pytest.mark.parametrize("fmt", FMTS)
def test_unaligned_addresses_long_list(fmt):
    """The same two misalignments on a tensor of 5 M elements, whose list
    is selected by the passes over the list (a general batch), not by a
    thread-block cluster."""
    n = 5_000_011
    base_g = _t(n + 8, 18)
    base_e = _t(n + 8, 19, 1e-4)
    check_topk_step(base_g[1:n + 1], base_e[1:n + 1], [0, n], [5000], fmt)
    check_topk_step(base_g[2:n + 2], base_e[3:n + 3], [0, n], [5000], fmt)


def _sample_block_starts(n):
    """Starts of the sampled blocks of a streaming segment of n elements:
    min(4096, n // 1024) blocks of 64 contiguous elements, block b in the
    middle of the b-th of that many equal slots of n // nblk elements (the
    documented sampling rule of the library)."""
    nblk = min(4096, n // 1024)
    sp = n // nblk
    return np.arange(nblk, dtype=np.int64) * sp + (sp - 64) // 2


def test_sampled_threshold_too_high_falls_back():
    """Large values on exactly the sampled blocks push the sampled threshold
    above the true k-th key, so fewer than k candidates are found; the
    whole-segment select must take over (after putting g back at the
    candidates) and still give the oracle's answer."""
    n, k = 1 << 20, 10486
    g = torch.full((n,), 1e-4, device=DEV) * torch.linspace(1, 2, n, device=DEV)
    starts = _sample_block_starts(n)
    pos = (starts[:, None] + np.arange(64)[None, :]).ravel()
    big = 1.0 + np.arange(pos.size, dtype=np.float32) * 1e-6
    g[torch.from_numpy(pos).to(DEV)] = torch.from_numpy(big).to(DEV)
    check_topk_step(g, torch.zeros(n, device=DEV), [0, n], [k])


@pytest.mark.parametrize("fmt", FMTS)
def test_kth_key_far_above_sampled_threshold(fmt):
    """The k largest values (about 1.0) sit off the sampled blocks, among
    small lognormal ones (about 1e-4), so the sampled threshold comes from
    the small values: the candidate list (about 23 k entries) still fits,
    but the k-th key lies some 2^26 key units above the threshold.  The
    finish's two-pass select, whose first digit counts from the threshold,
    cannot place it and must hand over to the three-pass select."""
    n, k = 1 << 20, 10486
    rng = np.random.default_rng(5)
    g_np = (1e-4 * np.exp(rng.standard_normal(n))).astype(np.float32)
    starts = _sample_block_starts(n)
    sampled = np.zeros(n, bool)
    sampled[(starts[:, None] + np.arange(64)[None, :]).ravel()] = True
    big = rng.choice(np.flatnonzero(~sampled), k, replace=False)
    g_np[big] = (1.0 + rng.random(k)).astype(np.float32)
    check_topk_step(torch.from_numpy(g_np).to(DEV), torch.zeros(n, device=DEV), [0, n], [k], fmt)


def _values(kind, n, rng):
    """Seeded gradient-like values of several shapes: very wide and very
    narrow dynamic ranges, heavy ties, mostly zeros, both signed zeros."""
    if kind == "lognormal_wide":
        return (1e-3 * np.exp(6.0 * rng.standard_normal(n)) * rng.choice([-1, 1], n)).astype(np.float32)
    if kind == "cauchy":
        return (1e-4 * rng.standard_cauchy(n)).astype(np.float32)
    if kind == "uniform_narrow":
        return (1.0 + 1e-3 * rng.random(n)).astype(np.float32)
    if kind == "few_values":
        return (rng.integers(-4, 5, n) * 0.25).astype(np.float32)
    if kind == "mostly_zero":
        g = np.zeros(n, np.float32)
        nz = rng.choice(n, n // 50, replace=False)
        g[nz] = (rng.standard_normal(nz.size) * 1e-3).astype(np.float32)
        return g
    if kind == "signed_zeros":
        g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        g[rng.random(n) < 0.5] = -0.0
        return g
    raise ValueError(kind)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("kind", ["lognormal_wide", "cauchy", "uniform_narrow", "few_values",
                                  "mostly_zero", "signed_zeros"])
@pytest.mark.parametrize("n,k", [(1_500_007, 10_000), (3_000_001, 3_000)])
def test_compact_select_over_value_shapes(kind, n, k, fmt):
    """One tensor in a compact batch (its list finished by a thread-block
    cluster, the select counted from the sampled threshold) over values of
    very different shapes: the k-th key far from or close to the
    threshold, ties at the cut, zeros that must never be listed."""
    rng = np.random.default_rng(sum(map(ord, kind)) * 7919 + n)
    g = torch.from_numpy(_values(kind, n, rng)).to(DEV)
    e = torch.from_numpy((_values(kind, n, rng) * np.float32(0.5)).astype(np.float32)).to(DEV)
    check_topk_step(g, e, [0, n], [k], fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_candidate_list_over_capacity_falls_back(fmt):
    """5 % of the elements tie at the largest value: every one is a
    candidate (about 200 per 4096-element warp span, within the staging
    buffers) but together they exceed the list capacity 4k + 65536; the
    candidates past the capacity keep g, the fused pass's zeros are undone,
    and the whole-segment select picks the lowest-index ties."""
    n, k = 2_000_000, 1000
    rng = np.random.default_rng(17)
    g_np = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    g_np[rng.choice(n, n // 20, replace=False)] = 0.5
    check_topk_step(torch.from_numpy(g_np).to(DEV), torch.zeros(n, device=DEV), [0, n], [k], fmt)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n,k", [(3_000_000, 3000), (5_000_000, 5000)])
def test_clustered_candidates_overflow_a_warps_staging(n, k, fmt):
    """The largest values sit in one contiguous run, as when a few rows of a
    gradient carry all the large entries: one warp's span holds far more
    candidates than its staging buffer.  A segment of 3 M elements is in a
    compact batch, one of 5 M in a general one."""
    rng = np.random.default_rng(n % 997)
    g_np = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    start = n // 3 + 7
    g_np[start:start + 2 * k] = (0.5 + rng.random(2 * k)).astype(np.float32)
    check_topk_step(torch.from_numpy(g_np).to(DEV), torch.zeros(n, device=DEV), [0, n], [k], fmt)


def test_multistep_carries_residual():
    n, k = 500_000, 500
    e = torch.zeros(n, device=DEV)
    for step in range(4):
        g = _t(n, 100 + step)
        want, _ = check_topk_step(g, e, [0, n], [k])
        e.copy_(torch.from_numpy(want["e"]))       # lockstep: continue from the oracle


def test_deterministic_repeat():
    n = 700_001
    g = _t(n, 31)
    e0 = _t(n, 32, 1e-4)
    outs = []
    for _ in range(2):
        e = e0.clone()
        o = gpu_topk(g, e, [0, n], [7000])
        outs.append((host(o["indices"]), host(o["values"]), host(e)))
    for a, b in zip(outs[0], outs[1]):
        assert_bits_equal(a, b, "repeat")


@pytest.mark.parametrize("fmt", FMTS)
def test_many_tensors_use_several_batches(fmt):
    """300 streaming tensors (more than one batch of 128) interleaved with
    1100 small ones (more than one launch of 512), in one layerwise call."""
    rng = np.random.default_rng(21)
    sizes, ks = [], []
    for i in range(1400):
        if i % 14 < 3:                       # 300 streaming tensors
            n_i = int(rng.integers(32769, 60000))
            ks.append(int(rng.integers(0, 400)))
        else:                                # 1100 small tensors
            n_i = int(rng.integers(1, 300))
            ks.append(int(rng.integers(0, n_i + 1)))
        sizes.append(n_i)
    offs = wl.segments_from_sizes(sizes)
    n = offs[-1]
    assert sum(1 for s in sizes if s > 32768) == 300
    check_topk_step(_t(n, 41), _t(n, 42, 1e-4), offs, ks, fmt)
