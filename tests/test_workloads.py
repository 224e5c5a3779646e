"""Host-side checks of the workload recipe (shapes, k rule, seeds)."""

import torch

from error_feedback_gradient_gb300 import workloads as wl


def test_resnet50_shapes():
    shapes = wl.resnet50_param_shapes()
    assert len(shapes) == 161
    assert sum(wl.numel(s) for _, s in shapes) == 25_557_032
    sizes = [wl.numel(s) for _, s in shapes]
    assert max(sizes) == 2_359_296 and min(sizes) == 64
    assert sum(1 for s in sizes if s >= 1_000_000) == 10


def test_resnet50_k_rule():
    offs, ks = wl.resnet50_segments()
    assert offs[0] == 0 and offs[-1] == 25_557_032
    assert sum(ks) == 107_379
    assert min(ks) >= 1


def test_bert_large_size():
    assert sum(wl.numel(s) for _, s in wl.bert_large_param_shapes()) == 335_141_888


def test_k_from_ratio():
    assert wl.k_from_ratio(1 << 20, 1, 100) == 10_486
    assert wl.k_from_ratio(335_141_888, 1, 1000) == 335_142
    assert wl.k_from_ratio(1 << 31, 1, 1000) == 2_147_484
    assert wl.k_from_ratio(64, 1, 100) == 1          # minimum 1
    assert wl.k_from_ratio(0, 1, 100) == 0
    assert wl.k_from_ratio(150, 1, 100) == 2         # 1.5 rounds half up


def test_workload_table():
    w = wl.workload("topk_2p20")
    assert (w.n, w.total_k, w.steps, w.workers) == (1 << 20, 10_486, 3, 1)
    w = wl.workload("bert_large")
    assert (w.n, w.total_k, w.workers) == (335_141_888, 335_142, 8)
    w = wl.workload("slab_2p31")
    assert (w.n, w.total_k, w.workers) == (1 << 31, 2_147_484, 4)
    assert wl.workload("sign_2p24").steps == 10


def test_generators_are_seeded_and_shaped():
    a = wl.student_t3(10_000, 1e-3, 5)
    b = wl.student_t3(10_000, 1e-3, 5)
    assert torch.equal(a, b) and a.dtype == torch.float32
    c = wl.student_t3(10_000, 1e-3, 6)
    assert not torch.equal(a, c)
    # heavy tails: Student-t(3) has kurtosis well above a normal's
    x = wl.student_t3(200_000, 1.0, 1).double()
    assert (x.abs() > 5).float().mean() > 0.005
    lap = wl.laplace(200_000, 1e-4, 2).double()
    assert abs(lap.abs().mean().item() - 1e-4) < 5e-6   # E|X| = b
    nrm = wl.normal(200_000, 1e-3, 3).double()
    assert abs(nrm.std().item() - 1e-3) < 2e-5


def test_resnet_gradient_scales_fixed_across_steps():
    w = wl.workload("resnet50")
    g1 = w.gradient(0, 1)
    g2 = w.gradient(0, 2)
    assert g1.numel() == w.n and not torch.equal(g1, g2)
    a, b = w.seg_offsets[0], w.seg_offsets[1]
    r = (g1[a:b].std() / g2[a:b].std()).item()
    assert 0.9 < r < 1.1
