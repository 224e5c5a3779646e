"""GPU parity at the five workloads' full sizes, in the launch configuration
bench.py times (same entry points, same segment tables, W workers as
separate buffers on one GPU).

Steps run in lockstep: each GPU step and the oracle step get the same inputs;
after a step both continue from the oracle's state, so a difference cannot
cascade.  Every output is compared in full, at every element, including the
2^31-element slab; the oracle's elementwise work at that size and the eight
BERT-large workers' steps run in a pool of host processes
(``oracle_pool``), in pieces whose results are the whole arrays'.
"""

import numpy as np
import pytest
import torch

import error_feedback_gradient_gb300 as efg
from error_feedback_gradient_gb300 import workloads as wl
from efcheck import assert_bits_equal, assert_close, check_topk_step, gpu_topk, host
import oracle
import oracle_pool

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _apply(packets_gpu, ks, n, eta, w_gpu, fmt=efg.IDX_INT32):
    G = torch.empty(n, device=DEV)
    vals = [p["values"] for p in packets_gpu]
    if fmt == efg.IDX_INT32:
        efg.sparse_aggregate_apply(vals, [p["indices"] for p in packets_gpu], None, ks, n, eta,
                                   G, w_gpu, idx_format=fmt)
    else:
        efg.sparse_aggregate_apply(vals, None, [p["bitmap"] for p in packets_gpu], ks, n, eta,
                                   G, w_gpu, idx_format=fmt)
    return G


def test_topk_2p20_three_steps_with_apply():
    w = wl.workload("topk_2p20")
    e = torch.zeros(w.n, device=DEV)
    wt = w.weights(DEV)
    for step in range(1, w.steps + 1):
        g = w.gradient(0, step, DEV)
        w_before = host(wt)
        want, out = check_topk_step(g, e, w.seg_offsets, w.seg_k)
        G = _apply([out], [w.total_k], w.n, w.eta, wt)
        G_want = oracle.sparse_aggregate([want], w.n)
        w_want = oracle.sgd_apply(w_before, G_want, w.eta)
        torch.cuda.synchronize()
        assert_close(G, G_want, "G")
        assert_close(wt, w_want, "w")
        assert_bits_equal(wt, w_want, "w (bitwise)")
        e.copy_(torch.from_numpy(want["e"]))
        wt.copy_(torch.from_numpy(w_want))


def test_sign_2p24_ten_steps_with_momentum():
    w = wl.workload("sign_2p24")
    eps = torch.zeros(w.n, device=DEV)
    m = torch.zeros(w.n, device=DEV)
    eps_ref = np.zeros(w.n, np.float32)
    m_ref = np.zeros(w.n, np.float32)
    bits = torch.empty((w.n + 31) // 32, dtype=torch.int32, device=DEV)
    for step in range(1, w.steps + 1):
        g = w.gradient(0, step, DEV)
        efg.sign_compress(g, eps, w.beta1, bits)
        efg.sign_aggregate_apply([bits], w.n, efg.APPLY_MOMENTUM, 0.0, w.beta1, None, m)
        bits_want, eps_ref = oracle.sign_ef_step(host(g), eps_ref, w.beta1)
        m_ref = oracle.onebit_momentum(m_ref, oracle.decode_signs(bits_want, w.n), w.beta1)
        torch.cuda.synchronize()
        assert_bits_equal(bits, bits_want, f"bits step {step}")
        assert_close(eps, eps_ref, f"eps step {step}")
        assert_close(m, m_ref, f"m step {step}")
        eps.copy_(torch.from_numpy(eps_ref))
        m.copy_(torch.from_numpy(m_ref))


@pytest.mark.parametrize("fmt", [efg.IDX_INT32, efg.IDX_BITMAP])
def test_resnet50_layerwise_three_steps(fmt):
    w = wl.workload("resnet50")
    e = torch.zeros(w.n, device=DEV)
    steps = w.steps if fmt == efg.IDX_INT32 else 1
    for step in range(1, steps + 1):
        g = w.gradient(0, step, DEV)
        want, _ = check_topk_step(g, e, w.seg_offsets, w.seg_k, fmt)
        e.copy_(torch.from_numpy(want["e"]))


def test_bert_large_eight_workers_three_steps():
    """The configuration as stated: eight workers, each with its own
    Laplace(0, 1e-4) gradient per step and its own residual from e0 = 0,
    three chained steps of top-0.1 % over the flat 335,141,888-element
    vector, each followed by the sum of the eight packets and SGD."""
    w = wl.workload("bert_large")
    W, n = w.workers, w.n
    wt = w.weights(DEV)
    es = [torch.zeros(n, device=DEV) for _ in range(W)]
    with oracle_pool.pool(W) as p:
        for step in range(1, w.steps + 1):
            gs = [w.gradient(k, step, DEV) for k in range(W)]
            g_np, e_np = [host(g) for g in gs], [host(e) for e in es]
            w_before = host(wt)
            outs = [gpu_topk(g, e, w.seg_offsets, w.seg_k) for g, e in zip(gs, es)]
            G = _apply(outs, [w.total_k] * W, n, w.eta, wt)
            wants = oracle_pool.topk_ef_steps(p, g_np, e_np, w.seg_offsets, w.seg_k)
            del g_np, e_np
            torch.cuda.synchronize()
            for k, (out, want) in enumerate(zip(outs, wants)):
                assert efg.workspace_status(out["ws"]) == 0
                assert_bits_equal(out["indices"], want["indices"], f"indices w{k} s{step}")
                assert_bits_equal(out["values"], want["values"], f"values w{k} s{step}")
                assert_bits_equal(es[k], want["e"], f"residual w{k} s{step}")
            G_want = oracle.sparse_aggregate(wants, n)
            w_want = oracle.sgd_apply(w_before, G_want, w.eta)
            assert_close(G, G_want, f"G s{step}")
            assert_bits_equal(G, G_want, f"G (bitwise) s{step}")
            assert_close(wt, w_want, f"w s{step}")
            assert_bits_equal(wt, w_want, f"w (bitwise) s{step}")
            for k in range(W):       # lockstep: continue from the oracle's state
                es[k].copy_(torch.from_numpy(wants[k]["e"]))
            wt.copy_(torch.from_numpy(w_want))
            del outs, wants, gs, G, G_want, w_want


def test_slab_2p31_topk_one_worker_in_full():
    w = wl.workload("slab_2p31")
    n, k = w.n, w.total_k
    g = w.gradient(0, 1, DEV)
    e0 = wl.student_t3(n, 1e-4, wl.seed(5, 0, 0), DEV)           # a carried residual
    g_np, e_np = host(g), host(e0)
    want = oracle.topk_ef_step(g_np, e_np, w.seg_offsets, w.seg_k, "int32")
    del e_np
    e = e0.clone()
    out = gpu_topk(g, e, w.seg_offsets, w.seg_k, efg.IDX_INT32)
    torch.cuda.synchronize()
    assert efg.workspace_status(out["ws"]) == 0
    assert_bits_equal(out["indices"], want["indices"], "indices")
    assert_bits_equal(out["values"], want["values"], "values")
    assert_bits_equal(e, want["e"], "residual")
    del out
    # the bitmap format of the same step
    e.copy_(e0)
    out = gpu_topk(g, e, w.seg_offsets, w.seg_k, efg.IDX_BITMAP)
    flags = np.zeros(n, bool)
    flags[want["indices"]] = True
    torch.cuda.synchronize()
    assert_bits_equal(out["bitmap"], oracle.pack_bits(flags), "bitmap")
    assert_bits_equal(out["values"], want["values"], "values (bitmap)")
    assert_bits_equal(e, want["e"], "residual (bitmap)")
    del out, flags
    # the same step with 8-bit values: the oracle's quantiser on the oracle's
    # selection (topk_q8_ef_step is exactly this composition)
    e.copy_(e0)
    q = torch.empty(k, dtype=torch.int8, device=DEV)
    sc = torch.empty(1, device=DEV)
    idx = torch.empty(k, dtype=torch.int32, device=DEV)
    ws = torch.empty(efg.topk_q8_workspace_size(n, w.seg_offsets, w.seg_k), dtype=torch.uint8,
                     device=DEV)
    efg.topk_compress_q8(g, e, w.seg_offsets, w.seg_k, q, sc, idx, None, ws)
    s_want = oracle.q8_scale(want["values"])
    q_want = oracle.q8_quantize(want["values"], s_want)
    e_want = want["e"]
    e_want[want["indices"]] = np.subtract(want["values"], oracle.q8_dequantize(q_want, s_want),
                                          dtype=np.float32)
    torch.cuda.synchronize()
    assert efg.workspace_status(ws) == 0
    assert_bits_equal(idx, want["indices"], "indices (q8)")
    assert np.array_equal(host(q), q_want), "codes (q8)"
    assert_bits_equal(sc, np.array([s_want], np.float32), "scale (q8)")
    assert_bits_equal(e, e_want, "residual (q8)")
    del e, e_want, ws, q
    # the packet's indices through the three index codecs, byte for byte
    for codec, enc in [(efg.CODEC_LOCAL16, oracle.encode_local16),
                       (efg.CODEC_BLOCK256, oracle.encode_block256),
                       (efg.CODEC_RUNVARINT, oracle.encode_runvarint)]:
        mb, wb = efg.index_codec_sizes(codec, k, n)
        buf = torch.empty((mb + 3) // 4, dtype=torch.int32, device=DEV)
        ob = torch.zeros(1, dtype=torch.int64, device=DEV)
        wsc = torch.empty(wb, dtype=torch.uint8, device=DEV)
        efg.index_encode(codec, idx, n, buf, ob, wsc)
        stream_want = enc(want["indices"].astype(np.int64), n)
        nbytes = int(ob.item())
        assert efg.workspace_status(wsc) == 0 and nbytes == stream_want.size
        assert np.array_equal(host(buf).view(np.uint8)[:nbytes], stream_want), codec
        back = torch.empty(k, dtype=torch.int32, device=DEV)
        efg.index_decode(codec, buf, nbytes, k, n, back, wsc)
        assert torch.equal(back, idx) and efg.workspace_status(wsc) == 0


def _exact_abs_sum(x: np.ndarray) -> float:
    """Exact sum of the finite |x| of a float32 array, rounded once to
    float64, by a route independent of the oracle's math.fsum: every |x| is
    an integer mantissa m < 2^24 times 2^(sh - 149); per chunk of 2^27
    elements the mantissas are summed per sh with numpy's bincount (float64
    weights, exact: every partial sum stays below 2^51), the chunk sums are
    combined as Python integers, and the exact rational is rounded by
    Python's correctly rounded int/int division."""
    from fractions import Fraction
    acc = [0] * 254
    for j in range(0, x.size, 1 << 27):
        b = x[j:j + (1 << 27)].view(np.uint32) & np.uint32(0x7FFFFFFF)
        b = b[b < np.uint32(0x7F800000)]
        E = (b >> np.uint32(23)).astype(np.int32)
        m = (b & np.uint32(0x7FFFFF)) | np.where(E > 0, np.uint32(1 << 23), np.uint32(0))
        sh = np.maximum(E, 1) - 1
        for i, v in enumerate(np.bincount(sh, weights=m.astype(np.float64), minlength=254)):
            acc[i] += int(v)
    total = sum(v << i for i, v in enumerate(acc))
    return float(Fraction(total, 1 << 149))


def test_slab_2p31_random_sparsification_sampled():
    """Random magnitude-proportional sparsification at 2^31 elements: the
    coefficient from an exact |g| sum computed independently on the host;
    every kept element passes its draw (Philox word from the oracle's
    generator), a sample of a million others fails it, values and residual
    agree at all of them, and the count matches."""
    w = wl.workload("slab_2p31")
    n, k = w.n, w.total_k
    g = w.gradient(0, 2, DEV)
    e = torch.zeros(n, device=DEV)
    g_np = host(g)
    cap = 2 * k
    vals = torch.empty(cap, device=DEV)
    idx = torch.empty(cap, dtype=torch.int32, device=DEV)
    counts = torch.empty(2, dtype=torch.int64, device=DEV)
    ws = torch.empty(efg.randk_workspace_size(n, [0, n], [k]), dtype=torch.uint8, device=DEV)
    seed, step = 0x5EED, 3
    efg.randk_compress(g, e, [0, n], [k], seed, step, vals, idx, counts, ws)
    S = _exact_abs_sum(g_np)
    c = np.float32(float(k) / S)
    torch.cuda.synchronize()
    assert efg.workspace_status(ws) == 0
    total = int(host(counts)[-1])
    kept = host(idx[:total]).astype(np.int64)
    assert np.all(np.diff(kept) > 0)
    rng = np.random.default_rng(1)
    others = np.setdiff1d(rng.integers(0, n, 1_000_000), kept)
    probe = np.concatenate([kept, others])
    # Philox words of the probed elements, one generator call per element
    words = np.empty(probe.size, np.uint32)
    for j in range(0, probe.size, 1 << 20):
        p_ = probe[j:j + (1 << 20)].astype(np.uint64)
        q_ = p_ >> np.uint64(2)
        out = oracle.philox4x32_10(q_ & np.uint64(0xFFFFFFFF), q_ >> np.uint64(32),
                                   np.uint64(step), np.uint64(0), np.uint64(seed), np.uint64(0))
        words[j:j + p_.size] = np.stack(out)[(p_ & np.uint64(3)).astype(np.int64),
                                             np.arange(p_.size)]
    a = np.abs(g_np[probe])
    p = np.ones(probe.size, np.float32)
    fin = np.isfinite(a)
    p[fin] = np.fmin(np.float32(1), np.multiply(c, a[fin], dtype=np.float32))
    u = (words >> np.uint32(8)).astype(np.float32) * np.float32(2.0 ** -24)
    keep = u < p
    assert keep[:kept.size].all(), "a sent element failed its draw"
    assert not keep[kept.size:].any(), "a sampled element passed its draw but was not sent"
    assert_bits_equal(vals[:total], g_np[kept], "values")
    e_probe = host(e[torch.from_numpy(probe).to(DEV)])
    want_e = g_np[probe].copy()
    want_e[:kept.size] = 0.0
    assert_bits_equal(e_probe, want_e, "residual (probed)")
    pv = np.minimum(1.0, float(c) * np.abs(g_np.astype(np.float64)))
    assert abs(total - pv.sum()) < 6 * np.sqrt(np.sum(pv * (1 - pv)))


def test_slab_2p31_sign_two_steps_in_full():
    """1-bit error feedback on one worker's 2^31-element slab from eps0 = 0,
    two chained steps; the bits and eps are compared at every element."""
    w = wl.workload("slab_2p31")
    n = w.n
    eps = torch.zeros(n, device=DEV)
    bits = torch.empty((n + 31) // 32, dtype=torch.int32, device=DEV)
    with oracle_pool.pool() as p:
        for step in (1, 2):
            g = w.gradient(1, step, DEV)
            g_np, e_np = host(g), host(eps)
            efg.sign_compress(g, eps, w.beta1, bits)
            del g
            bits_want, eps_want = oracle_pool.sign_ef_step(p, g_np, e_np, w.beta1)
            del g_np, e_np
            torch.cuda.synchronize()
            assert_bits_equal(bits, bits_want, f"bits step {step}")
            assert_bits_equal(eps, eps_want, f"eps step {step}")
            eps.copy_(torch.from_numpy(eps_want))
            del bits_want, eps_want


def test_slab_2p31_sign_receive_in_full():
    """Four workers' 1-bit packets over 2^31 elements (drawn by the input
    generator as random words), summed and applied with SGD; G and w are
    compared at every element."""
    w = wl.workload("slab_2p31")
    n = w.n
    nw = (n + 31) // 32
    gen = torch.Generator(device=DEV)
    gen.manual_seed(wl.seed(5, 9, 9))
    bit_list = [torch.randint(-2**31, 2**31 - 1, (nw,), dtype=torch.int32, device=DEV,
                              generator=gen) for _ in range(w.workers)]
    wt = w.weights(DEV)
    w_np = host(wt)
    G = torch.empty(n, device=DEV)
    efg.sign_aggregate_apply(bit_list, n, efg.APPLY_SGD, w.eta, w.beta1, G, wt)
    bits_np = [host(b).view(np.uint32) for b in bit_list]
    del bit_list
    with oracle_pool.pool() as p:
        G_want, w_want = oracle_pool.sign_aggregate_sgd(p, bits_np, n, w_np, w.eta)
    del bits_np, w_np
    torch.cuda.synchronize()
    assert_bits_equal(G, G_want, "G")
    del G, G_want
    assert_bits_equal(wt, w_want, "w")


@pytest.mark.parametrize("fmt", [efg.IDX_INT32, efg.IDX_BITMAP])
def test_slab_2p31_receive_side_four_workers(fmt):
    """W = 4 packets of 2,147,484 entries each (drawn by the input generator:
    sorted random positions, Student-t values, overlapping between workers),
    as indices or as bitmaps, summed into a dense G over 2^31 elements and
    applied with SGD; G and w are compared at every element."""
    w = wl.workload("slab_2p31")
    n, k = w.n, w.total_k
    rng = np.random.default_rng(11)
    common = rng.choice(n, k // 4, replace=False)
    packets = []
    for i in range(w.workers):
        idx = np.unique(np.concatenate([rng.choice(n, k - k // 4, replace=False), common]))
        vals = (rng.standard_t(3, idx.size) * 1e-3).astype(np.float32)
        packets.append({"indices": idx.astype(np.int32), "values": vals})
    wt = w.weights(DEV)
    w_np = host(wt)
    gpu_pk = []
    for p in packets:
        q = {"values": torch.from_numpy(p["values"]).to(DEV)}
        if fmt == efg.IDX_INT32:
            q["indices"] = torch.from_numpy(p["indices"]).to(DEV)
        else:   # element i -> bit i % 32 of word i // 32
            words = np.zeros((n + 31) // 32, np.uint32)
            ix = p["indices"].astype(np.int64)
            np.bitwise_or.at(words, ix >> 5, np.left_shift(1, ix & 31).astype(np.uint32))
            q["bitmap"] = torch.from_numpy(words.view(np.int32)).to(DEV)
        gpu_pk.append(q)
    G = _apply(gpu_pk, [p["values"].size for p in packets], n, w.eta, wt, fmt)
    del gpu_pk
    G_want = oracle.sparse_aggregate(packets, n)
    torch.cuda.synchronize()
    assert_bits_equal(G, G_want, "G")
    del G
    w_want = oracle.sgd_apply(w_np, G_want, w.eta)
    del G_want, w_np
    assert_bits_equal(wt, w_want, "w")


def test_bitmap_format_beyond_int32_range():
    """Bitmap packets have no index limit: a step over n = 2^31 + 69,995
    elements whose second tensor lies entirely beyond index 2^31 (the first,
    just under 2^31 elements, keeps k = 0 and is only compensated); then the
    receive side of that packet and a 1-bit step with a ragged tail."""
    big = (1 << 31) - 5
    small = 70_000
    n = big + small
    offs, ks = [0, big, n], [0, 700]
    g = wl.student_t3(n, 1e-3, wl.seed(5, 7, 1), DEV)
    e = wl.normal(n, 1e-4, wl.seed(5, 7, 2), DEV)
    g_np, e_np = host(g), host(e)
    want = oracle.topk_ef_step(g_np, e_np, offs, ks, "bitmap")
    out = gpu_topk(g, e, offs, ks, efg.IDX_BITMAP)
    torch.cuda.synchronize()
    assert efg.workspace_status(out["ws"]) == 0
    assert_bits_equal(out["values"], want["values"], "values")
    nz = np.flatnonzero(want["bitmap"])
    assert nz.min() >= (1 << 26) - 1                     # every set word lies past 2^31
    assert_bits_equal(out["bitmap"], want["bitmap"], "bitmap")
    assert_bits_equal(e, want["e"], "residual")
    del e, e_np
    # receive side of the bitmap packet over the same 2^31+ index space,
    # every element of G and w (the bitmap's set bits are want's selection)
    wt = wl.normal(n, 0.02, wl.seed(5, 7, 3), DEV)
    w_np = host(wt)
    sel = want["selected"]
    G = torch.empty(n, device=DEV)
    efg.sparse_aggregate_apply([out["values"]], None, [out["bitmap"]], [sum(ks)], n, 0.1, G, wt,
                               idx_format=efg.IDX_BITMAP)
    G_want = oracle.sparse_aggregate([{"indices": sel, "values": want["values"]}], n)
    torch.cuda.synchronize()
    assert_bits_equal(G, G_want, "G")
    assert_bits_equal(wt, oracle.sgd_apply(w_np, G_want, 0.1), "w")
    del G, wt, w_np, G_want
    # 1-bit step over the same length (ragged tail past 2^31), every element
    eps = wl.normal(n, 0.05, wl.seed(5, 7, 4), DEV)
    e_np = host(eps)
    bits = torch.empty((n + 31) // 32, dtype=torch.int32, device=DEV)
    efg.sign_compress(g, eps, 0.9, bits)
    with oracle_pool.pool() as p:
        bits_want, eps_want = oracle_pool.sign_ef_step(p, g_np, e_np, 0.9)
    torch.cuda.synchronize()
    assert_bits_equal(bits, bits_want, "bits")
    assert_bits_equal(eps, eps_want, "eps")
    last = host(bits[-1:]).view(np.uint32)[0]
    assert last >> (n % 32) == 0                         # padding bits are 0
