"""Pins for the CPU oracle, independent of the oracle's own code.

Each test ties an oracle function to something other than itself: the
hand-computed worked examples under tests/golden/ (with their citations),
brute force over tiny inputs with Python's own sort and the float's bit
pattern read through ``struct``, exact rational arithmetic (``fractions``)
on inputs where every float32 operation is exact, a library routine
(torch's stable sort), closed forms and invariants.  The last group plants
plausible mistakes into copies of the oracle and checks that the pins fail.
"""

import bisect
import json
import math
import os
import random
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import ef_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f(x):
    return float(x) if not isinstance(x, str) else float(x)


def _arr(xs):
    return np.array([_f(x) for x in xs], dtype=F32)


def _bits_of(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def _close(a, b, rel=1e-6):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    scale = max(np.max(np.abs(b)), 1e-30)
    return np.max(np.abs(a - b)) <= rel * scale


# ---------------------------------------------------------------------------
# top-k
# ---------------------------------------------------------------------------


def check_topk_golden(topk_step=None):
    topk_step = topk_step or oracle.topk_ef_step
    fx = _load("topk_two_steps.json")
    e = np.zeros(6, F32)
    for st in fx["steps"]:
        out = topk_step(_arr(st["g_raw"]), e, [0, 6], [fx["k"]])
        assert out["indices"].tolist() == st["indices"]
        assert out["values"].tolist() == st["values"]
        assert out["e"].tolist() == st["e"]
        e = out["e"]


def test_topk_worked_example():
    check_topk_golden()


def _brute_key(x):
    return 0x7FFFFFFF if math.isnan(x) else (_bits_of(x) & 0x7FFFFFFF)


def _brute_topk(vals, k):
    """Python sort of (-|x| bit pattern, index): the definition, by brute force."""
    keyed = sorted(range(len(vals)), key=lambda i: (-_brute_key(vals[i]), i))
    return sorted(keyed[:k])


def _tiny_cases(rng):
    levels = [0.0, -0.0, 1.0, -1.0, 0.5, -0.5, 2.0, 1e-30, -1e-30, 3.0e38]
    for n in list(range(1, 17)) + [31, 32, 33, 47, 64]:
        yield [rng.choice(levels) for _ in range(n)]               # many ties
        yield [rng.uniform(-1, 1) for _ in range(n)]               # distinct
        yield [rng.choice([0.25, -0.25]) for _ in range(n)]        # all one key
        yield [float("inf") if i % 7 == 3 else rng.gauss(0, 1) for i in range(n)]
        yield [float("nan") if i % 5 == 1 else rng.choice(levels) for i in range(n)]


def check_topk_bruteforce(topk_indices=None):
    topk_indices = topk_indices or oracle.topk_indices
    rng = random.Random(7)
    for vals in _tiny_cases(rng):
        g = np.array(vals, dtype=F32)
        gl = [float(x) for x in g]        # values after float32 rounding
        for k in range(len(vals) + 1):
            assert topk_indices(g, k).tolist() == _brute_topk(gl, k), (gl, k)


def test_topk_bruteforce_tiny():
    check_topk_bruteforce()


def test_topk_nan_ranks_above_inf():
    g = np.array([1.0, np.inf, np.nan, -np.inf, 2.0], dtype=F32)
    assert oracle.topk_indices(g, 1).tolist() == [2]
    assert oracle.topk_indices(g, 3).tolist() == [1, 2, 3]
    # NaNs tie whatever their payload: the lower index wins
    raw = np.array([0x7FC00000, 0x7FC00001, 0xFFC00000, 0x7F800001, 0x3F800000], np.uint32)
    g = raw.view(F32)
    assert oracle.topk_indices(g, 2).tolist() == [0, 1]
    assert oracle.topk_indices(g, 4).tolist() == [0, 1, 2, 3]


def test_topk_matches_torch_stable_sort():
    """Library routine: torch's stable descending sort of the |g| key gives
    the same index set (stable => lower index first among ties)."""
    rng = np.random.default_rng(3)
    for n, k in [(1000, 10), (4097, 41), (20000, 20), (5000, 5000), (777, 0)]:
        g = (rng.standard_t(3, n) * 1e-3).astype(F32)
        g[rng.integers(0, n, n // 10)] = F32(1e-3)          # plant ties
        g[rng.integers(0, n, n // 20)] = F32(-1e-3)
        key = torch.from_numpy(g.view(np.uint32).astype(np.int64) & 0x7FFFFFFF)
        order = torch.sort(key, descending=True, stable=True).indices[:k]
        want = torch.sort(order).values.numpy()
        assert np.array_equal(oracle.topk_indices(g, k), want)


def test_topk_invariants():
    rng = np.random.default_rng(11)
    n = 30011
    offs = [0, 5, 6, 1000, 1000, 17000, n]
    ks = [5, 1, 37, 0, 160, 13011]
    g_raw = (rng.standard_t(3, n) * 1e-3).astype(F32)
    g_raw[::97] = F32(2e-3)                                  # ties across segments
    e = (rng.standard_normal(n) * 1e-4).astype(F32)
    out = oracle.topk_ef_step(g_raw, e, offs, ks)
    g = (g_raw.astype(np.float64) + e.astype(np.float64)).astype(F32)  # exact-rounded sum
    idx = out["indices"].astype(np.int64)
    assert idx.size == sum(ks)
    assert np.all(np.diff(idx) > 0)
    dense = np.zeros(n, F32)
    dense[idx] = out["values"]
    # g~ + e' == g elementwise (values equal; the selected residual is +0)
    assert np.array_equal(dense + out["e"], g)
    assert np.all(out["e"][idx].view(np.uint32) == 0)
    key = g.view(np.uint32) & np.uint32(0x7FFFFFFF)
    for s, k in enumerate(ks):
        a, b = offs[s], offs[s + 1]
        sel = idx[(idx >= a) & (idx < b)]
        assert sel.size == k
        rest = np.setdiff1d(np.arange(a, b), sel)
        if k and rest.size:
            kmin = key[sel].min()
            assert kmin >= key[rest].max()
            # on the boundary key, every unselected index lies above every selected one
            tied_sel = sel[key[sel] == kmin]
            tied_rest = rest[key[rest] == kmin]
            if tied_rest.size:
                assert tied_sel.max() < tied_rest.min()


def test_topk_telescoping_exact():
    """Error feedback delays but never loses gradient ([SPARSE] §必不可少的误差补偿):
    sum_t g~_t + e_T = sum_t g_raw_t, exact here because every value is a
    small binary fraction (all float32 additions are exact)."""
    rng = np.random.default_rng(5)
    n, k, T = 257, 9, 12
    e = np.zeros(n, F32)
    sent = np.zeros(n, np.float64)
    total = np.zeros(n, np.float64)
    for _ in range(T):
        g_raw = (rng.integers(-64, 65, n) / 64.0).astype(F32)
        out = oracle.topk_ef_step(g_raw, e, [0, n], [k], "bitmap")
        idx = np.flatnonzero(oracle.unpack_bits(out["bitmap"], n))
        sent[idx] += out["values"].astype(np.float64)
        total += g_raw.astype(np.float64)
        e = out["e"]
    assert np.array_equal(sent + e.astype(np.float64), total)


def test_topk_edge_cases():
    g = np.array([3.0, -1.0, 2.0, -0.0, 0.0], dtype=F32)
    e = np.zeros(5, F32)
    out = oracle.topk_ef_step(g, e, [0, 5], [0])            # k = 0: nothing sent
    assert out["values"].size == 0 and np.array_equal(out["e"], g)
    out = oracle.topk_ef_step(g, e, [0, 5], [5])            # k = n: everything sent
    assert out["indices"].tolist() == [0, 1, 2, 3, 4]
    assert np.all(out["e"].view(np.uint32) == 0)
    out = oracle.topk_ef_step(np.full(9, 0.5, F32), np.zeros(9, F32), [0, 9], [4])
    assert out["indices"].tolist() == [0, 1, 2, 3]           # all equal: lowest indices
    out = oracle.topk_ef_step(np.zeros(0, F32), np.zeros(0, F32), [0, 0], [0])
    assert out["values"].size == 0
    with pytest.raises(ValueError):
        oracle.topk_ef_step(g, e, [0, 5], [6])


def check_layerwise_bruteforce(step=None):
    """A layerwise step against its definition written out independently:
    g = RN32(g_raw + e) formed in float64 and rounded once (exact for a sum
    of two floats, since 53 >= 2 * 24 + 2), each segment's top-k by the
    brute-force sort, global indices ascending, and a residual that is g off
    the selection and +0 on it."""
    step = step or oracle.topk_ef_step
    rng = np.random.default_rng(12)
    sizes, ks = [9, 40, 1, 33, 16], [3, 4, 1, 0, 16]
    offs = np.concatenate([[0], np.cumsum(sizes)]).tolist()
    n = offs[-1]
    levels = np.array([0.0, -0.0, 0.5, -0.5, 1.0, -1.0, 0.25], F32)
    for trial in range(4):
        g_raw = rng.choice(levels, n).astype(F32) if trial % 2 else rng.standard_normal(n).astype(F32)
        e = (rng.standard_normal(n) * 0.5).astype(F32)
        g = (g_raw.astype(np.float64) + e.astype(np.float64)).astype(F32)
        gl = [float(x) for x in g]
        want = []
        for s, k in enumerate(ks):
            want += [offs[s] + i for i in _brute_topk(gl[offs[s]:offs[s + 1]], k)]
        e_want = g.copy()
        e_want[want] = F32(0.0)
        out = step(g_raw, e, offs, ks)
        assert out["indices"].tolist() == want
        assert out["values"].view(np.uint32).tolist() == g[want].view(np.uint32).tolist()
        assert out["e"].view(np.uint32).tolist() == e_want.view(np.uint32).tolist()


def test_layerwise_bruteforce():
    check_layerwise_bruteforce()


def test_layerwise_equals_separate_tensors():
    """[SPARSE] §分层自适应Top-k: each tensor selects on its own, so one
    layerwise call equals one call per tensor (indices shifted)."""
    rng = np.random.default_rng(2)
    sizes, ks = [7, 100, 1, 64], [2, 10, 1, 0]
    offs = np.concatenate([[0], np.cumsum(sizes)]).tolist()
    g = rng.standard_normal(offs[-1]).astype(F32)
    e = rng.standard_normal(offs[-1]).astype(F32)
    whole = oracle.topk_ef_step(g, e, offs, ks)
    for s in range(len(sizes)):
        a, b = offs[s], offs[s + 1]
        part = oracle.topk_ef_step(g[a:b], e[a:b], [0, b - a], [ks[s]])
        m = (whole["indices"] >= a) & (whole["indices"] < b)
        assert np.array_equal(whole["indices"][m] - a, part["indices"])
        assert np.array_equal(whole["values"][m], part["values"])
        assert np.array_equal(whole["e"][a:b], part["e"])


def test_bitmap_packet_equals_index_packet():
    rng = np.random.default_rng(9)
    n = 1000
    g = rng.standard_normal(n).astype(F32)
    z = np.zeros(n, F32)
    a = oracle.topk_ef_step(g, z, [0, 300, n], [5, 17], "int32")
    b = oracle.topk_ef_step(g, z, [0, 300, n], [5, 17], "bitmap")
    assert np.array_equal(np.flatnonzero(oracle.unpack_bits(b["bitmap"], n)), a["indices"])
    assert np.array_equal(a["values"], b["values"])
    assert np.array_equal(a["e"], b["e"])


# ---------------------------------------------------------------------------
# bit layout
# ---------------------------------------------------------------------------


def check_pack_bits(pack=None):
    pack = pack or oracle.pack_bits
    rng = random.Random(1)
    for n in [1, 3, 31, 32, 33, 64, 65, 100]:
        flags = [rng.random() < 0.4 for _ in range(n)]
        want = [0] * ((n + 31) // 32)
        for i, f in enumerate(flags):
            if f:
                want[i // 32] |= 1 << (i % 32)
        assert pack(np.array(flags)).tolist() == want
    assert pack(np.array([True, False, True, True])).tolist() == [13]


def test_pack_bits_lsb_first():
    check_pack_bits()
    flags = np.random.default_rng(0).random(77) < 0.5
    assert np.array_equal(oracle.unpack_bits(oracle.pack_bits(flags), 77), flags)


# ---------------------------------------------------------------------------
# 1-bit sign error feedback and momentum
# ---------------------------------------------------------------------------


def check_sign_golden(sign_step=None, momentum=None):
    sign_step = sign_step or oracle.sign_ef_step
    momentum = momentum or oracle.onebit_momentum
    fx = _load("sign_two_steps.json")
    eps = np.zeros(4, F32)
    m = np.zeros(4, F32)
    for st in fx["steps"]:
        words, eps = sign_step(_arr(st["g"]), eps, fx["beta1"])
        assert words.tolist() == st["words"]
        assert _close(eps, _arr(st["eps"]))
        m = momentum(m, oracle.decode_signs(words, 4), fx["beta1"])
        assert _close(m, _arr(st["m"]))


def test_sign_worked_example():
    check_sign_golden()


def test_sign_bits_definition():
    """bit = 1 unless g + eps < 0: sign(0) = +1 for +0 and -0; NaN gives 1."""
    g = np.array([0.0, -0.0, -1e-45, 1e-45, np.nan, -np.inf, np.inf, -2.0, 2.0], F32)
    words, _ = oracle.sign_ef_step(g, np.zeros_like(g), 0.9)
    want = sum(1 << i for i, x in enumerate(g.tolist()) if not (x < 0))
    assert words.tolist() == [want]
    # eps shifts the decision: g + eps crosses zero
    words, _ = oracle.sign_ef_step(np.array([0.5, -0.5], F32),
                                   np.array([-1.0, 1.0], F32), 0.9)
    assert words.tolist() == [0b10]


def _sign_exact(g, eps, beta1):
    """The §2.1 formulas in exact rational arithmetic."""
    v = [Fraction(a) + Fraction(b) for a, b in zip(g, eps)]
    s = [Fraction(-1) if x < 0 else Fraction(1) for x in v]
    d = [x - y for x, y in zip(v, s)]
    b1 = Fraction(beta1)
    return s, [b1 * Fraction(e) + (1 - b1) * dd for e, dd in zip(eps, d)]


def test_sign_exact_rational():
    """Binary-fraction inputs and beta1 in {0.5, 0.75}: every float32 step is
    exact, so the oracle must equal the formulas evaluated in Fractions."""
    rng = random.Random(4)
    for beta1 in (0.5, 0.75, 0.0, 1.0):
        n = 70
        eps = np.zeros(n, F32)
        m = np.zeros(n, F32)
        m_exact = [Fraction(0)] * n
        for _ in range(4):
            g = np.array([rng.randint(-32, 32) / 16 for _ in range(n)], F32)
            s, eps_exact = _sign_exact(g.tolist(), eps.tolist(), beta1)
            words, eps = oracle.sign_ef_step(g, eps, beta1)
            assert [Fraction(x) for x in eps.tolist()] == eps_exact
            assert oracle.decode_signs(words, n).tolist() == [float(x) for x in s]
            b1 = Fraction(beta1)
            m_exact = [b1 * a + (1 - b1) * b for a, b in zip(m_exact, s)]
            m = oracle.onebit_momentum(m, oracle.decode_signs(words, n), beta1)
            assert [Fraction(x) for x in m.tolist()] == m_exact


def test_sign_closed_forms():
    rng = np.random.default_rng(8)
    g = rng.standard_normal(1000).astype(F32)
    eps = rng.standard_normal(1000).astype(F32)
    v = (g + eps).astype(F32)
    s = np.where(v < 0, F32(-1), F32(1))
    _, e0 = oracle.sign_ef_step(g, eps, 0.0)     # beta1 = 0: eps' = Delta
    assert np.array_equal(e0, (v - s).astype(F32))
    _, e1 = oracle.sign_ef_step(g, eps, 1.0)     # beta1 = 1: eps' = eps
    assert np.array_equal(e1, eps)


def test_one_minus_beta1_in_float32():
    # 1 - float32(0.9) = 0.10000002384185791015625 exactly (Sterbenz)
    _, eps = oracle.sign_ef_step(np.array([-1.0], F32), np.zeros(1, F32), 0.9)
    # v = -1, s = -1, Delta = 0 -> eps' = 0
    assert eps.tolist() == [0.0]
    m = oracle.onebit_momentum(np.zeros(1, F32), np.ones(1, F32), 0.9)
    assert m.tolist() == [0.10000002384185791015625]


# ---------------------------------------------------------------------------
# receive side
# ---------------------------------------------------------------------------


def _packets(ex):
    return [{"indices": np.array(p["indices"], np.int32), "values": _arr(p["values"])}
            for p in ex["packets"]]


def check_aggregate_golden(aggregate=None, sgd=None):
    aggregate = aggregate or oracle.sparse_aggregate
    sgd = sgd or oracle.sgd_apply
    fx = _load("aggregate_examples.json")
    for ex in fx["examples"]:
        G = aggregate(_packets(ex), ex["n"])
        assert G.tolist() == [float(x) for x in ex["G"]], ex["name"]
        if "G_signbit" in ex:
            assert np.signbit(G).tolist() == ex["G_signbit"]
        w = sgd(_arr(ex["w0"]), G, ex["eta"])
        want = _arr(ex["w"])
        if ex["name"] == "two_workers":
            assert _close(w, want)
            assert w[5] == 1.0 and w[0] == 1.0
        else:
            assert w.view(np.uint32).tolist() == want.view(np.uint32).tolist()


def test_aggregate_worked_examples():
    check_aggregate_golden()


def test_aggregate_exact_rational():
    rng = random.Random(12)
    n, W = 300, 5
    packets, exact = [], [Fraction(0)] * n
    for _ in range(W):
        idx = sorted(rng.sample(range(n), rng.randint(0, 60)))
        vals = [rng.randint(-1000, 1000) / 256 for _ in idx]
        packets.append({"indices": np.array(idx, np.int32), "values": np.array(vals, F32)})
        for i, v in zip(idx, vals):
            exact[i] += Fraction(v)
    G = oracle.sparse_aggregate(packets, n)
    assert [Fraction(x) for x in G.tolist()] == exact
    w0 = np.array([rng.randint(-100, 100) / 8 for _ in range(n)], F32)
    w = oracle.sgd_apply(w0, G, 0.25)
    assert [Fraction(x) for x in w.tolist()] == [
        Fraction(a) - Fraction(1, 4) * b for a, b in zip(w0.tolist(), exact)]


def test_aggregate_single_worker_is_scatter():
    rng = np.random.default_rng(6)
    n = 5000
    idx = np.sort(rng.choice(n, 300, replace=False)).astype(np.int32)
    vals = rng.standard_normal(300).astype(F32)
    G = oracle.sparse_aggregate([{"indices": idx, "values": vals}], n)
    want = np.zeros(n, F32)
    want[idx] = vals
    assert np.array_equal(G, want)


def test_sgd_leaves_untouched_bitwise():
    w = np.array([1.5, -0.0, 0.0, np.inf, 3.0e-45], F32)
    out = oracle.sgd_apply(w, np.zeros(5, F32), 0.37)
    assert out.view(np.uint32).tolist() == w.view(np.uint32).tolist()


def test_aggregate_rejects_unsorted():
    with pytest.raises(ValueError):
        oracle.sparse_aggregate([{"indices": np.array([3, 1], np.int32),
                                  "values": np.ones(2, F32)}], 5)


def check_sign_aggregate_counts(aggregate=None):
    aggregate = aggregate or oracle.sign_aggregate
    rng = random.Random(3)
    n, W = 77, 6
    flags = [[rng.random() < 0.5 for _ in range(n)] for _ in range(W)]
    G = aggregate([oracle.pack_bits(np.array(f)) for f in flags], n)
    want = [sum(1 if flags[w][i] else -1 for w in range(W)) for i in range(n)]
    assert G.tolist() == [float(x) for x in want]


def test_sign_aggregate_counts():
    check_sign_aggregate_counts()


# ---------------------------------------------------------------------------
# 8-bit quantisation of the selected values
# ---------------------------------------------------------------------------


def _fx(x):
    return float(x)   # json strings "inf" / "nan" parse through float()


def check_q8_golden(scale=None, quantize=None, dequantize=None):
    scale = scale or oracle.q8_scale
    quantize = quantize or oracle.q8_quantize
    dequantize = dequantize or oracle.q8_dequantize
    for ex in _load("q8_examples.json")["quantise"]:
        v = np.array([_fx(x) for x in ex["values"]], F32)
        s = scale(v)
        assert float(s) == ex["scale"], ex["name"]
        q = quantize(v, s)
        assert q.dtype == np.int8 and q.tolist() == ex["q"], ex["name"]
        dq = dequantize(q, s)
        assert dq.tolist() == ex["dequantised"], ex["name"]
        with np.errstate(invalid="ignore"):
            r = np.subtract(v, dq, dtype=F32)
        want = np.array([_fx(x) for x in ex["residual"]], F32)
        assert np.array_equal(np.isnan(r), np.isnan(want)), ex["name"]
        ok = ~np.isnan(want)
        assert [_bits_of(float(x)) for x in r[ok]] == [_bits_of(float(x)) for x in want[ok]]


def check_q8_ef_golden(step=None):
    step = step or oracle.topk_q8_ef_step
    fx = _load("q8_examples.json")["ef_step"]
    out = step(_arr(fx["g_raw"]), np.zeros(6, F32), [0, 6], [fx["k"]])
    assert out["indices"].tolist() == fx["indices"]
    assert out["values"].tolist() == fx["values"]
    assert out["scales"].tolist() == [fx["scale"]]
    assert out["q"].tolist() == fx["q"]
    assert out["e"].tolist() == fx["e"]


def test_q8_worked_examples():
    check_q8_golden()
    check_q8_ef_golden()


def test_q8_invariants_random():
    """On random finite values: |q| <= 127; the largest |v| maps to +-127;
    sign(q) is 0 or sign(v); q is monotone in v; |v - q s| <= s / 2 (one
    rounding of slack); and q s + (v - q s) == v bit for bit, because for
    q != 0 the two terms lie within a factor 2 of each other (Sterbenz), so
    the residual subtraction is exact: the receiver's value plus the new
    residual gives back g exactly."""
    rng = np.random.default_rng(4)
    for trial in range(50):
        n = int(rng.integers(1, 2000))
        v = (rng.standard_t(3, n) * 10.0 ** rng.uniform(-8, 3)).astype(F32)
        s = oracle.q8_scale(v)
        assert s == np.float32(np.max(np.abs(v))) / np.float32(127)
        q = oracle.q8_quantize(v, s)
        assert np.all(np.abs(q.astype(np.int32)) <= 127)
        assert abs(int(q[np.argmax(np.abs(v))])) == 127
        assert np.all((q == 0) | (np.sign(q) == np.sign(v)))
        order = np.argsort(v, kind="stable")
        assert np.all(np.diff(q[order].astype(np.int32)) >= 0)
        dq = oracle.q8_dequantize(q, s)
        r = np.subtract(v, dq, dtype=F32)
        assert np.all(np.abs(r.astype(np.float64)) <= 0.5 * float(s) * (1 + 2.0 ** -20))
        assert np.array_equal(np.add(dq, r, dtype=F32).view(np.uint32), v.view(np.uint32))


def test_q8_ef_step_residual_identity():
    """A quantised top-k EF step against the plain step: same selection and
    values; off the selection the residuals agree bit for bit; on it the
    receiver's value plus the residual is g exactly; per-segment scales."""
    rng = np.random.default_rng(9)
    n = 5000
    offs, ks = [0, 100, 1700, 5000], [7, 40, 90]
    g_raw = (rng.standard_t(3, n) * 1e-3).astype(F32)
    e = (rng.standard_normal(n) * 1e-4).astype(F32)
    plain = oracle.topk_ef_step(g_raw, e, offs, ks)
    q8 = oracle.topk_q8_ef_step(g_raw, e, offs, ks)
    assert q8["indices"].tolist() == plain["indices"].tolist()
    assert q8["values"].tolist() == plain["values"].tolist()
    off = np.ones(n, bool)
    off[plain["indices"]] = False
    assert np.array_equal(q8["e"][off].view(np.uint32), plain["e"][off].view(np.uint32))
    j = 0
    for si, k in enumerate(ks):
        v = plain["values"][j:j + k]
        assert q8["scales"][si] == oracle.q8_scale(v)
        dq = oracle.q8_dequantize(q8["q"][j:j + k], q8["scales"][si])
        idx = plain["indices"][j:j + k]
        g = oracle.compensate(g_raw, e)[idx]
        assert np.array_equal(np.add(dq, q8["e"][idx], dtype=F32).view(np.uint32), g.view(np.uint32))
        j += k


# ---------------------------------------------------------------------------
# index codecs
# ---------------------------------------------------------------------------

CODECS = {"local16": ("encode_local16", "decode_local16"),
          "runvarint": ("encode_runvarint", "decode_runvarint"),
          "block256": ("encode_block256", "decode_block256")}


def check_codec_golden(name, encode=None, decode=None):
    enc = encode or getattr(oracle, CODECS[name][0])
    dec = decode or getattr(oracle, CODECS[name][1])
    ex = _load("index_codec_examples.json")[name]
    b = enc(np.array(ex["indices"], np.int64), ex["n"])
    assert b.dtype == np.uint8 and b.tolist() == ex["bytes"], name
    assert dec(np.array(ex["bytes"], np.uint8), len(ex["indices"]), ex["n"]).tolist() == ex["indices"]


def check_leb128(leb=None):
    leb = leb or oracle.leb128
    fx = _load("index_codec_examples.json")["leb128"]
    assert leb(fx["value"]) == fx["bytes"]
    # closed form: ceil(bits / 7) bytes, at least one; each byte's low 7 bits
    # are the value's 7-bit groups from the least significant up
    for x in [0, 1, 127, 128, 16383, 16384, 2**21 - 1, 2**21, 2**28, 2**31 - 1]:
        bs = leb(x)
        assert len(bs) == max(1, -(-x.bit_length() // 7))
        assert all(b & 0x80 for b in bs[:-1]) and not bs[-1] & 0x80
        assert sum((b & 0x7F) << (7 * i) for i, b in enumerate(bs)) == x


def test_codec_worked_examples():
    for name in CODECS:
        check_codec_golden(name)
    check_leb128()


def _random_index_sets(rng):
    yield np.zeros(0, np.int64), 1000
    yield np.array([999], np.int64), 1000
    yield np.arange(70000, dtype=np.int64), 70000           # every element
    for _ in range(20):
        n = int(rng.integers(1, 400_000))
        k = int(rng.integers(0, min(n, 5000) + 1))
        yield np.sort(rng.choice(n, k, replace=False)).astype(np.int64), n
    # clustered: runs of neighbours and long gaps
    n = 3_000_000
    starts = np.sort(rng.choice(n - 300, 40, replace=False))
    yield np.unique(np.concatenate([s + np.arange(int(rng.integers(1, 300))) for s in starts])), n


def test_codec_sizes_and_round_trip():
    """Every codec's stream length follows from its definition in closed
    form, and decoding gives the packet back."""
    rng = np.random.default_rng(12)
    for idx, n in _random_index_sets(rng):
        K = idx.size
        nblk = -(-n // 65536)
        nb = -(-n // 256)
        runs = np.diff(np.concatenate([[-1], idx])) - 1
        sizes = {"local16": 4 * (nblk + 1) + 2 * K,
                 "runvarint": int(sum(max(1, -(-int(r).bit_length() // 7)) for r in runs)),
                 "block256": 4 * (-(-nb // 32)) + np.unique(idx // 256).size + K}
        for name, (e, d) in CODECS.items():
            b = getattr(oracle, e)(idx, n)
            assert b.size == sizes[name], (name, n, K)
            assert getattr(oracle, d)(b, K, n).astype(np.int64).tolist() == idx.tolist(), name


# ---------------------------------------------------------------------------
# random magnitude-proportional sparsification
# ---------------------------------------------------------------------------


def check_philox_kat(philox=None):
    philox = philox or oracle.philox4x32_10
    for v in _load("randk_examples.json")["philox_kat"]:
        c = [int(x, 16) for x in v["ctr"]]
        k = [int(x, 16) for x in v["key"]]
        out = philox(*c, *k)
        assert ["%08x" % int(x) for x in out] == v["out"]


def check_randk_golden(step_fn=None):
    step_fn = step_fn or oracle.randk_ef_step
    for name in ("step", "step2"):
        fx = _load("randk_examples.json")[name]
        out = step_fn(_arr(fx["g_raw"]), np.zeros(4, F32), [0, 4], [fx["k"]], fx["seed"],
                      fx["step"], 10)
        assert out["values"].tolist() == fx["values"], name
        assert out["indices"].tolist() == fx["indices"], name
        assert out["e"].tolist() == fx["e"], name


def test_randk_worked_example_and_generator():
    check_philox_kat()
    check_randk_golden()
    # words of elements 4..7 come from counter 1: its first word differs
    w = oracle.randk_words(0, 8, 0, 0)
    assert ["%08x" % x for x in w[:4]] == _load("randk_examples.json")["philox_kat"][0]["out"]
    assert w[4] != w[0]


def test_randk_scale_is_the_exact_sum():
    """S equals the exact rational sum of the |g| (fractions), rounded once
    to float64 by Python's correctly rounded conversion."""
    rng = np.random.default_rng(21)
    for trial in range(30):
        n = int(rng.integers(1, 3000))
        g = (rng.standard_t(2, n) * 10.0 ** rng.uniform(-30, 30, n)).astype(F32)
        g[rng.integers(0, n, 3)] = np.float32("nan")
        fin = g[np.isfinite(g)]
        exact = sum((Fraction(float(abs(x))) for x in fin), Fraction(0))
        assert oracle.randk_scale(g) == float(exact)


def test_randk_keep_statistics():
    """Over many seeds the kept count averages k (no element is clipped
    here) and each element's keep frequency is p_i = k |g_i| / S."""
    rng = np.random.default_rng(8)
    n, k = 400, 40
    g = (rng.standard_normal(n) * 1e-3).astype(F32)
    p = np.abs(g).astype(np.float64) * float(oracle.randk_coefficient(g, k))
    assert abs(p.sum() - k) < 1e-4 * k
    assert p.max() < 1
    trials = 2000
    freq = np.zeros(n)
    counts = []
    for t in range(trials):
        keep = oracle.randk_keep(g, k, 0, seed=1234, step=t)
        freq += keep
        counts.append(keep.sum())
    assert abs(np.mean(counts) - k) < 4 * np.sqrt(np.sum(p * (1 - p)) / trials)
    z = (freq / trials - p) / np.sqrt(p * (1 - p) / trials)
    assert np.max(np.abs(z)) < 5.5


def test_randk_special_cases():
    g = np.array([0, 0, 0, 0, 0], F32)
    assert not oracle.randk_keep(g, 3, 0, 1, 1).any()                     # S = 0
    g = np.array([1e30, 1e-3, np.inf, np.nan, 1e-3], F32)
    keep = oracle.randk_keep(g, 2, 0, 5, 6)
    assert keep[0] and keep[2] and keep[3]            # clipped to 1, and the non-finite
    out = oracle.randk_ef_step(np.ones(1000, F32), np.zeros(1000, F32), [0, 1000], [1000], 9, 9, 7)
    assert out["kept"] == 1000 and out["indices"].tolist() == list(range(7))   # capacity cut
    assert np.all(out["e"][7:] == 1) and np.all(out["e"][:7] == 0)


# ---------------------------------------------------------------------------
# packet split for the index-range exchange ([SPARSE] §详细算法流程 step 5)
# ---------------------------------------------------------------------------


def check_packet_split(split=oracle.packet_split):
    # worked by hand: entries 2, 5, 9, 10; ranges [0,5), [5,10), [10,11), [11,...)
    assert split([2, 5, 9, 10], [0, 5, 10, 11, 20]).tolist() == [0, 1, 3, 4, 4]
    assert split([], [0, 7]).tolist() == [0, 0]
    assert split([0], [0, 1]).tolist() == [0, 1]
    # the lower bound of a sorted list, as the standard library's bisection finds it
    rng = np.random.default_rng(33)
    for _ in range(200):
        n = int(rng.integers(1, 80))
        idx = np.sort(rng.choice(n, int(rng.integers(0, n + 1)), replace=False))
        bounds = np.sort(rng.integers(0, n + 2, int(rng.integers(1, 9))))
        got = split(idx, bounds)
        want = [bisect.bisect_left(idx.tolist(), int(b)) for b in bounds]
        assert got.tolist() == want
        # consecutive slices hold exactly the entries of their ranges
        for q in range(len(bounds) - 1):
            part = idx[got[q]:got[q + 1]]
            assert np.all((part >= bounds[q]) & (part < bounds[q + 1]))


def test_packet_split_pins():
    check_packet_split()


# ---------------------------------------------------------------------------
# planted mistakes: the pins above must catch them
# ---------------------------------------------------------------------------


def _topk_ties_to_higher_index(g, k):
    g = np.ascontiguousarray(g, dtype=F32)
    n = g.size
    if k == 0:
        return np.zeros(0, np.int64)
    rank = (oracle.abs_key(g).astype(np.uint64) << np.uint64(32)) | np.arange(n, dtype=np.uint64)
    rank.partition(n - k)
    return np.sort((rank[n - k:] & np.uint64(0xFFFFFFFF)).astype(np.int64))


def _topk_signed_not_abs(g, k):
    g = np.ascontiguousarray(g, dtype=F32)
    if k == 0:
        return np.zeros(0, np.int64)
    order = np.argsort(-g.astype(np.float64), kind="stable")
    return np.sort(order[:k])


def _pack_msb_first(flags):
    flags = np.asarray(flags, dtype=bool)
    words = oracle.pack_bits(flags)
    return np.array([int(f"{int(w):032b}"[::-1], 2) for w in words], np.uint32)


def _sign_step_wrong_ema(g, eps, beta1):
    bits, _ = oracle.sign_ef_step(g, eps, beta1)
    v = (g + eps).astype(F32)
    s = np.where(v < 0, F32(-1), F32(1))
    # mistake: the two EMA weights swapped
    return bits, ((F32(1) - F32(beta1)) * eps + F32(beta1) * (v - s)).astype(F32)


def _sign_zero_is_zero(g, eps, beta1):
    # mistake: torch-style sign(0) = 0 would mark 0 as "not positive"
    v = (np.asarray(g, F32) + np.asarray(eps, F32)).astype(F32)
    bits = oracle.pack_bits(v > 0)
    _, e = oracle.sign_ef_step(g, eps, beta1)
    return bits, e


def _step_segment_local_indices(g_raw, e, offs, ks, idx_format="int32"):
    out = oracle.topk_ef_step(g_raw, e, offs, ks, idx_format)
    seg = np.searchsorted(np.asarray(offs), out["selected"], side="right") - 1
    out["indices"] = (out["selected"] - np.asarray(offs)[seg]).astype(np.int32)
    return out


def _step_selects_over_the_whole_buffer(g_raw, e, offs, ks, idx_format="int32"):
    n = len(g_raw)
    return oracle.topk_ef_step(g_raw, e, [0, n], [sum(ks)], idx_format)


def _step_compensates_with_minus(g_raw, e, offs, ks, idx_format="int32"):
    return oracle.topk_ef_step(g_raw, (-np.asarray(e, F32)).astype(F32), offs, ks, idx_format)


def _step_residual_keeps_selection(g_raw, e, offs, ks, idx_format="int32"):
    out = oracle.topk_ef_step(g_raw, e, offs, ks, idx_format)
    out["e"] = oracle.compensate(g_raw, e)
    return out


def _sign_decision_ignores_eps(g, eps, beta1):
    # mistake: the sign taken of g alone, the error buffer only in the update
    _, e = oracle.sign_ef_step(g, eps, beta1)
    return oracle.pack_bits(~(np.asarray(g, F32) < 0)), e


def _momentum_swapped_weights(m, ghat, beta1):
    b1 = F32(beta1)
    return ((F32(1) - b1) * np.asarray(m, F32) + b1 * np.asarray(ghat, F32)).astype(F32)


def _sign_aggregate_bit_one_is_minus(bit_vectors, n):
    return (-oracle.sign_aggregate(bit_vectors, n)).astype(F32)


def _aggregate_averages(packets, n):
    # mistake: the receiver divides by the worker count (the pages add)
    return (oracle.sparse_aggregate(packets, n) / F32(len(packets))).astype(F32)


def _aggregate_reverse_order(packets, n):
    return oracle.sparse_aggregate(list(reversed(packets)), n)


def _sgd_wrong_sign(w, G, eta):
    return (np.asarray(w, F32) + F32(eta) * np.asarray(G, F32)).astype(F32)


def _leb128_high_group_first(x):
    return list(reversed([b & 0x7F for b in oracle.leb128(x)]))


def _runvarint_plain_delta(idx, n):
    prev, out = 0, []
    for i in np.asarray(idx, np.int64).tolist():
        out.extend(oracle.leb128(i - prev))
        prev = i
    return np.array(out, np.uint8)


def _block256_counts_not_minus_one(idx, n):
    b = oracle.encode_block256(idx, n)
    nfw = -(-(-(-n // 256)) // 32)
    nnzb = b.size - 4 * nfw - len(idx)
    b[4 * nfw:4 * nfw + nnzb] += 1
    return b


def _local16_starts_after_block(idx, n):
    b = oracle.encode_local16(idx, n)
    nblk = -(-n // 65536)
    starts = b[:4 * (nblk + 1)].view("<u4").copy()
    return np.concatenate([np.append(starts[1:], starts[-1]).astype("<u4").view(np.uint8),
                           b[4 * (nblk + 1):]])


def _philox_key_bumped_first(c0, c1, c2, c3, k0, k1):
    return ef_oracle.philox4x32_10(c0, c1, c2, c3, (k0 + 0x9E3779B9) & 0xFFFFFFFF,
                                   (k1 + 0xBB67AE85) & 0xFFFFFFFF)


def _randk_scaled_by_inverse_p(g_raw, e, offs, ks, seed, step, capacity):
    out = oracle.randk_ef_step(g_raw, e, offs, ks, seed, step, capacity)
    g = oracle.compensate(g_raw, e)
    c = oracle.randk_coefficient(g, ks[0])
    p = np.minimum(F32(1), c * np.abs(g[out["indices"]]))
    out["values"] = (out["values"] / p).astype(F32)
    return out


def _randk_uses_element_index_as_counter(g_raw, e, offs, ks, seed, step, capacity):
    g = oracle.compensate(g_raw, e)
    c = oracle.randk_coefficient(g, ks[0])
    i = np.arange(g.size)
    w = np.array([int(oracle.philox4x32_10(x, 0, step, 0, seed, 0)[0]) for x in i], np.uint32)
    u = (w >> np.uint32(8)).astype(F32) * F32(2.0 ** -24)
    keep = u < np.minimum(F32(1), c * np.abs(g))
    sel = np.flatnonzero(keep)[:capacity]
    e2 = g.copy()
    e2[sel] = 0
    return {"values": g[sel], "indices": sel.astype(np.int32), "e": e2}


def _q8_round_half_away(values, s):
    v = np.asarray(values, F32)
    q = np.zeros(v.size, np.int8)
    if F32(s) == F32(0):
        return q
    ok = ~np.isnan(v)
    t = np.clip(np.divide(v[ok], F32(s), dtype=F32), -127, 127)
    q[ok] = (np.sign(t) * np.floor(np.abs(t) + F32(0.5))).astype(np.int8)
    return q


def _q8_scale_over_128(values):
    return np.float32(oracle.q8_scale(values) * np.float32(127) / np.float32(128))


def _q8_scale_with_inf(values):
    v = np.asarray(values, F32)
    m = np.max(np.abs(v[~np.isnan(v)])) if v.size else F32(0)
    return np.divide(F32(m), F32(127), dtype=F32)


def _q8_step_drops_quantisation_error(g_raw, e, offs, ks, idx_format="int32"):
    out = oracle.topk_q8_ef_step(g_raw, e, offs, ks, idx_format)
    out["e"][out["selected"]] = F32(0)
    return out


def _split_counts_equal_too(indices, bounds):
    idx = np.asarray(indices, dtype=np.int64)
    return np.array([int(np.count_nonzero(idx <= int(b))) for b in bounds], dtype=np.int64)


@pytest.mark.parametrize("check,kwargs", [
    (check_topk_bruteforce, {"topk_indices": _topk_ties_to_higher_index}),
    (check_topk_bruteforce, {"topk_indices": _topk_signed_not_abs}),
    (check_layerwise_bruteforce, {"step": _step_segment_local_indices}),
    (check_layerwise_bruteforce, {"step": _step_selects_over_the_whole_buffer}),
    (check_layerwise_bruteforce, {"step": _step_compensates_with_minus}),
    (check_layerwise_bruteforce, {"step": _step_residual_keeps_selection}),
    (check_pack_bits, {"pack": _pack_msb_first}),
    (check_sign_golden, {"sign_step": _sign_step_wrong_ema}),
    (check_sign_golden, {"sign_step": _sign_zero_is_zero}),
    (check_sign_golden, {"sign_step": _sign_decision_ignores_eps}),
    (check_sign_golden, {"momentum": _momentum_swapped_weights}),
    (check_sign_aggregate_counts, {"aggregate": _sign_aggregate_bit_one_is_minus}),
    (check_aggregate_golden, {"aggregate": _aggregate_reverse_order}),
    (check_aggregate_golden, {"aggregate": _aggregate_averages}),
    (check_aggregate_golden, {"sgd": _sgd_wrong_sign}),
    (check_q8_golden, {"quantize": _q8_round_half_away}),
    (check_q8_golden, {"scale": _q8_scale_over_128}),
    (check_q8_golden, {"scale": _q8_scale_with_inf}),
    (check_q8_ef_golden, {"step": _q8_step_drops_quantisation_error}),
    (check_leb128, {"leb": _leb128_high_group_first}),
    (check_philox_kat, {"philox": _philox_key_bumped_first}),
    (check_randk_golden, {"step_fn": _randk_scaled_by_inverse_p}),
    (check_randk_golden, {"step_fn": _randk_uses_element_index_as_counter}),
    (lambda **kw: check_codec_golden("runvarint", **kw), {"encode": _runvarint_plain_delta}),
    (lambda **kw: check_codec_golden("block256", **kw), {"encode": _block256_counts_not_minus_one}),
    (lambda **kw: check_codec_golden("local16", **kw), {"encode": _local16_starts_after_block}),
    (check_packet_split, {"split": _split_counts_equal_too}),
])
def test_pins_catch_planted_mistakes(check, kwargs):
    with pytest.raises(AssertionError):
        check(**kwargs)


def test_topk_golden_catches_dropped_residual():
    def no_feedback(g_raw, e, offs, ks, idx_format="int32"):
        return ef_oracle.topk_ef_step(g_raw, np.zeros_like(e), offs, ks, idx_format)
    with pytest.raises(AssertionError):
        check_topk_golden(no_feedback)
