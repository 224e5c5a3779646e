"""The C-ABI library loads on a machine without a GPU, exports every symbol
include/efgrad.h declares, and its host-side validation rejects bad
arguments before touching the device (no compute calls here)."""

import ctypes
import os
import re

import pytest

import error_feedback_gradient_gb300 as efg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "efgrad.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(efg.library_path()):
        import __graft_entry__
        __graft_entry__.build()
    return efg.library()


def _declared():
    text = open(HEADER).read()
    return re.findall(r"^EF_API\s+[\w\s\*]+?\b(\w+)\(", text, flags=re.M)


def _header_defines():
    text = open(HEADER).read()
    return {m[0]: int(m[1]) for m in re.findall(r"^#define (EF_\w+)\s+(-?\d+)", text, flags=re.M)}


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 11
    for name in names:
        assert hasattr(lib, name), name


def test_binding_covers_header(lib):
    from error_feedback_gradient_gb300 import binding
    assert set(_declared()) == set(binding._SIGNATURES)


def test_constants_match_header():
    d = _header_defines()
    from error_feedback_gradient_gb300 import binding
    assert d["EF_IDX_INT32"] == binding.IDX_INT32 and d["EF_IDX_BITMAP"] == binding.IDX_BITMAP
    assert d["EF_APPLY_SGD"] == binding.APPLY_SGD
    assert d["EF_APPLY_MOMENTUM"] == binding.APPLY_MOMENTUM
    assert d["EF_KERNEL_TOPK_FUSED"] == binding.KERNEL_TOPK_FUSED


def test_status_strings(lib):
    d = _header_defines()
    for name, v in d.items():
        if name.startswith("EF_ERR_") or name == "EF_OK":
            s = lib.ef_status_string(v)
            assert s and b"unknown" not in s, name
    assert lib.ef_abi_version() == d["EF_ABI_VERSION"]


def _i64(xs):
    return (ctypes.c_int64 * len(xs))(*xs)


def _ws_size(lib, n, offs, ks, fmt=0):
    out = ctypes.c_size_t(0)
    st = lib.ef_topk_workspace_size(n, len(ks), _i64(offs), _i64(ks), fmt, ctypes.byref(out))
    return st, out.value


def test_topk_workspace_queries(lib):
    d = _header_defines()
    st, small = _ws_size(lib, 1000, [0, 1000], [10])
    assert st == d["EF_OK"] and small >= 256
    st, big = _ws_size(lib, 1 << 24, [0, 1 << 24], [16777])
    assert st == d["EF_OK"] and big > 4 * 16777 * 8          # candidate list
    st, _ = _ws_size(lib, 100, [0, 50, 100], [51, 1])
    assert st == d["EF_ERR_K"]
    st, _ = _ws_size(lib, 100, [0, 60, 50, 100], [1, 1, 1])
    assert st == d["EF_ERR_SEGMENTS"]
    st, _ = _ws_size(lib, 100, [0, 99], [1])
    assert st == d["EF_ERR_SEGMENTS"]
    st, _ = _ws_size(lib, 100, [0, 100], [1], fmt=7)
    assert st == d["EF_ERR_ARG"]
    st, _ = _ws_size(lib, (1 << 31) + 1, [0, 1 << 30, (1 << 31) + 1], [1, 1], fmt=0)
    assert st == d["EF_ERR_SIZE"]                             # int32 indices overflow
    st, _ = _ws_size(lib, (1 << 31) + 1, [0, 1 << 30, (1 << 31) + 1], [1, 1], fmt=1)
    assert st == d["EF_OK"]                                   # bitmap has no index limit
    st, _ = _ws_size(lib, 1 << 31, [0, 1 << 31], [1], fmt=0)
    assert st == d["EF_OK"]                                   # one segment of 2^31
    st, _ = _ws_size(lib, (1 << 31) + 1, [0, (1 << 31) + 1], [1], fmt=1)
    assert st == d["EF_ERR_SIZE"]                             # one segment > 2^31


def test_topk_workspace_sizes_of_the_workloads(lib):
    """What the header and the design state about workspace sizes: the
    allocation-free entry point's scratch holds a BERT-large-sized flat
    tensor at top-0.1 % and the layerwise ResNet-50 call, the 2^31 tensor's
    workspace is about 76 MB, and the size never shrinks as k grows (the
    candidate list's capacity is min(len, 4k + 65 536) per segment)."""
    from error_feedback_gradient_gb300 import workloads as wl
    d = _header_defines()
    cap = d["EF_NOALLOC_SCRATCH_BYTES"]
    n = 335_141_888
    for fmt in (0, 1):
        st, b = _ws_size(lib, n, [0, n], [wl.k_from_ratio(n, 1, 1000)], fmt)
        assert st == d["EF_OK"] and b <= cap
    offs, ks = wl.resnet50_segments()
    st, b = _ws_size(lib, offs[-1], offs, ks)
    assert st == d["EF_OK"] and b <= cap
    n = 1 << 31
    st, b = _ws_size(lib, n, [0, n], [wl.k_from_ratio(n, 1, 1000)])
    assert st == d["EF_OK"] and 70e6 < b < 80e6
    n = 1 << 24
    sizes = [_ws_size(lib, n, [0, n], [k])[1] for k in (0, 1, 100, 10**4, 10**6, n // 4, n)]
    assert sizes == sorted(sizes) and sizes[-1] > n * 8     # a list of every element fits


def test_topk_rejects_before_device(lib):
    d = _header_defines()
    ws = ctypes.c_void_p(256 * 1000)           # never dereferenced: validation fails first
    fake = ctypes.c_void_p(4096)
    st = lib.ef_topk_compress(fake, ctypes.c_void_p(8192), 100, 1, _i64([0, 100]), _i64([101]),
                              0, fake, fake, None, ws, 1 << 20, None)
    assert st == d["EF_ERR_K"]
    st = lib.ef_topk_compress(fake, ctypes.c_void_p(8192), 100, 1, _i64([0, 100]), _i64([5]),
                              0, fake, fake, None, None, 0, None)
    assert st == d["EF_ERR_WORKSPACE"]
    st = lib.ef_topk_compress(fake, ctypes.c_void_p(8192), 100, 1, _i64([0, 100]), _i64([5]),
                              0, fake, fake, None, ctypes.c_void_p(255), 1 << 20, None)
    assert st == d["EF_ERR_WORKSPACE"]                        # misaligned
    st = lib.ef_topk_compress(fake, fake, 100, 1, _i64([0, 100]), _i64([5]),
                              0, ctypes.c_void_p(1 << 20), ctypes.c_void_p(2 << 20), None, ws,
                              1 << 20, None)
    assert st == d["EF_ERR_ALIAS"]                            # g_raw == e
    st = lib.ef_topk_compress(ctypes.c_void_p(4098), ctypes.c_void_p(1 << 20), 100, 1,
                              _i64([0, 100]), _i64([5]), 0, ctypes.c_void_p(2 << 20),
                              ctypes.c_void_p(3 << 20), None, ws, 1 << 20, None)
    assert st == d["EF_ERR_ALIGN"]
    st = lib.ef_topk_compress(fake, ctypes.c_void_p(1 << 20), 100, 1, _i64([0, 100]),
                              _i64([5]), 0, None, ctypes.c_void_p(3 << 20), None, ws, 1 << 20,
                              None)
    assert st == d["EF_ERR_NULL"]


def test_sign_rejects_before_device(lib):
    d = _header_defines()
    a, b, c = ctypes.c_void_p(1 << 20), ctypes.c_void_p(2 << 20), ctypes.c_void_p(3 << 20)
    assert lib.ef_sign_compress(a, b, -1, 0.9, c, None) == d["EF_ERR_SIZE"]
    assert lib.ef_sign_compress(a, b, 10, float("nan"), c, None) == d["EF_ERR_ARG"]
    assert lib.ef_sign_compress(a, a, 10, 0.9, c, None) == d["EF_ERR_ALIAS"]
    assert lib.ef_sign_compress(None, b, 10, 0.9, c, None) == d["EF_ERR_NULL"]
    assert lib.ef_sign_compress(a, b, 0, 0.9, c, None) == d["EF_OK"]      # empty: no work
    bits = (ctypes.c_void_p * 1)(c)
    assert lib.sign_aggregate_apply(0, bits, 10, 0, 0.1, 0.9, None, a, None) == d["EF_ERR_WORKERS"]
    assert lib.sign_aggregate_apply(1, bits, 10, 5, 0.1, 0.9, None, a, None) == d["EF_ERR_ARG"]
    assert lib.sign_aggregate_apply(1, bits, 10, 0, float("inf"), 0.9, None, a,
                                    None) == d["EF_ERR_ARG"]


def test_aggregate_rejects_before_device(lib):
    d = _header_defines()
    out = ctypes.c_size_t(0)
    assert lib.ef_aggregate_workspace_size(0, 0, 10, ctypes.byref(out)) == d["EF_ERR_WORKERS"]
    assert lib.ef_aggregate_workspace_size(65, 0, 10, ctypes.byref(out)) == d["EF_ERR_WORKERS"]
    assert lib.ef_aggregate_workspace_size(8, 1, 1 << 20, ctypes.byref(out)) == d["EF_OK"]
    vals = (ctypes.c_void_p * 1)(ctypes.c_void_p(1 << 20))
    inds = (ctypes.c_void_p * 1)(ctypes.c_void_p(2 << 20))
    ws = ctypes.c_void_p(256 * 4096)
    w = ctypes.c_void_p(3 << 20)
    st = lib.sparse_aggregate_apply(1, 0, vals, inds, None, _i64([11]), 10, 0.1, None, w, ws,
                                    1 << 20, None)
    assert st == d["EF_ERR_K"]
    st = lib.sparse_aggregate_apply(1, 0, vals, None, None, _i64([1]), 10, 0.1, None, w, ws,
                                    1 << 20, None)
    assert st == d["EF_ERR_NULL"]
    st = lib.sparse_aggregate_apply(1, 0, vals, inds, None, _i64([1]), 10, 0.1, None, w, ws,
                                    8, None)
    assert st == d["EF_ERR_WORKSPACE"]
    st = lib.sparse_aggregate_apply(1, 0, vals, inds, None, _i64([1]), 10, 0.1, w, w, ws,
                                    1 << 20, None)
    assert st == d["EF_ERR_ALIAS"]


def _randk_ws(lib, n, offs, ks):
    out = ctypes.c_size_t(0)
    st = lib.ef_randk_workspace_size(n, len(ks), _i64(offs), _i64(ks), ctypes.byref(out))
    return st, out.value


def test_randk_workspace_and_rejects_before_device(lib):
    d = _header_defines()
    st, small = _randk_ws(lib, 1000, [0, 1000], [10])
    assert st == d["EF_OK"] and small >= 256
    st, big = _randk_ws(lib, 1 << 31, [0, 1 << 31], [1 << 21])
    assert st == d["EF_OK"] and big >= (1 << 31) // 8          # keep bits: n / 8 bytes
    assert _randk_ws(lib, 100, [0, 50, 100], [51, 1])[0] == d["EF_ERR_K"]
    assert _randk_ws(lib, 100, [0, 60, 50, 100], [1, 1, 1])[0] == d["EF_ERR_SEGMENTS"]
    assert _randk_ws(lib, (1 << 31) + 4, [0, (1 << 31) + 4], [1])[0] == d["EF_ERR_SIZE"]
    n, offs, ks = 1000, [0, 1000], [10]
    _, wsb = _randk_ws(lib, n, offs, ks)
    g, e = ctypes.c_void_p(1 << 20), ctypes.c_void_p(2 << 20)
    vals, idx = ctypes.c_void_p(3 << 20), ctypes.c_void_p(4 << 20)
    cnt, ws = ctypes.c_void_p(5 << 20), ctypes.c_void_p(6 << 20)

    def call(g=g, e=e, ks=ks, vals=vals, idx=idx, cap=100, cnt=cnt, ws=ws, wsb=wsb):
        return lib.ef_randk_compress(g, e, n, len(ks), _i64(offs), _i64(ks), 1, 0, vals, idx,
                                     cap, cnt, ws, wsb, None)
    assert call(ks=[1001]) == d["EF_ERR_K"]
    assert call(ws=None) == d["EF_ERR_WORKSPACE"]
    assert call(ws=ctypes.c_void_p((6 << 20) + 128)) == d["EF_ERR_WORKSPACE"]   # misaligned
    assert call(wsb=wsb - 1) == d["EF_ERR_WORKSPACE"]
    assert call(cap=-1) == d["EF_ERR_ARG"]
    assert call(cnt=None) == d["EF_ERR_NULL"]
    assert call(vals=None) == d["EF_ERR_NULL"]
    assert call(cnt=ctypes.c_void_p((5 << 20) + 4)) == d["EF_ERR_ALIGN"]
    assert call(e=g) == d["EF_ERR_ALIAS"]
    assert call(idx=ctypes.c_void_p((3 << 20) + 8)) == d["EF_ERR_ALIAS"]  # inside the values


def _codec_sizes(lib, codec, K, n):
    mb, wb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    st = lib.ef_index_codec_sizes(codec, K, n, ctypes.byref(mb), ctypes.byref(wb))
    return st, mb.value, wb.value


def test_codec_sizes_follow_the_header(lib):
    d = _header_defines()
    for K, n in [(0, 1), (1, 1), (1000, 100_000), (2_147_484, 1 << 31)]:
        nblk = -(-n // 65536)
        nfw = -(-(-(-n // 256)) // 32)
        st, mb, wb = _codec_sizes(lib, d["EF_CODEC_LOCAL16"], K, n)
        assert st == d["EF_OK"] and mb == 4 * (nblk + 1) + 2 * K and wb >= 256
        st, mb, _ = _codec_sizes(lib, d["EF_CODEC_RUNVARINT"], K, n)
        assert st == d["EF_OK"] and mb == 5 * K
        st, mb, _ = _codec_sizes(lib, d["EF_CODEC_BLOCK256"], K, n)
        assert st == d["EF_OK"] and mb == 4 * nfw + 2 * K
    assert _codec_sizes(lib, 9, 10, 100)[0] == d["EF_ERR_ARG"]
    assert _codec_sizes(lib, d["EF_CODEC_LOCAL16"], 101, 100)[0] == d["EF_ERR_K"]
    assert _codec_sizes(lib, d["EF_CODEC_LOCAL16"], 1, (1 << 31) + 1)[0] == d["EF_ERR_SIZE"]


def test_codec_rejects_before_device(lib):
    d = _header_defines()
    K, n = 100, 100_000
    idx, out = ctypes.c_void_p(1 << 20), ctypes.c_void_p(2 << 20)
    ob, ws = ctypes.c_void_p(3 << 20), ctypes.c_void_p(4 << 20)
    for codec in (d["EF_CODEC_LOCAL16"], d["EF_CODEC_RUNVARINT"], d["EF_CODEC_BLOCK256"]):
        _, mb, wb = _codec_sizes(lib, codec, K, n)
        enc = lambda **kw: lib.ef_index_encode(  # noqa: E731
            codec, kw.get("idx", idx), K, n, out, kw.get("cap", mb), kw.get("ob", ob),
            kw.get("ws", ws), wb, None)
        assert enc(ws=None) == d["EF_ERR_WORKSPACE"]
        assert enc(idx=None) == d["EF_ERR_NULL"]
        assert enc(cap=mb - 1) == d["EF_ERR_SIZE"]
        assert enc(ob=ctypes.c_void_p((3 << 20) + 4)) == d["EF_ERR_ALIGN"]
        assert enc(idx=ctypes.c_void_p((2 << 20) + 16)) == d["EF_ERR_ALIAS"]   # inside out
        assert lib.ef_index_decode(codec, out, mb, K, n, None, ws, wb, None) == d["EF_ERR_NULL"]
    # lengths the formats cannot have
    _, mb, wb = _codec_sizes(lib, d["EF_CODEC_LOCAL16"], K, n)
    assert lib.ef_index_decode(d["EF_CODEC_LOCAL16"], out, mb - 2, K, n, idx, ws, wb,
                               None) == d["EF_ERR_PACKET"]
    _, mb, wb = _codec_sizes(lib, d["EF_CODEC_RUNVARINT"], K, n)
    assert lib.ef_index_decode(d["EF_CODEC_RUNVARINT"], out, K - 1, K, n, idx, ws, wb,
                               None) == d["EF_ERR_PACKET"]
    _, mb, wb = _codec_sizes(lib, d["EF_CODEC_BLOCK256"], K, n)
    nfw = -(-(-(-n // 256)) // 32)
    assert lib.ef_index_decode(d["EF_CODEC_BLOCK256"], out, 4 * nfw + K, K, n, idx, ws, wb,
                               None) == d["EF_ERR_PACKET"]      # no flagged block counts


def test_q8_rejects_before_device(lib):
    d = _header_defines()
    out = ctypes.c_size_t(0)
    assert lib.ef_topk_q8_workspace_size(1000, 1, _i64([0, 1000]), _i64([10]), 0,
                                         ctypes.byref(out)) == d["EF_OK"]
    wsb = out.value
    assert wsb >= 256
    assert lib.ef_topk_q8_workspace_size(1000, 1, _i64([0, 1000]), _i64([1001]), 0,
                                         ctypes.byref(out)) == d["EF_ERR_K"]
    g, e = ctypes.c_void_p(1 << 20), ctypes.c_void_p(2 << 20)
    q, sc, idx = ctypes.c_void_p(3 << 20), ctypes.c_void_p(4 << 20), ctypes.c_void_p(5 << 20)
    ws = ctypes.c_void_p(6 << 20)

    def call(q=q, sc=sc, ws=ws):
        return lib.ef_topk_compress_q8(g, e, 1000, 1, _i64([0, 1000]), _i64([10]), 0, q, sc,
                                       idx, None, ws, wsb, None)
    assert call(ws=None) == d["EF_ERR_WORKSPACE"]
    assert call(sc=None) == d["EF_ERR_NULL"]
    assert call(q=None) == d["EF_ERR_NULL"]
    assert call(sc=ctypes.c_void_p((4 << 20) + 2)) == d["EF_ERR_ALIGN"]
    assert call(sc=ctypes.c_void_p((3 << 20) + 4)) == d["EF_ERR_ALIAS"]      # inside the codes
    vals = ctypes.c_void_p(7 << 20)
    assert lib.ef_q8_dequantize(q, sc, 0, _i64([1]), vals, None) == d["EF_ERR_SEGMENTS"]
    assert lib.ef_q8_dequantize(q, sc, 1, _i64([-1]), vals, None) == d["EF_ERR_K"]
    assert lib.ef_q8_dequantize(None, None, 1, _i64([0]), None, None) == d["EF_OK"]  # nothing
    assert lib.ef_q8_dequantize(None, sc, 1, _i64([4]), vals, None) == d["EF_ERR_NULL"]
    assert lib.ef_q8_dequantize(q, ctypes.c_void_p((4 << 20) + 1), 1, _i64([4]), vals,
                                None) == d["EF_ERR_ALIGN"]


def test_exchange_steps_reject_before_device(lib):
    d = _header_defines()
    idx, starts = ctypes.c_void_p(4096), ctypes.c_void_p(1 << 20)
    split = lib.ef_packet_split
    assert split(idx, -1, 2, _i64([0, 5, 9]), starts, None) == d["EF_ERR_SIZE"]
    assert split(idx, (1 << 31) + 1, 2, _i64([0, 5, 9]), starts, None) == d["EF_ERR_SIZE"]
    assert split(idx, 10, 0, _i64([0]), starts, None) == d["EF_ERR_ARG"]
    assert split(idx, 10, 1025, _i64(range(1026)), starts, None) == d["EF_ERR_ARG"]
    assert split(idx, 10, 2, _i64([0, 9, 5]), starts, None) == d["EF_ERR_SEGMENTS"]
    assert split(None, 10, 2, _i64([0, 5, 9]), starts, None) == d["EF_ERR_NULL"]
    assert split(idx, 10, 2, None, starts, None) == d["EF_ERR_NULL"]
    assert split(idx, 10, 2, _i64([0, 5, 9]), None, None) == d["EF_ERR_NULL"]
    assert split(ctypes.c_void_p(4098), 10, 2, _i64([0, 5, 9]), starts, None) == d["EF_ERR_ALIGN"]
    assert split(idx, 10, 2, _i64([0, 5, 9]), ctypes.c_void_p((1 << 20) + 4),
                 None) == d["EF_ERR_ALIGN"]
    assert split(idx, 10, 2, _i64([0, 5, 9]), ctypes.c_void_p(4096 + 16),
                 None) == d["EF_ERR_ALIAS"]
    rebase = lib.ef_index_rebase
    assert rebase(idx, -1, 0, None) == d["EF_ERR_SIZE"]
    assert rebase(idx, 10, -1, None) == d["EF_ERR_ARG"]
    assert rebase(None, 10, 0, None) == d["EF_ERR_NULL"]
    assert rebase(ctypes.c_void_p(4098), 10, 0, None) == d["EF_ERR_ALIGN"]
    assert rebase(None, 0, 5, None) == d["EF_OK"]                     # empty: no work
