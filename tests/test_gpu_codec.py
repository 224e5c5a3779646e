"""GPU parity of the index codecs (ef_index_encode / ef_index_decode) against
the oracle: the encoded byte streams and the decoded indices bit for bit,
malformed inputs reported without out-of-bounds access."""

import numpy as np
import pytest
import torch

import error_feedback_gradient_gb300 as efg
from error_feedback_gradient_gb300 import workloads as wl
from efcheck import gpu_topk, host
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"
CODECS = {efg.CODEC_LOCAL16: (oracle.encode_local16, oracle.decode_local16),
          efg.CODEC_RUNVARINT: (oracle.encode_runvarint, oracle.decode_runvarint),
          efg.CODEC_BLOCK256: (oracle.encode_block256, oracle.decode_block256)}


def _encode(codec, idx_np, n):
    K = idx_np.size
    mb, wb = efg.index_codec_sizes(codec, K, n)
    idx = torch.from_numpy(idx_np.astype(np.int32)).to(DEV)
    out = torch.full(((max(mb, 4) + 3) // 4,), -1, dtype=torch.int32, device=DEV)   # 4-byte aligned
    ob = torch.zeros(1, dtype=torch.int64, device=DEV)
    ws = torch.empty(wb, dtype=torch.uint8, device=DEV)
    efg.index_encode(codec, idx, n, out, ob, ws)
    torch.cuda.synchronize()
    nbytes = int(ob.item())
    return host(out).view(np.uint8)[:nbytes].copy(), efg.workspace_status(ws), nbytes, mb


def _decode(codec, stream_np, K, n):
    mb, wb = efg.index_codec_sizes(codec, K, n)
    buf = np.zeros(((stream_np.size + 3) // 4) * 4, np.uint8)
    buf[:stream_np.size] = stream_np
    st = torch.from_numpy(buf.view(np.int32)).to(DEV)
    out = torch.full((K,), -7, dtype=torch.int32, device=DEV)
    ws = torch.empty(wb, dtype=torch.uint8, device=DEV)
    efg.index_decode(codec, st, stream_np.size, K, n, out, ws)
    torch.cuda.synchronize()
    return host(out), efg.workspace_status(ws)


def _roundtrip(codec, idx, n):
    enc, dec = CODECS[codec]
    want = enc(idx, n)
    got, status, nbytes, mb = _encode(codec, idx, n)
    assert status == 0
    assert nbytes == want.size <= mb
    assert np.array_equal(got, want), f"codec {codec}: stream differs"
    back, status = _decode(codec, want, idx.size, n)
    assert status == 0
    assert np.array_equal(back.astype(np.int64), idx.astype(np.int64))


def _sets():
    rng = np.random.default_rng(31)
    yield np.zeros(0, np.int64), 1000
    yield np.array([0], np.int64), 1
    yield np.array([999], np.int64), 1000
    yield np.arange(70_001, dtype=np.int64), 70_001              # every element
    for n, k in [(5000, 50), (1_000_003, 10_000), (4_000_037, 400_000), (200_000, 150_000)]:
        yield np.sort(rng.choice(n, k, replace=False)).astype(np.int64), n
    # runs of neighbours, long gaps (multi-byte runs), several chunks
    n = 30_000_000
    starts = np.sort(rng.choice(n - 400, 3000, replace=False))
    yield np.unique(np.concatenate([s + np.arange(int(rng.integers(1, 400))) for s in starts])), n


@pytest.mark.parametrize("codec", list(CODECS))
def test_codec_matches_oracle(codec):
    for idx, n in _sets():
        _roundtrip(codec, idx, n)


@pytest.mark.parametrize("codec", list(CODECS))
def test_codec_on_a_topk_packet(codec):
    """The codecs applied to a real top-k packet of a 2^24-element tensor."""
    n, k = 1 << 24, 16_777
    out = gpu_topk(wl.student_t3(n, 1e-3, 3, DEV), torch.zeros(n, device=DEV), [0, n], [k])
    idx = host(out["indices"]).astype(np.int64)
    _roundtrip(codec, idx, n)


def test_codec_top_index_range():
    """Indices up to 2^31 - 1 (the largest int32 packet): long first run,
    the last 65536-block and the last 256-block."""
    n = 1 << 31
    idx = np.array([5, 70_000_000, n - 300, n - 2, n - 1], np.int64)
    for codec in CODECS:
        _roundtrip(codec, idx, n)


def test_codec_sizes_and_compression():
    """Stream bounds from ef_index_codec_sizes and the sizes the formats give
    on a top-0.1 % packet (4 bytes per index in int32 form)."""
    n, k = 1 << 26, 67_109
    idx = np.sort(np.random.default_rng(4).choice(n, k, replace=False)).astype(np.int64)
    sizes = {c: _encode(c, idx, n)[2] for c in CODECS}
    assert sizes[efg.CODEC_LOCAL16] == 4 * (1024 + 1) + 2 * k
    assert sizes[efg.CODEC_BLOCK256] == 4 * 8192 + np.unique(idx // 256).size + k
    assert sizes[efg.CODEC_RUNVARINT] < 2 * k            # mean gap 1000: two bytes each
    assert all(s < 4 * k for s in sizes.values())


@pytest.mark.parametrize("codec", list(CODECS))
def test_codec_rejects_unsorted_input(codec):
    n = 10_000
    idx = torch.tensor([5, 100, 50, 7000], dtype=torch.int32, device=DEV)
    mb, wb = efg.index_codec_sizes(codec, 4, n)
    out = torch.empty((mb + 3) // 4, dtype=torch.int32, device=DEV)
    ob = torch.zeros(1, dtype=torch.int64, device=DEV)
    ws = torch.empty(wb, dtype=torch.uint8, device=DEV)
    efg.index_encode(codec, idx, n, out, ob, ws)
    assert efg.workspace_status(ws) == 13                # EF_ERR_PACKET


@pytest.mark.parametrize("codec", list(CODECS))
def test_codec_malformed_streams_are_reported(codec):
    """Corrupted streams decode to EF_ERR_PACKET (or are refused by length)
    and never touch memory outside their buffers."""
    n, K = 50_000, 40
    idx = np.sort(np.random.default_rng(6).choice(n, K, replace=False)).astype(np.int64)
    good = CODECS[codec][0](idx, n)
    bad = []
    if codec == efg.CODEC_LOCAL16:
        b = good.copy()
        b[4:8] = 255                                     # a block start far past K
        bad.append(b)
    elif codec == efg.CODEC_RUNVARINT:
        bad.append(np.concatenate([good[:-1], [0x80]]).astype(np.uint8))   # unterminated
        bad.append(np.full(good.size, 0xFF, np.uint8))  # no terminator at all
        bad.append(np.concatenate([good, [1]]).astype(np.uint8))           # K+1 entries
    else:
        b = good.copy()
        b[:4] = 0xFF                                     # more flagged blocks than counts
        bad.append(b)
        b = good.copy()
        nfw = -(-(-(-n // 256)) // 32)
        b[4 * nfw] = 200                                 # first block claims 201 entries
        bad.append(b)
    for b in bad:
        try:
            _, status = _decode(codec, b, K, n)
        except efg.EFError as ex:
            assert ex.status == 13
            continue
        assert status == 13
