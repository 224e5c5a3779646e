"""Plain CPU oracle for error-feedback gradient compression.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import this module.  The CUDA library and its Python binding
never import it, and it imports nothing from them: the two sides share no
code, no helpers and no constants.  Inputs reach both sides from the seeded
generators in ``error_feedback_gradient_gb300/workloads.py``, which hold none
of the arithmetic below.

Sources (web pages, cited by title and section):

* [SPARSE] "梯度稀疏化：只传输重要的梯度元素" ("Gradient sparsification:
  transmit only the important gradient elements"), freeguideonline.com
  tutorial.  Sections used: 梯度稀疏化的基本原理 (basic principle: select the
  k largest |g|, send values + indices, the receiver sums by index);
  必不可少的误差补偿 (error compensation); Top-k 稀疏化; 分层阈值与自适应稀疏率
  and 分层自适应Top-k (each tensor selects independently); 详细算法流程
  (the seven-step algorithm: steps 2-7); 索引编码压缩 (bitmap index);
  与其他压缩技术的比较 (top-k followed by 8-bit quantisation of the selected
  values).
* [ONEBIT] "1bit Adam梯度压缩技术原理与分布式训练优化" ("1-bit Adam gradient
  compression: principle and distributed-training optimisation"),
  intelliparadigm.com article.  Sections used: 2.1 量化与误差补偿机制 (sign
  quantisation, quantisation error, EMA error buffer); 2.2 动量修正策略
  (momentum on the quantised gradient).

Precision.  Both pages work with FP32 gradients ([ONEBIT] §1 assumes FP32,
[SPARSE] §为什么要做梯度压缩 counts 32-bit floats), so every array here is
float32 and every arithmetic operation is a single IEEE-754 float32 operation
rounded to nearest-even.  numpy evaluates each ufunc separately, so no
multiply-add is ever fused; the operation order written in each function is
the order used.

Readings taken where the pages are silent (each repeated where it is used):

* ties in |g| go to the lower index, and |g| is compared as the IEEE bit
  pattern with the sign bit cleared (so +0 ties -0); every NaN ranks above
  +Inf and all NaNs tie whatever their payload (NaN payload bits are not
  part of any result: two NaNs compare equal);
* a packet lists its entries in ascending index order, with global int32
  indices into the flat buffer (or, in bitmap form, one bit per element,
  element i at bit i % 32 of word i // 32, padding bits 0);
* the residual at a selected position is +0.0;
* sign(0) = +1 (also for -0 and NaN): a bit is 1 unless v < 0;
* the receiver adds packets in worker order 0..W-1 starting from +0.0 and
  does not average;
* (1 - beta1) is formed in float32 before it multiplies;
* index codecs (the pages name the ideas, not the formats): a packet's
  ascending int32 index list becomes one byte stream, little-endian --
  LOCAL16: uint32 block_start[nblk + 1] (entries before each 65536-element
  block) then each index's uint16 offset in its block; RUNVARINT: for each
  index the number of unselected elements since the previous one (the first
  counts from element 0), as LEB128 (7 bits per byte, low group first, high
  bit set when more bytes follow); BLOCK256: one bit per 256-element block
  (bit b % 32 of word b // 32, set when the block holds an index), then for
  each such block in order its entry count - 1 as uint8, then each index's
  uint8 offset in its block;
* random magnitude-proportional sparsification ([SPARSE] §随机稀疏化): keep
  element i with probability p_i = min(1, c |g_i|), c = k / S, S = the
  exact sum of |g| over the segment's finite elements rounded once to
  float64 (the pages normalise once so that the p_i add up to k; where
  c |g_i| > 1 the element is kept surely, so the expected count falls short
  of k by the clipped excess).  The per-element arithmetic is float32, the
  gradients' precision: c is rounded to float32 once, p_i = min(1,
  RN(c |g_i|)), and the draw u_i = (w >> 8) / 2^24 (exact in float32) with
  w word i % 4 of Philox4x32-10 (counter (i // 4 low, high word, step low,
  high word), key (seed low, high word)); kept iff u_i < p_i.  Non-finite
  elements are kept surely; S = 0 keeps nothing; kept values are sent as
  they are (no 1/p scaling: the residual carries the rest), in ascending
  index order, and a packet stops at its capacity (later kept elements
  stay in the residual);
* 8-bit quantisation of a packet's values (the pages give no formula): one
  float32 scale per segment, s = max |v| / 127 over the segment's finite
  selected values (0 if none); q = round-half-even(v / s) clamped to
  [-127, 127], q = 0 for NaN and whenever s = 0; the receiver's value is
  q * s, and the residual at a selected position is v - q * s, so the error
  feedback also carries the quantisation error.

Parity pins for every function live in ``tests/test_oracle_pins.py``; no
function here is parity-unpinned.
"""

from __future__ import annotations

import numpy as np

F32 = np.float32
U32 = np.uint32
U64 = np.uint64

# --------------------------------------------------------------------------
# small helpers (bit layout, ordering key)
# --------------------------------------------------------------------------


def abs_key(g: np.ndarray) -> np.ndarray:
    """Ordering key for |g|: the float32 bit pattern with the sign bit cleared.

    For non-NaN values this uint32 is monotone in |g| ([SPARSE] §Top-k 稀疏化
    ranks elements by absolute value).  Every NaN gets the largest key,
    0x7FFFFFFF, so NaNs rank above +Inf and tie with each other.
    """
    g = np.ascontiguousarray(g, dtype=F32)
    key = g.view(U32) & U32(0x7FFFFFFF)
    key[np.isnan(g)] = U32(0x7FFFFFFF)
    return key


def pack_bits(flags: np.ndarray) -> np.ndarray:
    """Pack a boolean vector 32 to a uint32 word, element i -> bit i % 32 of
    word i // 32 (least significant bit first), padding bits 0."""
    flags = np.asarray(flags, dtype=bool).ravel()
    n = flags.size
    nw = (n + 31) // 32
    padded = np.zeros(nw * 32, dtype=bool)
    padded[:n] = flags
    cols = padded.reshape(nw, 32)
    words = np.zeros(nw, dtype=U32)
    for j in range(32):
        words |= cols[:, j].astype(U32) << U32(j)
    return words


def unpack_bits(words: np.ndarray, n: int) -> np.ndarray:
    """Inverse of :func:`pack_bits` for the first ``n`` elements."""
    words = np.asarray(words, dtype=U32).ravel()
    nw = (n + 31) // 32
    if words.size < nw:
        raise ValueError("bit vector too short")
    out = np.zeros((nw, 32), dtype=bool)
    for j in range(32):
        out[:, j] = ((words[:nw] >> U32(j)) & U32(1)).astype(bool)
    return out.ravel()[:n]


# --------------------------------------------------------------------------
# top-k error feedback  ([SPARSE] 详细算法流程, steps 2-5)
# --------------------------------------------------------------------------


def compensate(g_raw: np.ndarray, e: np.ndarray) -> np.ndarray:
    """Step 2: g = g_raw + e (the carried residual is added back).

    [SPARSE] §必不可少的误差补偿 and §详细算法流程 step 2; e starts at 0.
    """
    return np.add(np.asarray(g_raw, F32), np.asarray(e, F32), dtype=F32)


def topk_indices(g: np.ndarray, k: int) -> np.ndarray:
    """Step 3: the k elements of largest |g|, returned in ascending index order.

    [SPARSE] §梯度稀疏化的基本原理 step 2 and §Top-k 稀疏化: keep the k
    entries of largest absolute value, zero the rest.  The pages do not say
    which entry wins a tie; the lower index does.

    The selection is the plain definition: order every element by
    (|g| descending, index ascending) and keep the first k.  That order is
    encoded in one unsigned 64-bit number per element,
    ``abs_key << 32 | (2**32 - 1 - index)``, whose descending order is exactly
    the order above (a larger key wins; for equal keys the lower index has the
    larger low word).  numpy's partition (a library selection routine) then
    puts the k largest of those numbers last; their low words give back the
    indices.  Requires len(g) < 2**32.
    """
    g = np.ascontiguousarray(g, dtype=F32)
    n = g.size
    if k < 0 or k > n:
        raise ValueError(f"k={k} outside [0, {n}]")
    if k == 0:
        return np.zeros(0, dtype=np.int64)
    if n >= 2**32:
        raise ValueError("segment too long for the 64-bit rank encoding")
    rank = abs_key(g).astype(U64) << U64(32)
    rank |= U64(0xFFFFFFFF) - np.arange(n, dtype=U64)
    rank.partition(n - k)
    top = rank[n - k:]
    idx = (U64(0xFFFFFFFF) - (top & U64(0xFFFFFFFF))).astype(np.int64)
    idx.sort()
    return idx


def topk_ef_step(g_raw, e, seg_offsets, seg_k, idx_format: str = "int32"):
    """One layerwise top-k error-feedback step over a flat fp32 buffer.

    [SPARSE] §详细算法流程 steps 2-5, applied independently to every segment
    (tensor) as §分层阈值与自适应稀疏率 / §分层自适应Top-k prescribe:

    2. g = g_raw + e_prev
    3. g~ keeps the k_s largest |g| of segment s, zero elsewhere
    4. e = g - g~  (= g off the selection, +0.0 on it)
    5. pack the non-zeros of g~ with their indices

    ``seg_offsets`` has nseg+1 entries (0 ... n); ``seg_k`` has nseg.
    Packets list segment 0's entries first, each segment in ascending index
    order, so the whole packet is in ascending global index order.

    Returns a dict with ``values`` (float32[sum k]), ``indices`` (int32
    global indices, only for ``idx_format == "int32"``), ``bitmap``
    (uint32[ceil(n/32)], only for ``"bitmap"``), ``e`` (the new residual,
    float32[n]) and ``selected`` (the global indices as int64, for callers
    inside the oracle).
    """
    g_raw = np.ascontiguousarray(g_raw, dtype=F32)
    e_prev = np.ascontiguousarray(e, dtype=F32)
    n = g_raw.size
    if e_prev.size != n:
        raise ValueError("g_raw and e differ in length")
    offs = [int(x) for x in seg_offsets]
    ks = [int(x) for x in seg_k]
    if len(offs) != len(ks) + 1 or offs[0] != 0 or offs[-1] != n:
        raise ValueError("segment table does not span [0, n)")

    g = compensate(g_raw, e_prev)                         # step 2
    e_new = g.copy()                                      # step 4 off the selection
    picked = []
    for s, k in enumerate(ks):
        a, b = offs[s], offs[s + 1]
        if b < a:
            raise ValueError("segment offsets must not decrease")
        picked.append(topk_indices(g[a:b], k) + a)        # step 3
    sel = np.concatenate(picked) if picked else np.zeros(0, np.int64)
    values = g[sel].copy()                                # step 5 (values)
    e_new[sel] = F32(0.0)                                 # step 4 on the selection
    out = {"values": values, "e": e_new, "selected": sel}
    if idx_format == "int32":
        if n > 2**31:
            raise ValueError("int32 indices need n <= 2**31")
        out["indices"] = sel.astype(np.int32)
    elif idx_format == "bitmap":
        flags = np.zeros(n, dtype=bool)
        flags[sel] = True
        out["bitmap"] = pack_bits(flags)
    else:
        raise ValueError(idx_format)
    return out


# --------------------------------------------------------------------------
# 8-bit quantisation of the selected values  ([SPARSE] §与其他压缩技术的比较)
# --------------------------------------------------------------------------

Q8_LEVELS = 127


def q8_scale(values) -> np.float32:
    """Scale of one segment's packet: s = max |v| / 127 in float32.

    [SPARSE] §与其他压缩技术的比较 quantises the top-k values to 8 bits after
    the selection and gives no formula; the reading here is symmetric int8
    with one scale per segment (tensor).  Only finite values count towards
    the maximum; with none (or an empty segment) s = 0.
    """
    v = np.asarray(values, dtype=F32)
    fin = v[np.isfinite(v)]
    m = np.max(np.abs(fin)) if fin.size else F32(0.0)
    return np.divide(F32(m), F32(Q8_LEVELS), dtype=F32)


def q8_quantize(values, s) -> np.ndarray:
    """q = round-half-even(v / s) clamped to [-127, 127], as int8.

    v / s is one float32 division; q = 0 for NaN values and for every value
    when s = 0; +-Inf clamps to +-127.
    """
    v = np.asarray(values, dtype=F32)
    s = F32(s)
    q = np.zeros(v.size, dtype=np.int8)
    if s == F32(0.0):
        return q
    ok = ~np.isnan(v)
    with np.errstate(over="ignore", invalid="ignore"):
        t = np.divide(v[ok], s, dtype=F32)
    t = np.minimum(np.maximum(t, F32(-Q8_LEVELS)), F32(Q8_LEVELS))
    q[ok] = np.rint(t).astype(np.int8)
    return q


def q8_dequantize(q, s) -> np.ndarray:
    """The receiver's value of each entry: q * s, one float32 multiply."""
    return np.multiply(np.asarray(q, dtype=np.int8).astype(F32), F32(s), dtype=F32)


def topk_q8_ef_step(g_raw, e, seg_offsets, seg_k, idx_format: str = "int32"):
    """A top-k error-feedback step whose packet values are 8-bit quantised.

    [SPARSE] §详细算法流程 steps 2-5 (topk_ef_step) followed by the 8-bit
    quantisation of §与其他压缩技术的比较, per segment: s = q8_scale of the
    segment's selected values, q = q8_quantize(v, s).  What the packet
    carries at a selected position is q * s, so step 4's residual
    e = g - g~ becomes v - q * s there (one float32 subtraction) and stays g
    elsewhere.

    Returns the topk_ef_step dict with ``q`` (int8[sum k]), ``scales``
    (float32[nseg]) and ``e`` replaced by this residual; ``values`` keeps the
    unquantised selected values.
    """
    out = topk_ef_step(g_raw, e, seg_offsets, seg_k, idx_format)
    ks = [int(x) for x in seg_k]
    v = out["values"]
    sel = out["selected"]
    e_new = out["e"]
    q = np.zeros(v.size, dtype=np.int8)
    scales = np.zeros(len(ks), dtype=F32)
    j = 0
    for s_i, k in enumerate(ks):
        vs = v[j:j + k]
        sc = q8_scale(vs)
        qs = q8_quantize(vs, sc)
        with np.errstate(invalid="ignore"):
            e_new[sel[j:j + k]] = np.subtract(vs, q8_dequantize(qs, sc), dtype=F32)
        q[j:j + k] = qs
        scales[s_i] = sc
        j += k
    out["q"] = q
    out["scales"] = scales
    out["e"] = e_new
    return out


# --------------------------------------------------------------------------
# index codecs  ([SPARSE] §索引编码压缩, §快速上手指南 step 4)
# --------------------------------------------------------------------------

LOCAL16_BLOCK = 65536
BLOCK256 = 256


def _check_sorted(idx, n):
    idx = np.asarray(idx, dtype=np.int64)
    if idx.size and (idx[0] < 0 or idx[-1] >= n or np.any(np.diff(idx) <= 0)):
        raise ValueError("indices must be strictly ascending and inside [0, n)")
    return idx


def encode_local16(idx, n: int) -> np.ndarray:
    """16-bit local indices ([SPARSE] §快速上手指南 step 4: indices first go to
    16-bit integers).  A 16-bit value only reaches 65536 elements, so the
    index space is cut into blocks of 65536: the stream holds
    block_start[b] = number of indices below block b, for b = 0 .. nblk
    (uint32, nblk = ceil(n / 65536)), then each index's offset inside its
    block (uint16), in packet order."""
    idx = _check_sorted(idx, n)
    nblk = (n + LOCAL16_BLOCK - 1) // LOCAL16_BLOCK
    starts = np.searchsorted(idx, np.arange(nblk + 1, dtype=np.int64) * LOCAL16_BLOCK)
    low = (idx % LOCAL16_BLOCK).astype("<u2")
    return np.concatenate([starts.astype("<u4").view(np.uint8), low.view(np.uint8)])


def decode_local16(stream, K: int, n: int) -> np.ndarray:
    nblk = (n + LOCAL16_BLOCK - 1) // LOCAL16_BLOCK
    b = np.asarray(stream, np.uint8)
    starts = b[:4 * (nblk + 1)].view("<u4").astype(np.int64)
    low = b[4 * (nblk + 1):4 * (nblk + 1) + 2 * K].view("<u2").astype(np.int64)
    blk = np.repeat(np.arange(nblk, dtype=np.int64), np.diff(starts))
    return (blk * LOCAL16_BLOCK + low).astype(np.int32)


def leb128(x: int) -> list:
    """Unsigned LEB128: 7-bit groups, least significant first, the high bit
    set on every byte but the last."""
    out = []
    while True:
        byte = x & 0x7F
        x >>= 7
        if x:
            out.append(byte | 0x80)
        else:
            out.append(byte)
            return out


def encode_runvarint(idx, n: int) -> np.ndarray:
    """Run-length / delta coding ([SPARSE] §索引编码压缩: variable-length codes
    for runs of zeros or index differences): for each index, the number of
    unselected elements since the previous index (i_j - i_{j-1} - 1, with
    i_{-1} = -1), written as LEB128."""
    idx = _check_sorted(idx, n)
    prev = -1
    out = []
    for i in idx.tolist():
        out.extend(leb128(i - prev - 1))
        prev = i
    return np.array(out, dtype=np.uint8)


def decode_runvarint(stream, K: int, n: int) -> np.ndarray:
    b = np.asarray(stream, np.uint8).tolist()
    idx, pos, prev = [], 0, -1
    for _ in range(K):
        x, shift = 0, 0
        while True:
            byte = b[pos]
            pos += 1
            x |= (byte & 0x7F) << shift
            shift += 7
            if not byte & 0x80:
                break
        prev = prev + x + 1
        idx.append(prev)
    return np.array(idx, dtype=np.int32)


def encode_block256(idx, n: int) -> np.ndarray:
    """Block-sparse index ([SPARSE] §索引编码压缩 按块稀疏): blocks of 256
    elements; a block without an index costs one flag bit, a block with
    indices also sends its entry count and each entry's offset inside it.
    Stream: uint32 flags[ceil(ceil(n / 256) / 32)] (bit b % 32 of word
    b // 32 for block b), then uint8 (count - 1) for every flagged block in
    order, then the uint8 offset of every index in packet order."""
    idx = _check_sorted(idx, n)
    nb = (n + BLOCK256 - 1) // BLOCK256
    blk = idx // BLOCK256
    flags = np.zeros(nb, dtype=bool)
    flags[blk] = True
    used, counts = np.unique(blk, return_counts=True)
    return np.concatenate([pack_bits(flags).astype("<u4").view(np.uint8),
                           (counts - 1).astype(np.uint8),
                           (idx % BLOCK256).astype(np.uint8)])


def decode_block256(stream, K: int, n: int) -> np.ndarray:
    nb = (n + BLOCK256 - 1) // BLOCK256
    nfw = (nb + 31) // 32
    b = np.asarray(stream, np.uint8)
    flags = unpack_bits(b[:4 * nfw].view("<u4"), nb)
    used = np.flatnonzero(flags)
    counts = b[4 * nfw:4 * nfw + used.size].astype(np.int64) + 1
    off = b[4 * nfw + used.size:4 * nfw + used.size + K].astype(np.int64)
    return (np.repeat(used, counts) * BLOCK256 + off).astype(np.int32)


# --------------------------------------------------------------------------
# random magnitude-proportional sparsification  ([SPARSE] §随机稀疏化)
# --------------------------------------------------------------------------

PHILOX_M = (0xD2511F53, 0xCD9E8D57)
PHILOX_W = (0x9E3779B9, 0xBB67AE85)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel
    random numbers: as easy as 1, 2, 3", SC 2011): each round multiplies
    two counter words by the constants M0, M1, mixes the high halves with
    the other two words and the key, and the key is bumped by the Weyl
    constants W0, W1 between rounds.  Works elementwise on numpy arrays of
    32-bit words (held in uint64); returns the four output words."""
    m = np.uint64(0xFFFFFFFF)
    c0, c1, c2, c3 = (np.asarray(x, np.uint64) & m for x in (c0, c1, c2, c3))
    k0, k1 = (np.asarray(x, np.uint64) & m for x in (k0, k1))
    for _ in range(10):
        p0 = np.uint64(PHILOX_M[0]) * c0
        p1 = np.uint64(PHILOX_M[1]) * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & m
        hi1, lo1 = p1 >> np.uint64(32), p1 & m
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0) & m, lo1, (hi0 ^ c3 ^ k1) & m, lo0
        k0 = (k0 + np.uint64(PHILOX_W[0])) & m
        k1 = (k1 + np.uint64(PHILOX_W[1])) & m
    return c0, c1, c2, c3


def randk_words(first: int, count: int, seed: int, step: int) -> np.ndarray:
    """The 32-bit random word of elements first .. first + count - 1: word
    i % 4 of Philox4x32-10 at counter (i // 4 low, i // 4 high, step low,
    step high) and key (seed low, seed high)."""
    i = np.arange(first, first + count, dtype=np.uint64)
    q = i >> np.uint64(2)
    out = philox4x32_10(q & np.uint64(0xFFFFFFFF), q >> np.uint64(32),
                        np.uint64(step & 0xFFFFFFFF), np.uint64(step >> 32),
                        np.uint64(seed & 0xFFFFFFFF), np.uint64(seed >> 32))
    words = np.stack(out)                       # 4 x count
    return words[(i & np.uint64(3)).astype(np.int64), np.arange(count)].astype(U32)


def randk_scale(g_segment) -> float:
    """S = sum of |g| over the finite elements, exact, rounded once to
    float64 (math.fsum returns the correctly rounded sum)."""
    import math
    a = np.abs(np.asarray(g_segment, F32))
    return math.fsum(a[np.isfinite(a)].astype(np.float64).tolist())


def randk_coefficient(g_segment, k: int) -> np.float32:
    """c = k / S (float64 division) rounded once to float32; 0 when S = 0."""
    S = randk_scale(g_segment)
    return np.float32(float(k) / S) if S > 0 else np.float32(0.0)


def randk_keep(g_segment, k: int, first: int, seed: int, step: int) -> np.ndarray:
    """Keep flags of one segment starting at global element ``first``, in
    float32: p = min(1, RN(c |g|)) (1 for non-finite elements); kept iff
    u < p with u = (randk_words >> 8) / 2^24."""
    g = np.asarray(g_segment, F32)
    c = randk_coefficient(g, k)
    a = np.abs(g)
    fin = np.isfinite(a)
    p = np.ones(g.size, F32)
    with np.errstate(over="ignore"):
        p[fin] = np.fmin(F32(1.0), np.multiply(c, a[fin], dtype=F32))   # NaN -> 1
    u = (randk_words(first, g.size, seed, step) >> U32(8)).astype(F32) * F32(2.0 ** -24)
    return u < p


def randk_ef_step(g_raw, e, seg_offsets, seg_k, seed: int, step: int, capacity: int):
    """One error-feedback step with random magnitude-proportional
    sparsification ([SPARSE] §随机稀疏化 in place of step 3 of §详细算法流程):
    g = g_raw + e; each segment keeps elements with probability
    proportional to |g| (randk_keep, expected count k_s up to clipping);
    the kept values go out unscaled with their global indices, ascending;
    e = g - g~.  A packet holds at most ``capacity`` entries: kept elements
    past it are not sent and keep g in the residual.

    Returns ``values``, ``indices`` (int32), ``e``, ``counts`` (entries sent
    per segment) and ``kept`` (elements kept before the capacity cut)."""
    g_raw = np.ascontiguousarray(g_raw, dtype=F32)
    g = compensate(g_raw, e)
    offs = [int(x) for x in seg_offsets]
    ks = [int(x) for x in seg_k]
    keep = np.zeros(g.size, bool)
    for s_i, k in enumerate(ks):
        a, b = offs[s_i], offs[s_i + 1]
        if k > 0 and b > a:
            keep[a:b] = randk_keep(g[a:b], k, a, seed, step)
    kept = np.flatnonzero(keep)
    sent = kept[:capacity]
    e_new = g.copy()
    e_new[sent] = F32(0.0)
    seg_of = np.searchsorted(np.array(offs[1:]), sent, side="right")
    counts = np.bincount(seg_of, minlength=len(ks)).astype(np.int64)
    return {"values": g[sent].copy(), "indices": sent.astype(np.int32), "e": e_new,
            "counts": counts, "kept": int(kept.size)}


# --------------------------------------------------------------------------
# 1-bit sign error feedback  ([ONEBIT] §2.1, §2.2)
# --------------------------------------------------------------------------


def sign_ef_step(g, eps, beta1: float):
    """One 1-bit error-feedback step ([ONEBIT] §2.1 量化与误差补偿机制).

    v      = g_t + eps_{t-1}
    ghat_t = sign(v)                   (+1 unless v < 0; sign(0) = +1)
    Delta  = v - ghat_t
    eps_t  = beta1 * eps_{t-1} + (1 - beta1) * Delta

    Float32 sequence: v = RN(g + eps); d = RN(v - s); c = RN(1 - beta1);
    eps' = RN(RN(beta1 * eps) + RN(c * d)).

    Returns (bits uint32[ceil(n/32)], eps' float32[n]).
    """
    g = np.ascontiguousarray(g, dtype=F32)
    eps = np.ascontiguousarray(eps, dtype=F32)
    b1 = F32(beta1)
    c = np.subtract(F32(1.0), b1, dtype=F32)
    v = np.add(g, eps, dtype=F32)
    bit = ~(v < F32(0.0))
    s = np.where(bit, F32(1.0), F32(-1.0)).astype(F32)
    delta = np.subtract(v, s, dtype=F32)
    eps_new = np.add(np.multiply(b1, eps, dtype=F32),
                     np.multiply(c, delta, dtype=F32), dtype=F32)
    return pack_bits(bit), eps_new


def decode_signs(bits, n: int) -> np.ndarray:
    """The +1 / -1 vector a sign packet stands for (bit 1 -> +1)."""
    return np.where(unpack_bits(bits, n), F32(1.0), F32(-1.0)).astype(F32)


def onebit_momentum(m, ghat, beta1: float) -> np.ndarray:
    """[ONEBIT] §2.2 动量修正策略: m_t = beta1 * m_{t-1} + (1 - beta1) * ghat_t.

    Float32 sequence: m' = RN(RN(beta1 * m) + RN(RN(1 - beta1) * ghat)).
    """
    m = np.ascontiguousarray(m, dtype=F32)
    ghat = np.ascontiguousarray(ghat, dtype=F32)
    b1 = F32(beta1)
    c = np.subtract(F32(1.0), b1, dtype=F32)
    return np.add(np.multiply(b1, m, dtype=F32),
                  np.multiply(c, ghat, dtype=F32), dtype=F32)


# --------------------------------------------------------------------------
# receive side  ([SPARSE] 详细算法流程 steps 6-7)
# --------------------------------------------------------------------------


def packet_indices(packet, n: int) -> np.ndarray:
    """Global indices of a packet, from its int32 list or its bitmap."""
    if packet.get("indices") is not None:
        return np.asarray(packet["indices"], dtype=np.int64)
    return np.flatnonzero(unpack_bits(packet["bitmap"], n)).astype(np.int64)


def sparse_aggregate(packets, n: int) -> np.ndarray:
    """Step 6: sum the W workers' sparse gradients by index into a dense G.

    [SPARSE] §梯度稀疏化的基本原理 (receiver adds values of equal index) and
    §详细算法流程 step 6.  Packets are added in worker order 0..W-1 onto a
    +0.0 vector, one float32 add per (worker, index); no averaging.
    """
    G = np.zeros(n, dtype=F32)
    for p in packets:
        idx = packet_indices(p, n)
        vals = np.asarray(p["values"], dtype=F32)
        if vals.size != idx.size:
            raise ValueError("packet values and indices differ in length")
        if idx.size and np.any(np.diff(idx) <= 0):
            raise ValueError("packet indices must be strictly ascending")
        G[idx] = np.add(G[idx], vals, dtype=F32)
    return G


def packet_split(indices, bounds) -> np.ndarray:
    """Slice bounds of a packet for index ranges: starts[q] = the number of
    entries whose index is below bounds[q].

    [SPARSE] §详细算法流程 step 5 and §与Allreduce的融合 exchange the packets
    between workers; in the index-range form each receiver gets the entries
    of its own index range, which in an ascending packet are the entries
    [starts[q], starts[q + 1]).  Written as the count it is, one bound at a
    time.
    """
    idx = np.asarray(indices, dtype=np.int64)
    return np.array([int(np.count_nonzero(idx < int(b))) for b in bounds], dtype=np.int64)


def sign_aggregate(bit_vectors, n: int) -> np.ndarray:
    """Step 6 for 1-bit packets: G = sum over workers of the decoded +-1 signs,
    added in worker order (exact: small integers)."""
    G = np.zeros(n, dtype=F32)
    for bits in bit_vectors:
        G = np.add(G, decode_signs(bits, n), dtype=F32)
    return G


def sgd_apply(w, G, eta: float) -> np.ndarray:
    """Step 7: w_{t+1} = w_t - eta * G  (float32: RN(w - RN(eta * G))).

    [SPARSE] §详细算法流程 step 7.  Where G == 0 the result equals w bit for
    bit, so untouched parameters keep their exact value.
    """
    w = np.ascontiguousarray(w, dtype=F32)
    G = np.ascontiguousarray(G, dtype=F32)
    return np.subtract(w, np.multiply(F32(eta), G, dtype=F32), dtype=F32)
