"""ctypes binding of libefgrad (the C ABI in include/efgrad.h).

Argument marshalling only: torch tensors are turned into device pointers,
Python lists into host arrays, and the current torch CUDA stream into the
``stream`` argument.  Every step of the computation runs in the library's
CUDA kernels.  The library is loaded on first use; if it has not been built
the call raises, there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import torch

IDX_INT32 = 0
IDX_BITMAP = 1
APPLY_SGD = 0
APPLY_MOMENTUM = 1

KERNEL_TOPK_FUSED = 1
KERNEL_SIGN = 2
KERNEL_SPARSE_APPLY = 3
KERNEL_SIGN_APPLY = 4

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libefgrad.so"
_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return os.path.join(_HERE, "lib", _LIB_NAME)


class EFError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({_status_string(status)})")


_c_i64p = ctypes.POINTER(ctypes.c_int64)
_c_vp = ctypes.c_void_p
_c_vpp = ctypes.POINTER(ctypes.c_void_p)

# name -> (restype, argtypes), mirroring include/efgrad.h
_SIGNATURES = {
    "ef_abi_version": (ctypes.c_int32, []),
    "ef_status_string": (ctypes.c_char_p, [ctypes.c_int32]),
    "ef_last_cuda_error": (ctypes.c_int32, []),
    "ef_kernel_launches": (ctypes.c_int64, []),
    "ef_topk_workspace_size": (ctypes.c_int32, [
        ctypes.c_int64, ctypes.c_int32, _c_i64p, _c_i64p, ctypes.c_int32,
        ctypes.POINTER(ctypes.c_size_t)]),
    "ef_topk_compress": (ctypes.c_int32, [
        _c_vp, _c_vp, ctypes.c_int64, ctypes.c_int32, _c_i64p, _c_i64p,
        ctypes.c_int32, _c_vp, _c_vp, _c_vp, _c_vp, ctypes.c_size_t, _c_vp]),
    "ef_topk_compress_noalloc": (ctypes.c_int32, [
        _c_vp, _c_vp, ctypes.c_int64, ctypes.c_int32, _c_i64p, _c_i64p,
        ctypes.c_int32, _c_vp, _c_vp, _c_vp, _c_vp]),
    "ef_topk_noalloc_status": (ctypes.c_int32, [_c_vp, ctypes.POINTER(ctypes.c_int32)]),
    "ef_topk_q8_workspace_size": (ctypes.c_int32, [
        ctypes.c_int64, ctypes.c_int32, _c_i64p, _c_i64p, ctypes.c_int32,
        ctypes.POINTER(ctypes.c_size_t)]),
    "ef_topk_compress_q8": (ctypes.c_int32, [
        _c_vp, _c_vp, ctypes.c_int64, ctypes.c_int32, _c_i64p, _c_i64p,
        ctypes.c_int32, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, ctypes.c_size_t, _c_vp]),
    "ef_q8_dequantize": (ctypes.c_int32, [
        _c_vp, _c_vp, ctypes.c_int32, _c_i64p, _c_vp, _c_vp]),
    "ef_index_codec_sizes": (ctypes.c_int32, [
        ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.POINTER(ctypes.c_size_t),
        ctypes.POINTER(ctypes.c_size_t)]),
    "ef_index_encode": (ctypes.c_int32, [
        ctypes.c_int32, _c_vp, ctypes.c_int64, ctypes.c_int64, _c_vp, ctypes.c_size_t, _c_vp,
        _c_vp, ctypes.c_size_t, _c_vp]),
    "ef_index_decode": (ctypes.c_int32, [
        ctypes.c_int32, _c_vp, ctypes.c_size_t, ctypes.c_int64, ctypes.c_int64, _c_vp, _c_vp,
        ctypes.c_size_t, _c_vp]),
    "ef_randk_workspace_size": (ctypes.c_int32, [
        ctypes.c_int64, ctypes.c_int32, _c_i64p, _c_i64p, ctypes.POINTER(ctypes.c_size_t)]),
    "ef_randk_compress": (ctypes.c_int32, [
        _c_vp, _c_vp, ctypes.c_int64, ctypes.c_int32, _c_i64p, _c_i64p, ctypes.c_uint64,
        ctypes.c_uint64, _c_vp, _c_vp, ctypes.c_int64, _c_vp, _c_vp, ctypes.c_size_t, _c_vp]),
    "ef_sign_compress": (ctypes.c_int32, [
        _c_vp, _c_vp, ctypes.c_int64, ctypes.c_float, _c_vp, _c_vp]),
    "ef_aggregate_workspace_size": (ctypes.c_int32, [
        ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
        ctypes.POINTER(ctypes.c_size_t)]),
    "sparse_aggregate_apply": (ctypes.c_int32, [
        ctypes.c_int32, ctypes.c_int32, _c_vpp, _c_vpp, _c_vpp, _c_i64p,
        ctypes.c_int64, ctypes.c_float, _c_vp, _c_vp, _c_vp, ctypes.c_size_t,
        _c_vp]),
    "sign_aggregate_apply": (ctypes.c_int32, [
        ctypes.c_int32, _c_vpp, ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
        ctypes.c_float, _c_vp, _c_vp, _c_vp]),
    "ef_packet_split": (ctypes.c_int32, [
        _c_vp, ctypes.c_int64, ctypes.c_int32, _c_i64p, _c_vp, _c_vp]),
    "ef_index_rebase": (ctypes.c_int32, [_c_vp, ctypes.c_int64, ctypes.c_int64, _c_vp]),
    "ef_workspace_status": (ctypes.c_int32, [
        _c_vp, _c_vp, ctypes.POINTER(ctypes.c_int32)]),
    "ef_profile_events": (ctypes.c_int32, [ctypes.c_int32, _c_vp, _c_vp]),
    "ef_selftest_wait_timeout": (ctypes.c_int32, [_c_vp, ctypes.c_size_t, ctypes.c_int64,
                                                  _c_vp]),
}


def library() -> ctypes.CDLL:
    """Load libefgrad.so (once).  Raises if it is missing: build it with
    ``python -c "import __graft_entry__ as g; g.build()"``."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is not built; the CUDA library is required "
                    "(run __graft_entry__.build())")
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _status_string(s: int) -> str:
    try:
        return library().ef_status_string(s).decode()
    except Exception:  # pragma: no cover
        return "?"


def _check(status: int, what: str) -> None:
    if status != 0:
        raise EFError(status, what)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _i64(xs: Sequence[int]):
    return (ctypes.c_int64 * len(xs))(*[int(x) for x in xs])


def _ptrs(ts: Sequence[Optional[torch.Tensor]]):
    return (ctypes.c_void_p * len(ts))(*[_ptr(t) for t in ts])


# ---------------------------------------------------------------------------
# top-k
# ---------------------------------------------------------------------------


def topk_workspace_size(n: int, seg_offsets: Sequence[int], seg_k: Sequence[int],
                        idx_format: int = IDX_INT32) -> int:
    out = ctypes.c_size_t(0)
    _check(library().ef_topk_workspace_size(
        int(n), len(seg_k), _i64(seg_offsets), _i64(seg_k), int(idx_format),
        ctypes.byref(out)), "ef_topk_workspace_size")
    return int(out.value)


def topk_compress(g_raw: torch.Tensor, e: torch.Tensor, seg_offsets: Sequence[int],
                  seg_k: Sequence[int], out_values: torch.Tensor,
                  out_indices: Optional[torch.Tensor] = None,
                  out_bitmap: Optional[torch.Tensor] = None,
                  workspace: Optional[torch.Tensor] = None,
                  idx_format: int = IDX_INT32, stream=None) -> None:
    n = g_raw.numel()
    if workspace is None:
        nbytes = topk_workspace_size(n, seg_offsets, seg_k, idx_format)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=g_raw.device)
    _check(library().ef_topk_compress(
        _ptr(g_raw), _ptr(e), n, len(seg_k), _i64(seg_offsets), _i64(seg_k),
        int(idx_format), _ptr(out_values), _ptr(out_indices), _ptr(out_bitmap),
        _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), "ef_topk_compress")


def topk_compress_noalloc(g_raw: torch.Tensor, e: torch.Tensor, seg_offsets: Sequence[int],
                          seg_k: Sequence[int], out_values: torch.Tensor,
                          out_indices: Optional[torch.Tensor] = None,
                          out_bitmap: Optional[torch.Tensor] = None,
                          idx_format: int = IDX_INT32, stream=None) -> None:
    """ef_topk_compress_noalloc: the same step with the library's own scratch
    array (no allocation by the library or here)."""
    _check(library().ef_topk_compress_noalloc(
        _ptr(g_raw), _ptr(e), g_raw.numel(), len(seg_k), _i64(seg_offsets), _i64(seg_k),
        int(idx_format), _ptr(out_values), _ptr(out_indices), _ptr(out_bitmap),
        _stream(stream)), "ef_topk_compress_noalloc")


def topk_noalloc_status(stream=None) -> int:
    """ef_topk_noalloc_status: the device-side status of the last
    allocation-free top-k call on the current device (synchronises)."""
    out = ctypes.c_int32(0)
    _check(library().ef_topk_noalloc_status(_stream(stream), ctypes.byref(out)),
           "ef_topk_noalloc_status")
    return int(out.value)


def topk_q8_workspace_size(n: int, seg_offsets: Sequence[int], seg_k: Sequence[int],
                           idx_format: int = IDX_INT32) -> int:
    out = ctypes.c_size_t(0)
    _check(library().ef_topk_q8_workspace_size(
        int(n), len(seg_k), _i64(seg_offsets), _i64(seg_k), int(idx_format),
        ctypes.byref(out)), "ef_topk_q8_workspace_size")
    return int(out.value)


def topk_compress_q8(g_raw: torch.Tensor, e: torch.Tensor, seg_offsets: Sequence[int],
                     seg_k: Sequence[int], out_q: torch.Tensor, out_scale: torch.Tensor,
                     out_indices: Optional[torch.Tensor] = None,
                     out_bitmap: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None,
                     idx_format: int = IDX_INT32, stream=None) -> None:
    """ef_topk_compress_q8: top-k EF step with int8 packet values and one
    fp32 scale per segment (see include/efgrad.h)."""
    n = g_raw.numel()
    if workspace is None:
        nbytes = topk_q8_workspace_size(n, seg_offsets, seg_k, idx_format)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=g_raw.device)
    _check(library().ef_topk_compress_q8(
        _ptr(g_raw), _ptr(e), n, len(seg_k), _i64(seg_offsets), _i64(seg_k),
        int(idx_format), _ptr(out_q), _ptr(out_scale), _ptr(out_indices), _ptr(out_bitmap),
        _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), "ef_topk_compress_q8")


def q8_dequantize(q: torch.Tensor, scales: torch.Tensor, seg_k: Sequence[int],
                  out_values: torch.Tensor, stream=None) -> None:
    """ef_q8_dequantize: out_values = q * scale of each entry's segment."""
    _check(library().ef_q8_dequantize(
        _ptr(q), _ptr(scales), len(seg_k), _i64(seg_k), _ptr(out_values),
        _stream(stream)), "ef_q8_dequantize")


# ---------------------------------------------------------------------------
# random magnitude-proportional sparsification
# ---------------------------------------------------------------------------


def randk_workspace_size(n: int, seg_offsets: Sequence[int], seg_k: Sequence[int]) -> int:
    out = ctypes.c_size_t(0)
    _check(library().ef_randk_workspace_size(int(n), len(seg_k), _i64(seg_offsets),
                                             _i64(seg_k), ctypes.byref(out)),
           "ef_randk_workspace_size")
    return int(out.value)


def randk_compress(g_raw: torch.Tensor, e: torch.Tensor, seg_offsets: Sequence[int],
                   seg_k: Sequence[int], seed: int, step: int, out_values: torch.Tensor,
                   out_indices: torch.Tensor, counts: torch.Tensor,
                   workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """ef_randk_compress: keep-with-probability-proportional-to-|g| EF step;
    ``counts`` (int64 [nseg + 1], device) receives the entries sent per
    segment and their total."""
    n = g_raw.numel()
    if workspace is None:
        workspace = torch.empty(randk_workspace_size(n, seg_offsets, seg_k), dtype=torch.uint8,
                                device=g_raw.device)
    _check(library().ef_randk_compress(
        _ptr(g_raw), _ptr(e), n, len(seg_k), _i64(seg_offsets), _i64(seg_k),
        int(seed) & (2**64 - 1), int(step) & (2**64 - 1), _ptr(out_values), _ptr(out_indices),
        out_values.numel(), _ptr(counts), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)), "ef_randk_compress")


# ---------------------------------------------------------------------------
# index codecs
# ---------------------------------------------------------------------------

CODEC_LOCAL16 = 1
CODEC_RUNVARINT = 2
CODEC_BLOCK256 = 3


def index_codec_sizes(codec: int, K: int, n: int):
    """(upper bound of the stream's bytes, workspace bytes) for K indices of n."""
    mb, wb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(library().ef_index_codec_sizes(int(codec), int(K), int(n), ctypes.byref(mb),
                                          ctypes.byref(wb)), "ef_index_codec_sizes")
    return int(mb.value), int(wb.value)


def index_encode(codec: int, indices: torch.Tensor, n: int, out: torch.Tensor,
                 out_bytes: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """ef_index_encode: int32 indices -> byte stream in ``out``; its length
    lands in ``out_bytes`` (one int64 on the device)."""
    _check(library().ef_index_encode(
        int(codec), _ptr(indices), indices.numel(), int(n), _ptr(out),
        out.numel() * out.element_size(), _ptr(out_bytes), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)), "ef_index_encode")


def index_decode(codec: int, stream_bytes: torch.Tensor, nbytes: int, K: int, n: int,
                 indices: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """ef_index_decode: the first ``nbytes`` bytes of ``stream_bytes`` -> K
    int32 indices."""
    _check(library().ef_index_decode(
        int(codec), _ptr(stream_bytes), int(nbytes), int(K), int(n), _ptr(indices),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
        "ef_index_decode")


# ---------------------------------------------------------------------------
# 1-bit
# ---------------------------------------------------------------------------


def sign_compress(g: torch.Tensor, eps: torch.Tensor, beta1: float,
                  out_bits: torch.Tensor, stream=None) -> None:
    _check(library().ef_sign_compress(
        _ptr(g), _ptr(eps), g.numel(), float(beta1), _ptr(out_bits),
        _stream(stream)), "ef_sign_compress")


def sign_aggregate_apply(bits: Sequence[torch.Tensor], n: int, mode: int,
                         eta: float, beta1: float, G: Optional[torch.Tensor],
                         w_or_m: torch.Tensor, stream=None) -> None:
    _check(library().sign_aggregate_apply(
        len(bits), _ptrs(bits), int(n), int(mode), float(eta), float(beta1),
        _ptr(G), _ptr(w_or_m), _stream(stream)), "sign_aggregate_apply")


# ---------------------------------------------------------------------------
# receive side
# ---------------------------------------------------------------------------


def aggregate_workspace_size(W: int, idx_format: int, n: int) -> int:
    out = ctypes.c_size_t(0)
    _check(library().ef_aggregate_workspace_size(
        int(W), int(idx_format), int(n), ctypes.byref(out)),
        "ef_aggregate_workspace_size")
    return int(out.value)


def sparse_aggregate_apply(values: Sequence[torch.Tensor],
                           indices: Optional[Sequence[torch.Tensor]],
                           bitmaps: Optional[Sequence[torch.Tensor]],
                           ks: Sequence[int], n: int, eta: float,
                           G: Optional[torch.Tensor], w: torch.Tensor,
                           workspace: Optional[torch.Tensor] = None,
                           idx_format: int = IDX_INT32, stream=None) -> None:
    W = len(values)
    if workspace is None:
        nbytes = aggregate_workspace_size(W, idx_format, n)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=w.device)
    ind = _ptrs(indices) if indices is not None else None
    bms = _ptrs(bitmaps) if bitmaps is not None else None
    _check(library().sparse_aggregate_apply(
        W, int(idx_format), _ptrs(values), ind, bms, _i64(ks), int(n),
        float(eta), _ptr(G), _ptr(w), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)),
        "sparse_aggregate_apply")


def kernel_launches() -> int:
    """Kernels this thread has launched through the library so far."""
    return int(library().ef_kernel_launches())


def workspace_status(workspace: torch.Tensor, stream=None) -> int:
    out = ctypes.c_int32(0)
    _check(library().ef_workspace_status(_ptr(workspace), _stream(stream),
                                         ctypes.byref(out)), "ef_workspace_status")
    return int(out.value)


def selftest_wait_timeout(workspace: torch.Tensor, limit_ns: int, stream=None) -> None:
    """Run the bounded-wait self-test (see include/efgrad.h)."""
    _check(library().ef_selftest_wait_timeout(
        _ptr(workspace), workspace.numel() * workspace.element_size(), int(limit_ns),
        _stream(stream)), "ef_selftest_wait_timeout")


def profile_events(kernel_id: int, start, stop) -> None:
    """Bracket every launch of ``kernel_id`` by this thread with the two
    torch.cuda.Event objects (recorded once beforehand so they exist)."""
    s = None if start is None else start.cuda_event
    t = None if stop is None else stop.cuda_event
    _check(library().ef_profile_events(int(kernel_id), s, t), "ef_profile_events")


# ---------------------------------------------------------------------------
# device steps of the index-range packet exchange
# ---------------------------------------------------------------------------


def packet_split(indices: torch.Tensor, k: int, bounds: Sequence[int],
                 starts: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """ef_packet_split: starts[q] = number of the first k entries of the
    ascending packet `indices` below bounds[q] (int64 device tensor of
    len(bounds) entries, allocated here unless given)."""
    if starts is None:
        starts = torch.empty(len(bounds), dtype=torch.int64, device=indices.device)
    _check(library().ef_packet_split(
        _ptr(indices), int(k), len(bounds) - 1, _i64(bounds), _ptr(starts),
        _stream(stream)), "ef_packet_split")
    return starts


def index_rebase(indices: torch.Tensor, count: int, base: int, stream=None) -> None:
    """ef_index_rebase: indices[:count] -= base, in place."""
    _check(library().ef_index_rebase(_ptr(indices), int(count), int(base), _stream(stream)),
           "ef_index_rebase")
