"""Error-feedback gradient compression on GB300 (sm_103a).

The compute lives in ``libefgrad.so`` (hand-written CUDA behind a C ABI,
declared in ``include/efgrad.h``).  ``binding`` marshals torch tensors to
that ABI; it loads the library on first use and raises if it was not built,
so there is no fallback path.  ``workloads`` holds the seeded synthetic
inputs.
"""

from .binding import (  # noqa: F401
    CODEC_BLOCK256,
    CODEC_LOCAL16,
    CODEC_RUNVARINT,
    EFError,
    IDX_BITMAP,
    IDX_INT32,
    APPLY_MOMENTUM,
    APPLY_SGD,
    index_codec_sizes,
    index_decode,
    index_encode,
    kernel_launches,
    library,
    library_path,
    randk_compress,
    randk_workspace_size,
    sign_aggregate_apply,
    sign_compress,
    sparse_aggregate_apply,
    q8_dequantize,
    topk_compress,
    topk_compress_q8,
    topk_q8_workspace_size,
    topk_workspace_size,
    aggregate_workspace_size,
    workspace_status,
)
