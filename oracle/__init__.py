"""CPU oracle for error-feedback gradient compression.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference legs of ``bench.py``, never by the product
library or its binding.  See ``ef_oracle.py`` for sources and readings.
"""

from .ef_oracle import (  # noqa: F401
    abs_key,
    compensate,
    decode_block256,
    decode_local16,
    decode_runvarint,
    decode_signs,
    encode_block256,
    encode_local16,
    encode_runvarint,
    leb128,
    onebit_momentum,
    pack_bits,
    packet_indices,
    packet_split,
    philox4x32_10,
    q8_dequantize,
    q8_quantize,
    q8_scale,
    randk_coefficient,
    randk_ef_step,
    randk_keep,
    randk_scale,
    randk_words,
    sgd_apply,
    sign_aggregate,
    sign_ef_step,
    sparse_aggregate,
    topk_ef_step,
    topk_q8_ef_step,
    topk_indices,
    unpack_bits,
)
