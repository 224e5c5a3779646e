// Library-internal entry points of the top-k path, shared by the public
// top-k and 8-bit-quantised top-k calls (not part of the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>

#include "efgrad.h"

namespace ef {

// Validates the segment table; returns the top-k workspace size and the
// packet length (sum of k).
ef_status topk_plan_info(int64_t n, int32_t nseg, const int64_t* h_seg_offsets,
                         const int64_t* h_seg_k, int32_t idx_format, size_t* bytes,
                         int64_t* total_k);

// ef_topk_compress with one more optional output: pos_out[j] = the position
// of packet entry j inside its segment (uint32[sum k], device; may be NULL).
ef_status topk_compress_impl(const float* g_raw, float* e, int64_t n, int32_t nseg,
                             const int64_t* h_seg_offsets, const int64_t* h_seg_k,
                             int32_t idx_format, float* out_values, int32_t* out_indices,
                             uint32_t* out_bitmap, uint32_t* pos_out, void* workspace,
                             size_t workspace_bytes, void* stream);

}  // namespace ef
