// 8-bit quantisation of top-k packet values ("梯度稀疏化：只传输重要的梯度元素",
// §与其他压缩技术的比较: top-k first, then the selected values quantised to
// 8 bits).  The page gives no formula; this library reads it as symmetric
// int8 with one float32 scale per segment (tensor):
//   s = max |v| / 127 over the segment's finite selected values (0 if none),
//   q = round-half-even(v / s) clamped to [-127, 127]  (0 for NaN or s = 0),
//   receiver value q * s,
//   residual at a selected position e = v - q * s  (§详细算法流程 step 4,
//   e = g - g~ with g~ what the packet carries),
// each step one float32 operation rounded to nearest.
//
// ef_topk_compress_q8 runs the top-k step (values and each entry's position
// land in the workspace), then two passes over the packet: a per-segment
// maximum of |v| (one CTA per chunk of kQChunk entries, one atomicMax per
// CTA on the float's bit pattern, which orders non-negative finite floats),
// and the quantiser, which writes q, the scale and the residual.  Packet
// entries of one segment are contiguous, so a chunk never spans segments.
// Per entry: 4 B value + 4 B position read twice, 1 B written, plus one
// scattered 4-byte residual write (the quantisation error).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "ef_common.cuh"
#include "ef_topk_internal.h"

namespace ef {
namespace {

constexpr int kQThreads = 256;
constexpr int kQChunk = 4096;    // packet entries per CTA
constexpr int kQBatch = 128;     // segments per launch
constexpr uint32_t kFiniteLimit = 0x7F800000u;  // |v| bit patterns below this are finite

// The segments of one launch and the chunks they are cut into.
struct QBatch {
  int64_t out_off[kQBatch];       // first packet entry of each segment
  int64_t seg_off[kQBatch];       // first element of each segment
  int64_t k[kQBatch];
  int64_t chunk_base[kQBatch + 1];  // first chunk of each segment; [nseg] = chunk total
  int32_t seg_id[kQBatch];        // segment number in the whole call
  int32_t nseg;
};

__device__ __forceinline__ int chunk_segment(const QBatch& b, int64_t c) {
  int lo = 0, hi = b.nseg - 1;  // last segment whose first chunk is <= c
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (b.chunk_base[mid] <= c) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Largest finite |v| of each segment: one block maximum per chunk, then one
// atomicMax on the bit pattern.
__global__ void __launch_bounds__(kQThreads)
q8_max(QBatch b, const float* __restrict__ values, uint32_t* maxbits) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint32_t red[kQThreads / 32];
  const int64_t c = blockIdx.x;
  const int s = chunk_segment(b, c);
  const int64_t j0 = b.out_off[s] + (c - b.chunk_base[s]) * kQChunk;
  const int64_t j1 = b.out_off[s] + min((c - b.chunk_base[s] + 1) * (int64_t)kQChunk, b.k[s]);
  uint32_t m = 0;
  for (int64_t j = j0 + threadIdx.x; j < j1; j += kQThreads) {
    const uint32_t a = __float_as_uint(values[j]) & 0x7FFFFFFFu;
    if (a < kFiniteLimit) m = max(m, a);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(kFull, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < kQThreads / 32 ? red[threadIdx.x] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(kFull, m, o));
    if (threadIdx.x == 0 && m) atomicMax(&maxbits[b.seg_id[s]], m);
  }
}

// s = RN(max / 127) from the segment's maximum bit pattern.
__device__ __forceinline__ float q8_segment_scale(uint32_t mbits) {
  return __fdiv_rn(__uint_as_float(mbits), 127.0f);
}

// q = round-half-even(clamp(RN(v / s), -127, 127)); 0 for NaN or s == 0.
__device__ __forceinline__ int q8_code(float v, float s) {
  if (s == 0.0f || isnan(v)) return 0;
  float t = __fdiv_rn(v, s);
  t = fminf(fmaxf(t, -127.0f), 127.0f);
  return __float2int_rn(t);
}

// Codes, scales and residuals of every chunk's entries.
__global__ void __launch_bounds__(kQThreads)
q8_quantize(QBatch b, const float* __restrict__ values, const uint32_t* __restrict__ pos,
            const uint32_t* __restrict__ maxbits, float* __restrict__ e,
            int8_t* __restrict__ out_q, float* __restrict__ out_scale) {
  pdl_wait();
  const int64_t c = blockIdx.x;
  const int s = chunk_segment(b, c);
  const float sc = q8_segment_scale(maxbits[b.seg_id[s]]);
  if (c == b.chunk_base[s] && threadIdx.x == 0) out_scale[b.seg_id[s]] = sc;
  const int64_t j0 = b.out_off[s] + (c - b.chunk_base[s]) * kQChunk;
  const int64_t j1 = b.out_off[s] + min((c - b.chunk_base[s] + 1) * (int64_t)kQChunk, b.k[s]);
  float* es = e + b.seg_off[s];
#pragma unroll 4
  for (int64_t j = j0 + threadIdx.x; j < j1; j += kQThreads) {
    const float v = values[j];
    const int q = q8_code(v, sc);
    out_q[j] = (int8_t)q;
    const float dq = __fmul_rn((float)q, sc);
    es[pos[j]] = __fsub_rn(v, dq);
  }
}

// Receiver: v = RN(q * s) for every entry.
__global__ void __launch_bounds__(kQThreads)
q8_dequantize(QBatch b, const int8_t* __restrict__ q, const float* __restrict__ scales,
              float* __restrict__ out_values) {
  pdl_wait();
  const int64_t c = blockIdx.x;
  const int s = chunk_segment(b, c);
  const float sc = scales[b.seg_id[s]];
  const int64_t j0 = b.out_off[s] + (c - b.chunk_base[s]) * kQChunk;
  const int64_t j1 = b.out_off[s] + min((c - b.chunk_base[s] + 1) * (int64_t)kQChunk, b.k[s]);
#pragma unroll 4
  for (int64_t j = j0 + threadIdx.x; j < j1; j += kQThreads)
    out_values[j] = __fmul_rn((float)q[j], sc);
}

// Cuts the segments with k > 0 into launches of at most kQBatch segments.
// seg_off may be NULL (dequantisation needs only packet offsets).
std::vector<QBatch> q8_batches(int32_t nseg, const int64_t* h_seg_offsets,
                               const int64_t* h_seg_k) {
  std::vector<QBatch> out;
  QBatch cur{};
  int64_t out_off = 0, chunks = 0;
  auto flush = [&]() {
    if (cur.nseg == 0) return;
    cur.chunk_base[cur.nseg] = chunks;
    out.push_back(cur);
    cur = QBatch{};
    chunks = 0;
  };
  for (int32_t i = 0; i < nseg; ++i) {
    const int64_t k = h_seg_k[i];
    if (k > 0) {
      const int t = cur.nseg;
      cur.out_off[t] = out_off;
      cur.seg_off[t] = h_seg_offsets ? h_seg_offsets[i] : 0;
      cur.k[t] = k;
      cur.chunk_base[t] = chunks;
      cur.seg_id[t] = i;
      chunks += (k + kQChunk - 1) / kQChunk;
      if (++cur.nseg == kQBatch) flush();
    }
    out_off += k;
  }
  flush();
  return out;
}

struct Q8Layout {
  size_t topk_bytes = 0, off_values = 0, off_pos = 0, off_max = 0, bytes = 0;
  int64_t total_k = 0;
};

ef_status q8_layout(int64_t n, int32_t nseg, const int64_t* offs, const int64_t* ks,
                    int32_t idx_format, Q8Layout* L) {
  ef_status st = topk_plan_info(n, nseg, offs, ks, idx_format, &L->topk_bytes, &L->total_k);
  if (st != EF_OK) return st;
  size_t off = round_up(std::max<size_t>(L->topk_bytes, 256), 256);
  L->off_values = off;
  off = round_up(off + (size_t)L->total_k * 4, 256);
  L->off_pos = off;
  off = round_up(off + (size_t)L->total_k * 4, 256);
  L->off_max = off;
  off = round_up(off + (size_t)nseg * 4, 256);
  L->bytes = off;
  return EF_OK;
}

}  // namespace
}  // namespace ef

extern "C" ef_status ef_topk_q8_workspace_size(int64_t n, int32_t nseg,
                                               const int64_t* h_seg_offsets,
                                               const int64_t* h_seg_k, int32_t idx_format,
                                               size_t* bytes) {
  if (!bytes) return EF_ERR_NULL;
  ef::Q8Layout L;
  ef_status st = ef::q8_layout(n, nseg, h_seg_offsets, h_seg_k, idx_format, &L);
  if (st != EF_OK) return st;
  *bytes = L.bytes;
  return EF_OK;
}

extern "C" ef_status ef_topk_compress_q8(const float* g_raw, float* e, int64_t n, int32_t nseg,
                                         const int64_t* h_seg_offsets, const int64_t* h_seg_k,
                                         int32_t idx_format, int8_t* out_q, float* out_scale,
                                         int32_t* out_indices, uint32_t* out_bitmap,
                                         void* workspace, size_t workspace_bytes,
                                         void* stream) {
  using namespace ef;
  Q8Layout L;
  ef_status st = q8_layout(n, nseg, h_seg_offsets, h_seg_k, idx_format, &L);
  if (st != EF_OK) return st;
  if (!workspace) return EF_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < L.bytes)
    return EF_ERR_WORKSPACE;
  if (L.total_k > 0 && !out_q) return EF_ERR_NULL;
  if (!out_scale) return EF_ERR_NULL;
  if (!aligned4(out_scale)) return EF_ERR_ALIGN;
  const size_t fb = (size_t)n * 4, kq = (size_t)L.total_k, sb = (size_t)nseg * 4;
  const void* ins[3] = {g_raw, e, workspace};
  const size_t inb[3] = {fb, fb, L.bytes};
  for (int i = 0; i < 3; ++i) {
    if (overlaps(out_q, kq, ins[i], inb[i]) || overlaps(out_scale, sb, ins[i], inb[i]))
      return EF_ERR_ALIAS;
  }
  if (overlaps(out_q, kq, out_scale, sb)) return EF_ERR_ALIAS;
  const bool bitmap = idx_format == EF_IDX_BITMAP;
  const size_t ob = bitmap ? (size_t)((n + 31) / 32) * 4 : (size_t)L.total_k * 4;
  const void* idx_out = bitmap ? (const void*)out_bitmap : (const void*)out_indices;
  if (overlaps(idx_out, ob, out_q, kq) || overlaps(idx_out, ob, out_scale, sb))
    return EF_ERR_ALIAS;

  char* ws = static_cast<char*>(workspace);
  float* values = reinterpret_cast<float*>(ws + L.off_values);
  uint32_t* pos = reinterpret_cast<uint32_t*>(ws + L.off_pos);
  uint32_t* maxbits = reinterpret_cast<uint32_t*>(ws + L.off_max);
  // The top-k step checks every remaining argument; its workspace is the
  // first L.topk_bytes bytes (packet values and positions live after it).
  st = topk_compress_impl(g_raw, e, n, nseg, h_seg_offsets, h_seg_k, idx_format, values,
                          out_indices, out_bitmap, pos, workspace, L.topk_bytes, stream);
  if (st != EF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (nseg > 0) {
    cudaError_t err = cudaMemsetAsync(out_scale, 0, sb, s);
    if (err == cudaSuccess) err = cudaMemsetAsync(maxbits, 0, sb, s);
    if (err != cudaSuccess) return cuda_fail(err);
  }
  for (const QBatch& b : q8_batches(nseg, h_seg_offsets, h_seg_k)) {
    const int64_t chunks = b.chunk_base[b.nseg];
    launch_pdl(q8_max, (unsigned)chunks, kQThreads, 0, s, b, values, maxbits);
    if ((st = check_launch()) != EF_OK) return st;
    launch_pdl(q8_quantize, (unsigned)chunks, kQThreads, 0, s, b, values, pos, maxbits, e, out_q,
                                                        out_scale);
    if ((st = check_launch()) != EF_OK) return st;
  }
  return EF_OK;
}

extern "C" ef_status ef_q8_dequantize(const int8_t* q, const float* scales, int32_t nseg,
                                      const int64_t* h_seg_k, float* out_values,
                                      void* stream) {
  using namespace ef;
  if (nseg < 1) return EF_ERR_SEGMENTS;
  if (!h_seg_k) return EF_ERR_NULL;
  int64_t total = 0;
  for (int32_t i = 0; i < nseg; ++i) {
    if (h_seg_k[i] < 0 || h_seg_k[i] > (int64_t(1) << 31)) return EF_ERR_K;
    total += h_seg_k[i];
  }
  if (total == 0) return EF_OK;
  if (!q || !scales || !out_values) return EF_ERR_NULL;
  if (!aligned4(scales) || !aligned4(out_values)) return EF_ERR_ALIGN;
  if (overlaps(out_values, (size_t)total * 4, q, (size_t)total) ||
      overlaps(out_values, (size_t)total * 4, scales, (size_t)nseg * 4))
    return EF_ERR_ALIAS;
  DeviceInfo dev;
  ef_status st = current_device(&dev);
  if (st != EF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (const QBatch& b : q8_batches(nseg, nullptr, h_seg_k)) {
    launch_pdl(q8_dequantize, (unsigned)b.chunk_base[b.nseg], kQThreads, 0, s, b, q, scales, out_values);
    if ((st = check_launch()) != EF_OK) return st;
  }
  return EF_OK;
}
