// Index codecs for top-k packets ("梯度稀疏化：只传输重要的梯度元素",
// §索引编码压缩 and §快速上手指南 step 4).  The page names the ideas -- 16-bit
// indices, block-sparse flags, run-length / delta codes of variable length
// -- and this library fixes three lossless byte formats for an ascending
// int32 index list of K entries from [0, n) (all little-endian):
//   LOCAL16    uint32 block_start[nblk + 1] (entries before each 65536-element
//              block, nblk = ceil(n / 65536)), then uint16 offset-in-block
//              per entry;
//   RUNVARINT  per entry the number of unselected elements since the
//              previous entry (i_j - i_{j-1} - 1, i_{-1} = -1) as unsigned
//              LEB128 (7-bit groups, low first, high bit = more follow);
//   BLOCK256   uint32 flags[ceil(nb / 32)] (bit b % 32 of word b / 32 set
//              when 256-element block b holds an entry, nb = ceil(n / 256)),
//              then uint8 (count - 1) per flagged block, then uint8
//              offset-in-block per entry.
//
// Every variable-length step is a prefix sum, done as a two-pass scan over
// chunks of kItems items: pass 1 reduces each chunk (one CTA per chunk),
// one CTA scans the chunk sums, pass 2 rescans each chunk with its offset
// and writes.  A codec phase is a small functor: value(j) is item j's
// contribution, apply(j, offset) writes item j given the sum of the items
// before it.  Malformed inputs (unsorted or out-of-range indices, streams
// that do not parse) are never read or written out of bounds; they set
// EF_ERR_PACKET in the workspace status word.
#include <cuda_runtime.h>

#include <algorithm>

#include "ef_common.cuh"

namespace ef {
namespace {

constexpr int kCT = 256;              // threads per CTA
constexpr int kPerThread = 16;        // consecutive items per thread
constexpr int kItems = kCT * kPerThread;  // items per chunk
constexpr int kScanThreads = 1024;
constexpr int64_t kL16Block = 65536;
constexpr int64_t kB256 = 256;
constexpr uint64_t kNoPos = ~0ull;

int64_t chunks_of(int64_t items) { return (items + kItems - 1) / kItems; }

__device__ __forceinline__ uint64_t warp_excl_u64(uint64_t v, uint64_t* total) {
  const unsigned lane = lane_id();
  uint64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(kFull, x, o);
    if (lane >= (unsigned)o) x += y;
  }
  *total = __shfl_sync(kFull, x, 31);
  return x - v;
}

// Exclusive scan of one value per thread over the CTA.
__device__ __forceinline__ uint64_t cta_excl_u64(uint64_t v, uint64_t* sh, uint64_t* total) {
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  uint64_t wt;
  const uint64_t ex = warp_excl_u64(v, &wt);
  if (lane_id() == 0) sh[warp] = wt;
  __syncthreads();
  if (warp == 0) {
    const uint64_t s = lane_id() < (unsigned)nw ? sh[lane_id()] : 0ull;
    uint64_t t;
    const uint64_t e2 = warp_excl_u64(s, &t);
    if (lane_id() < (unsigned)nw) sh[lane_id()] = e2;
    if (lane_id() == 0) sh[32] = t;
  }
  __syncthreads();
  const uint64_t r = ex + sh[warp];
  *total = sh[32];
  __syncthreads();
  return r;
}

// Pass 1: sum of value(j) over each chunk.
template <class Op>
__global__ void __launch_bounds__(kCT) chunk_sums(Op op, int64_t nitems, uint64_t* sums) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint64_t sh[33];
  const int64_t j0 = (int64_t)blockIdx.x * kItems + (int64_t)threadIdx.x * kPerThread;
  uint64_t v = 0;
  for (int u = 0; u < kPerThread; ++u)
    if (j0 + u < nitems) v += op.value(j0 + u);
  uint64_t total;
  cta_excl_u64(v, sh, &total);
  if (threadIdx.x == 0) sums[blockIdx.x] = total;
}

// One CTA: chunk sums -> exclusive chunk offsets, in place; the grand total
// goes to *total and, when given, to *total_copy.
__global__ void __launch_bounds__(kScanThreads)
scan_sums(uint64_t* sums, int64_t nchunks, uint64_t* total, uint64_t* total_copy,
          uint64_t total_bias) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint64_t sh[33];
  const int64_t per = (nchunks + kScanThreads - 1) / kScanThreads;
  const int64_t c0 = (int64_t)threadIdx.x * per;
  uint64_t local = 0;
  for (int64_t c = c0; c < c0 + per && c < nchunks; ++c) local += sums[c];
  uint64_t t;
  uint64_t run = cta_excl_u64(local, sh, &t);
  for (int64_t c = c0; c < c0 + per && c < nchunks; ++c) {
    const uint64_t v = sums[c];
    sums[c] = run;
    run += v;
  }
  if (threadIdx.x == 0) {
    *total = t;
    if (total_copy) *total_copy = t + total_bias;
  }
}

// Pass 2: apply(j, offset of j) for every item, offsets from the scanned sums.
template <class Op>
__global__ void __launch_bounds__(kCT) chunk_apply(Op op, int64_t nitems, const uint64_t* sums) {
  pdl_wait();
  __shared__ uint64_t sh[33];
  const int64_t j0 = (int64_t)blockIdx.x * kItems + (int64_t)threadIdx.x * kPerThread;
  uint64_t v[kPerThread];
  uint64_t local = 0;
#pragma unroll
  for (int u = 0; u < kPerThread; ++u) {
    v[u] = j0 + u < nitems ? op.value(j0 + u) : 0ull;
    local += v[u];
  }
  uint64_t total;
  uint64_t off = sums[blockIdx.x] + cta_excl_u64(local, sh, &total);
#pragma unroll
  for (int u = 0; u < kPerThread; ++u) {
    if (j0 + u < nitems) op.apply(j0 + u, off);
    off += v[u];
  }
}

template <class Op>
ef_status run_scan(Op op, int64_t nitems, uint64_t* sums, uint64_t* total,
                   uint64_t* total_copy, uint64_t bias, cudaStream_t s) {
  const int64_t nch = chunks_of(nitems);
  ef_status st;
  if (nch == 0) {  // nothing to scan: the totals are zero (plus the bias for the copy)
    launch_pdl(scan_sums, 1, kScanThreads, 0, s, sums, 0, total, total_copy, bias);
    return check_launch();
  }
  launch_pdl(chunk_sums<Op>, (unsigned)nch, kCT, 0, s, op, nitems, sums);
  if ((st = check_launch()) != EF_OK) return st;
  launch_pdl(scan_sums, 1, kScanThreads, 0, s, sums, nch, total, total_copy, bias);
  if ((st = check_launch()) != EF_OK) return st;
  launch_pdl(chunk_apply<Op>, (unsigned)nch, kCT, 0, s, op, nitems, sums);
  return check_launch();
}

// Validated index j of the packet (clamped into [0, n); order errors reported).
__device__ __forceinline__ int64_t checked_index(const int32_t* idx, int64_t j, int64_t n,
                                                 int32_t* status) {
  int64_t i = idx[j];
  const int64_t p = j > 0 ? (int64_t)idx[j - 1] : -1;
  if (i < 0 || i >= n || i <= p) {
    set_status(status, EF_ERR_PACKET);
    i = i < 0 ? 0 : (i >= n ? n - 1 : i);
  }
  return i;
}

// ---------------------------------------------------------------- LOCAL16

__global__ void __launch_bounds__(kCT)
l16_encode(const int32_t* idx, int64_t K, int64_t n, int64_t nblk, uint8_t* out,
           uint64_t* out_bytes, int32_t* status) {
  pdl_wait();
  uint32_t* starts = reinterpret_cast<uint32_t*>(out);
  uint16_t* low = reinterpret_cast<uint16_t*>(out + 4 * (nblk + 1));
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (tid == 0) *out_bytes = (uint64_t)(4 * (nblk + 1) + 2 * K);
  for (int64_t j = tid; j < K; j += nthr) {
    const int64_t i = checked_index(idx, j, n, status);
    int64_t p = j > 0 ? (int64_t)idx[j - 1] : -1;
    p = p < -1 ? -1 : (p >= n ? n - 1 : p);
    const int64_t b = i / kL16Block, bp = p < 0 ? -1 : p / kL16Block;
    for (int64_t bb = bp + 1; bb <= b; ++bb) starts[bb] = (uint32_t)j;
    low[j] = (uint16_t)(i % kL16Block);
    if (j == K - 1)
      for (int64_t bb = b + 1; bb <= nblk; ++bb) starts[bb] = (uint32_t)K;
  }
}

__global__ void __launch_bounds__(kCT)
l16_decode(const uint8_t* in, int64_t K, int64_t n, int64_t nblk, int32_t* idx, int32_t* status) {
  pdl_wait();
  const uint32_t* starts = reinterpret_cast<const uint32_t*>(in);
  const uint16_t* low = reinterpret_cast<const uint16_t*>(in + 4 * (nblk + 1));
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (tid == 0 && (starts[0] != 0 || (int64_t)starts[nblk] != K))
    set_status(status, EF_ERR_PACKET);
  for (int64_t j = tid; j < K; j += nthr) {
    int64_t lo = 0, hi = nblk - 1;  // last block whose start is <= j
    while (lo < hi) {
      const int64_t mid = (lo + hi + 1) >> 1;
      if ((int64_t)starts[mid] <= j) lo = mid;
      else hi = mid - 1;
    }
    int64_t i = lo * kL16Block + low[j];
    if ((int64_t)starts[lo] > j || (int64_t)starts[lo + 1] <= j || i >= n) {
      set_status(status, EF_ERR_PACKET);
      i = 0;
    }
    idx[j] = (int32_t)i;
  }
}

// ---------------------------------------------------------------- RUNVARINT

__device__ __forceinline__ uint32_t leb_len(uint64_t r) {
  uint32_t l = 1;
  while (r >= 128) {
    r >>= 7;
    ++l;
  }
  return l;
}

__device__ __forceinline__ uint64_t run_before(const int32_t* idx, int64_t j, int64_t n,
                                               int32_t* status) {
  const int64_t i = checked_index(idx, j, n, status);
  int64_t p = j > 0 ? (int64_t)idx[j - 1] : -1;
  p = p < -1 ? -1 : (p >= n ? n - 1 : p);
  return i > p ? (uint64_t)(i - p - 1) : 0ull;
}

// Encoder: item = entry, value = LEB128 length of its run.
struct RvEncode {
  const int32_t* idx;
  int64_t n;
  uint8_t* out;
  int32_t* status;
  __device__ uint64_t value(int64_t j) const { return leb_len(run_before(idx, j, n, status)); }
  __device__ void apply(int64_t j, uint64_t off) const {
    uint64_t r = run_before(idx, j, n, status);
    while (r >= 128) {
      out[off++] = (uint8_t)(r & 0x7F) | 0x80;
      r >>= 7;
    }
    out[off] = (uint8_t)r;
  }
};

// Decoder step 1: item = byte, value = 1 for a byte that ends an entry; the
// end of entry e is recorded at end[e].
struct RvTerminals {
  const uint8_t* in;
  int64_t K;
  uint64_t* end;
  int32_t* status;
  __device__ uint64_t value(int64_t b) const { return (in[b] & 0x80) ? 0ull : 1ull; }
  __device__ void apply(int64_t b, uint64_t e) const {
    if (in[b] & 0x80) return;
    if ((int64_t)e < K) end[e] = (uint64_t)b;
    else set_status(status, EF_ERR_PACKET);
  }
};

// Decoder step 2: item = entry, value = run + 1; index = prefix + value - 1.
struct RvIndices {
  const uint8_t* in;
  int64_t nbytes, K, n;
  const uint64_t* end;
  int32_t* idx;
  int32_t* status;
  __device__ uint64_t run(int64_t e) const {
    const uint64_t last = end[e];
    const uint64_t first = e > 0 ? end[e - 1] + 1 : 0;
    if (last == kNoPos || (e > 0 && end[e - 1] == kNoPos) || last < first ||
        last >= (uint64_t)nbytes || last - first >= 5) {
      set_status(status, EF_ERR_PACKET);
      return 0;
    }
    uint64_t r = 0;
    for (uint64_t b = first; b <= last; ++b) r |= (uint64_t)(in[b] & 0x7F) << (7 * (b - first));
    return r;
  }
  __device__ uint64_t value(int64_t e) const { return run(e) + 1; }
  __device__ void apply(int64_t e, uint64_t off) const {
    const uint64_t i = off + run(e);  // (sum of run + 1 over earlier entries) + run
    if (e == K - 1 && end[e] != (uint64_t)(nbytes - 1))
      set_status(status, EF_ERR_PACKET);  // bytes after the last entry
    if (i >= (uint64_t)n) {
      set_status(status, EF_ERR_PACKET);
      idx[e] = 0;
    } else {
      idx[e] = (int32_t)i;
    }
  }
};

// ---------------------------------------------------------------- BLOCK256

// Encoder: item = entry, value = 1 for the first entry of its block.
struct B256Encode {
  const int32_t* idx;
  int64_t n, K, nfw;
  uint8_t* out;
  const uint64_t* nnzb;  // device: flagged blocks (the scan's total)
  uint32_t* first_of;    // [flagged blocks] entry number of each block's first entry
  int32_t* status;
  __device__ bool first(int64_t j) const {
    const int64_t i = checked_index(idx, j, n, status);
    return j == 0 || i / kB256 != ((int64_t)idx[j - 1] < 0 ? -1 : (int64_t)idx[j - 1] / kB256);
  }
  __device__ uint64_t value(int64_t j) const { return first(j) ? 1ull : 0ull; }
  __device__ void apply(int64_t j, uint64_t rank) const {
    const int64_t i = checked_index(idx, j, n, status);
    const uint64_t nz = *nnzb;
    out[4 * nfw + nz + j] = (uint8_t)(i % kB256);
    if (first(j)) {
      const int64_t b = i / kB256;
      atomicOr(reinterpret_cast<uint32_t*>(out) + (b >> 5), 1u << (b & 31));
      if (rank < nz) first_of[rank] = (uint32_t)j;
    }
  }
};

__global__ void __launch_bounds__(kCT)
b256_counts(const uint32_t* first_of, const uint64_t* nnzb, int64_t K, int64_t nfw, uint8_t* out,
            int32_t* status) {
  pdl_trigger();
  pdl_wait();
  const uint64_t nz = *nnzb;
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < (int64_t)nz; r += nthr) {
    const int64_t next = r + 1 < (int64_t)nz ? (int64_t)first_of[r + 1] : K;
    const int64_t c = next - (int64_t)first_of[r];
    if (c < 1 || c > kB256) set_status(status, EF_ERR_PACKET);
    out[4 * nfw + r] = (uint8_t)(c - 1);
  }
}

// Decoder step 1: item = flag word, value = its set bits (inside nb); the
// r-th flagged block's number goes to block_of[r].
struct B256Flags {
  const uint32_t* flags;
  int64_t nb, nnzb;
  uint32_t* block_of;
  int32_t* status;
  __device__ uint32_t word(int64_t w) const {
    uint32_t x = flags[w];
    const int64_t rem = nb - w * 32;
    if (rem < 32) x &= (1u << rem) - 1u;
    return x;
  }
  __device__ uint64_t value(int64_t w) const { return __popc(word(w)); }
  __device__ void apply(int64_t w, uint64_t rank) const {
    uint32_t x = word(w);
    while (x) {
      const int bit = __ffs(x) - 1;
      x &= x - 1;
      if ((int64_t)rank < nnzb) block_of[rank] = (uint32_t)(w * 32 + bit);
      else set_status(status, EF_ERR_PACKET);
      ++rank;
    }
  }
};

// Decoder step 2: item = flagged block, value = its entry count.
struct B256Entries {
  const uint8_t* counts;
  const uint8_t* offsets;
  const uint32_t* block_of;
  int64_t K, n;
  int32_t* idx;
  int32_t* status;
  __device__ uint64_t value(int64_t r) const { return (uint64_t)counts[r] + 1; }
  __device__ void apply(int64_t r, uint64_t start) const {
    const uint64_t c = (uint64_t)counts[r] + 1;
    const int64_t b = block_of[r];
    for (uint64_t t = 0; t < c; ++t) {
      const uint64_t j = start + t;
      if (j >= (uint64_t)K) {
        set_status(status, EF_ERR_PACKET);
        return;
      }
      const int64_t i = b * kB256 + offsets[j];
      if (i >= n || (t > 0 && offsets[j] <= offsets[j - 1])) set_status(status, EF_ERR_PACKET);
      idx[j] = (int32_t)(i < n ? i : 0);
    }
  }
};

__global__ void check_total(const uint64_t* total, uint64_t want, int32_t* status) {
  pdl_wait();
  if (threadIdx.x == 0 && *total != want) set_status(status, EF_ERR_PACKET);
}

// ---------------------------------------------------------------- planning

struct CodecSizes {
  size_t max_stream = 0, workspace = 0;
  size_t off_sums = 0, off_total = 0, off_aux = 0;
};

ef_status codec_sizes(int32_t codec, int64_t K, int64_t n, CodecSizes* c) {
  if (n < 0 || n > (int64_t(1) << 31)) return EF_ERR_SIZE;
  if (K < 0 || K > n) return EF_ERR_K;
  const int64_t nblk = (n + kL16Block - 1) / kL16Block;
  const int64_t nfw = ((n + kB256 - 1) / kB256 + 31) / 32;
  int64_t items = 0;
  size_t aux = 0;
  switch (codec) {
    case EF_CODEC_LOCAL16:
      c->max_stream = (size_t)(4 * (nblk + 1) + 2 * K);
      break;
    case EF_CODEC_RUNVARINT:
      c->max_stream = (size_t)(5 * K);
      items = 5 * K;
      aux = (size_t)K * 8;
      break;
    case EF_CODEC_BLOCK256:
      c->max_stream = (size_t)(4 * nfw + 2 * K);
      items = std::max<int64_t>(K, nfw);
      aux = (size_t)K * 4;
      break;
    default:
      return EF_ERR_ARG;
  }
  size_t off = sizeof(WsHeader);
  c->off_sums = off;
  off = round_up(off + (size_t)(chunks_of(items) + 1) * 8, 256);
  c->off_total = off;
  off += 256;
  c->off_aux = off;
  off = round_up(off + aux, 256);
  c->workspace = off;
  return EF_OK;
}

}  // namespace
}  // namespace ef

extern "C" ef_status ef_index_codec_sizes(int32_t codec, int64_t K, int64_t n,
                                          size_t* max_stream_bytes, size_t* workspace_bytes) {
  if (!max_stream_bytes || !workspace_bytes) return EF_ERR_NULL;
  ef::CodecSizes c;
  ef_status st = ef::codec_sizes(codec, K, n, &c);
  if (st != EF_OK) return st;
  *max_stream_bytes = c.max_stream;
  *workspace_bytes = c.workspace;
  return EF_OK;
}

extern "C" ef_status ef_index_encode(int32_t codec, const int32_t* indices, int64_t K, int64_t n,
                                     uint8_t* out, size_t out_capacity, uint64_t* d_out_bytes,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  using namespace ef;
  CodecSizes c;
  ef_status st = codec_sizes(codec, K, n, &c);
  if (st != EF_OK) return st;
  if (!workspace) return EF_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < c.workspace)
    return EF_ERR_WORKSPACE;
  if (!d_out_bytes || (K > 0 && !indices) || (c.max_stream > 0 && !out)) return EF_ERR_NULL;
  if (out_capacity < c.max_stream) return EF_ERR_SIZE;
  if ((reinterpret_cast<uintptr_t>(d_out_bytes) & 7u) != 0 || (indices && !aligned4(indices)) ||
      (out && !aligned4(out)))
    return EF_ERR_ALIGN;
  const size_t ib = (size_t)K * 4;
  if (overlaps(out, c.max_stream, indices, ib) || overlaps(out, c.max_stream, workspace, c.workspace) ||
      overlaps(indices, ib, workspace, c.workspace) || overlaps(d_out_bytes, 8, out, c.max_stream) ||
      overlaps(d_out_bytes, 8, workspace, c.workspace))
    return EF_ERR_ALIAS;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != EF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  cudaError_t err = cudaMemsetAsync(ws, 0, sizeof(WsHeader), s);
  if (err != cudaSuccess) return cuda_fail(err);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  uint64_t* sums = reinterpret_cast<uint64_t*>(ws + c.off_sums);
  uint64_t* total = reinterpret_cast<uint64_t*>(ws + c.off_total);
  const int64_t nblk = (n + kL16Block - 1) / kL16Block;
  const int64_t nfw = ((n + kB256 - 1) / kB256 + 31) / 32;
  const int grid = (int)std::max<int64_t>(
      1, std::min<int64_t>((K + kCT - 1) / kCT, (int64_t)dev.sms * 8));
  if (codec == EF_CODEC_LOCAL16) {
    if (K == 0) {
      err = cudaMemsetAsync(out, 0, 4 * (nblk + 1), s);
      if (err != cudaSuccess) return cuda_fail(err);
    }
    launch_pdl(l16_encode, grid, kCT, 0, s, indices, K, n, nblk, out, d_out_bytes, status);
    return check_launch();
  }
  if (codec == EF_CODEC_RUNVARINT) {
    RvEncode op{indices, n, out, status};
    return run_scan(op, K, sums, total, d_out_bytes, 0, s);
  }
  // BLOCK256: flags cleared, then ranks of each block's first entry
  if (nfw > 0) {
    err = cudaMemsetAsync(out, 0, 4 * nfw, s);
    if (err != cudaSuccess) return cuda_fail(err);
  }
  uint32_t* first_of = reinterpret_cast<uint32_t*>(ws + c.off_aux);
  B256Encode op{indices, n, K, nfw, out, total, first_of, status};
  if ((st = run_scan(op, K, sums, total, d_out_bytes, (uint64_t)(4 * nfw + K), s)) != EF_OK)
    return st;
  if (K > 0) {
    launch_pdl(b256_counts, grid, kCT, 0, s, first_of, total, K, nfw, out, status);
    return check_launch();
  }
  return EF_OK;
}

extern "C" ef_status ef_index_decode(int32_t codec, const uint8_t* in, size_t in_bytes, int64_t K,
                                     int64_t n, int32_t* indices, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  using namespace ef;
  CodecSizes c;
  ef_status st = codec_sizes(codec, K, n, &c);
  if (st != EF_OK) return st;
  if (!workspace) return EF_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < c.workspace)
    return EF_ERR_WORKSPACE;
  if ((K > 0 && !indices) || (in_bytes > 0 && !in)) return EF_ERR_NULL;
  if ((indices && !aligned4(indices)) || (in && !aligned4(in))) return EF_ERR_ALIGN;
  const int64_t nblk = (n + kL16Block - 1) / kL16Block;
  const int64_t nb = (n + kB256 - 1) / kB256;
  const int64_t nfw = (nb + 31) / 32;
  // stream lengths the format cannot have
  if (codec == EF_CODEC_LOCAL16 && in_bytes != c.max_stream) return EF_ERR_PACKET;
  if (codec == EF_CODEC_RUNVARINT && (in_bytes < (size_t)K || in_bytes > c.max_stream))
    return EF_ERR_PACKET;
  const int64_t nnzb = (int64_t)in_bytes - 4 * nfw - K;
  if (codec == EF_CODEC_BLOCK256 && (nnzb < 0 || nnzb > K || (K > 0) != (nnzb > 0)))
    return EF_ERR_PACKET;
  const size_t ib = (size_t)K * 4;
  if (overlaps(indices, ib, in, in_bytes) || overlaps(indices, ib, workspace, c.workspace) ||
      overlaps(in, in_bytes, workspace, c.workspace))
    return EF_ERR_ALIAS;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != EF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  cudaError_t err = cudaMemsetAsync(ws, 0, sizeof(WsHeader), s);
  if (err != cudaSuccess) return cuda_fail(err);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  uint64_t* sums = reinterpret_cast<uint64_t*>(ws + c.off_sums);
  uint64_t* total = reinterpret_cast<uint64_t*>(ws + c.off_total);
  if (codec == EF_CODEC_LOCAL16) {
    if (K == 0) return EF_OK;
    const int grid = (int)std::max<int64_t>(
        1, std::min<int64_t>((K + kCT - 1) / kCT, (int64_t)dev.sms * 8));
    launch_pdl(l16_decode, grid, kCT, 0, s, in, K, n, nblk, indices, status);
    return check_launch();
  }
  if (codec == EF_CODEC_RUNVARINT) {
    if (K == 0) return EF_OK;
    uint64_t* end = reinterpret_cast<uint64_t*>(ws + c.off_aux);
    err = cudaMemsetAsync(end, 0xFF, (size_t)K * 8, s);
    if (err != cudaSuccess) return cuda_fail(err);
    RvTerminals t{in, K, end, status};
    if ((st = run_scan(t, (int64_t)in_bytes, sums, total, nullptr, 0, s)) != EF_OK) return st;
    launch_pdl(check_total, 1, 32, 0, s, total, (uint64_t)K, status);
    if ((st = check_launch()) != EF_OK) return st;
    RvIndices op{in, (int64_t)in_bytes, K, n, end, indices, status};
    return run_scan(op, K, sums, total, nullptr, 0, s);
  }
  if (K == 0) return EF_OK;
  uint32_t* block_of = reinterpret_cast<uint32_t*>(ws + c.off_aux);
  B256Flags f{reinterpret_cast<const uint32_t*>(in), nb, nnzb, block_of, status};
  if ((st = run_scan(f, nfw, sums, total, nullptr, 0, s)) != EF_OK) return st;
  launch_pdl(check_total, 1, 32, 0, s, total, (uint64_t)nnzb, status);
  if ((st = check_launch()) != EF_OK) return st;
  B256Entries en{in + 4 * nfw, in + 4 * nfw + nnzb, block_of, K, n, indices, status};
  if ((st = run_scan(en, nnzb, sums, total, nullptr, 0, s)) != EF_OK) return st;
  launch_pdl(check_total, 1, 32, 0, s, total, (uint64_t)K, status);
  return check_launch();
}
