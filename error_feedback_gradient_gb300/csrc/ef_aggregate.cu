// Receive side for top-k packets ("梯度稀疏化：只传输重要的梯度元素",
// §梯度稀疏化的基本原理 receiver and §详细算法流程 steps 6-7):
//   G[i] = (((+0 + p_0[i]) + p_1[i]) + ...) in worker order over the packets
//          that contain i;  w[i] -= eta * G[i] where some packet contains i.
//
// The dense index space is cut into tiles of kATile elements.  Because every
// packet is sorted, the entries of worker w that fall in tile t form one run
// [start[w][t], start[w][t+1]):
//   * int32 packets: one pass over the packet entries writes the run
//     boundaries (each entry fills the starts of the tiles between its
//     predecessor's tile and its own);
//   * bitmap packets: per-tile population counts, then one exclusive scan
//     per worker.
// The apply kernel then gives each tile to one CTA: it accumulates the runs
// worker by worker in a shared-memory copy of the tile (no atomics on
// values; indices inside one packet are distinct), writes the dense tile of G
// with 16-byte stores, and updates w only at the touched positions.
// Algorithmic traffic: 4 B per element for G, 8 B per packet entry (values +
// indices, or values + n/8 bitmap bytes per worker), 8 B per touched w.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "ef_common.cuh"

namespace ef {
namespace {

constexpr int kATile = 8192;
constexpr int kAThreads = 256;
constexpr int kAWords = kATile / 32;
static_assert(kAWords == kAThreads, "one bitmap word per thread");

struct AggArgs {
  const float* values[EF_MAX_WORKERS];
  const int32_t* indices[EF_MAX_WORKERS];
  const uint32_t* bitmaps[EF_MAX_WORKERS];
  int64_t k[EF_MAX_WORKERS];
  int64_t kbase[EF_MAX_WORKERS + 1];
  int32_t W;
  int32_t bitmap;
  int64_t n, ntiles;
  float eta;
};

__device__ __forceinline__ int64_t* starts_of(int64_t* start, const AggArgs& a, int w) {
  return start + (int64_t)w * (a.ntiles + 1);
}

__device__ __forceinline__ int64_t clamp_tile(int64_t idx, const AggArgs& a) {
  if (idx < 0) return -1;
  const int64_t t = idx / kATile;
  return t >= a.ntiles ? a.ntiles - 1 : t;
}

// Run boundaries for int32 packets; validates order and range.
__global__ void __launch_bounds__(kAThreads)
agg_starts_int32(AggArgs a, int64_t* start, int32_t* status) {
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = a.kbase[a.W];
  for (int64_t x = tid; x < total; x += nthr) {
    int w = 0;
    while (w + 1 < a.W && a.kbase[w + 1] <= x) ++w;
    const int64_t j = x - a.kbase[w];
    const int32_t* ind = a.indices[w];
    int64_t* st = starts_of(start, a, w);
    const int64_t idx = ind[j];
    const int64_t prev = j > 0 ? (int64_t)ind[j - 1] : -1;
    const bool ok = idx >= 0 && idx < a.n && (j == 0 || idx > prev);
    if (!ok) set_status(status, EF_ERR_PACKET);
    const int64_t t = clamp_tile(idx, a);
    const int64_t tp = j > 0 ? clamp_tile(prev, a) : -1;
    for (int64_t tt = tp + 1; tt <= t; ++tt) st[tt] = j;
    if (j == a.k[w] - 1)
      for (int64_t tt = (t < 0 ? 0 : t + 1); tt <= a.ntiles; ++tt) st[tt] = a.k[w];
  }
  const int64_t span = a.ntiles + 1;
  for (int64_t x = tid; x < (int64_t)a.W * span; x += nthr) {
    const int w = (int)(x / span);
    if (a.k[w] == 0) starts_of(start, a, w)[x % span] = 0;
  }
}

// Per-(worker, tile) population counts of bitmap packets.
__global__ void __launch_bounds__(kAThreads)
agg_count_bitmap(AggArgs a, uint32_t* counts) {
  __shared__ uint32_t red[kAThreads / 32];
  const int64_t nwords = (a.n + 31) / 32;
  for (int64_t x = blockIdx.x; x < (int64_t)a.W * a.ntiles; x += gridDim.x) {
    const int w = (int)(x / a.ntiles);
    const int64_t t = x % a.ntiles;
    const int64_t wi = t * kAWords + threadIdx.x;
    uint32_t c = wi < nwords ? __popc(__ldg(a.bitmaps[w] + wi)) : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(kFull, c, o);
    if (lane_id() == 0) red[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t s = 0;
      for (int i = 0; i < kAThreads / 32; ++i) s += red[i];
      counts[x] = s;
    }
    __syncthreads();
  }
}

// Exclusive scan of one worker's tile counts (one CTA per worker).  A
// thread's partial sum can exceed 32 bits when n >= 2^32, so the low 16 bits
// and the rest of each partial sum are scanned separately.
__global__ void __launch_bounds__(1024)
agg_scan_bitmap(AggArgs a, const uint32_t* counts, int64_t* start, int32_t* status) {
  __shared__ uint32_t scratch[64];
  const int w = blockIdx.x;
  const uint32_t* c = counts + (int64_t)w * a.ntiles;
  int64_t* st = starts_of(start, a, w);
  const int64_t per = (a.ntiles + blockDim.x - 1) / blockDim.x;
  const int64_t t0 = (int64_t)threadIdx.x * per;
  const int64_t t1 = min(t0 + per, a.ntiles);
  uint64_t local = 0;
  for (int64_t t = t0; t < t1; ++t) local += c[t];
  uint32_t tot_lo, tot_hi;
  const uint32_t ex_lo = block_excl_scan((uint32_t)(local & 0xFFFFu), scratch, &tot_lo);
  const uint32_t ex_hi = block_excl_scan((uint32_t)(local >> 16), scratch, &tot_hi);
  uint64_t run = ((uint64_t)ex_hi << 16) + ex_lo;
  for (int64_t t = t0; t < t1; ++t) {
    st[t] = (int64_t)run;
    run += c[t];
  }
  if (threadIdx.x == 0) {
    const uint64_t total = ((uint64_t)tot_hi << 16) + tot_lo;
    st[a.ntiles] = (int64_t)total;
    if ((int64_t)total != a.k[w]) set_status(status, EF_ERR_PACKET);
  }
}

__global__ void __launch_bounds__(kAThreads)
agg_apply(AggArgs a, const int64_t* start, float* __restrict__ G, float* __restrict__ wts) {
  __shared__ __align__(16) float acc[kATile];
  __shared__ uint32_t touched[kAWords];
  __shared__ uint32_t scratch[64];
  const int tid = threadIdx.x;
  const bool g_vec = (reinterpret_cast<uintptr_t>(G) & 15u) == 0;
  for (int64_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
    const int64_t t0 = tile * kATile;
    const int tlen = (int)min((int64_t)kATile, a.n - t0);
    int any = 0;
    if (tid < a.W) {
      const int64_t* st = start + (int64_t)tid * (a.ntiles + 1);
      any = st[tile + 1] > st[tile];
    }
    any = __syncthreads_or(any);
    if (!any && !G) continue;
    float4* acc4 = reinterpret_cast<float4*>(acc);
#pragma unroll
    for (int r = 0; r < kATile / 4 / kAThreads; ++r)
      acc4[r * kAThreads + tid] = make_float4(0.f, 0.f, 0.f, 0.f);
    touched[tid] = 0;
    __syncthreads();
    if (any) {
      for (int w = 0; w < a.W; ++w) {
        const int64_t* st = start + (int64_t)w * (a.ntiles + 1);
        const int64_t kw = a.k[w];
        int64_t lo = st[tile], hi = st[tile + 1];
        lo = lo < 0 ? 0 : (lo > kw ? kw : lo);
        hi = hi < lo ? lo : (hi > kw ? kw : hi);
        const float* vals = a.values[w];
        if (!a.bitmap) {
          const int32_t* ind = a.indices[w];
          for (int64_t j = lo + tid; j < hi; j += kAThreads) {
            const int64_t slot = (int64_t)ind[j] - t0;
            if (slot >= 0 && slot < tlen) {
              acc[slot] = __fadd_rn(acc[slot], vals[j]);
              atomicOr(&touched[slot >> 5], 1u << (slot & 31));
            }
          }
        } else {
          const int64_t wi = t0 / 32 + tid;
          uint32_t word = 0;
          if (tid * 32 < tlen) {
            word = __ldg(a.bitmaps[w] + wi);
            const int rem = tlen - tid * 32;
            if (rem < 32) word &= (1u << rem) - 1u;
          }
          uint32_t tot;
          const uint32_t ex = block_excl_scan(__popc(word), scratch, &tot);
          int64_t j = lo + ex;
          touched[tid] |= word;
          while (word) {
            const int b = __ffs(word) - 1;
            word &= word - 1;
            if (j < hi) acc[tid * 32 + b] = __fadd_rn(acc[tid * 32 + b], vals[j]);
            ++j;
          }
        }
        __syncthreads();
      }
    }
    if (G) {
      float* gt = G + t0;
      if (g_vec && tlen == kATile) {
#pragma unroll
        for (int r = 0; r < kATile / 4 / kAThreads; ++r)
          __stcs(reinterpret_cast<float4*>(gt) + r * kAThreads + tid, acc4[r * kAThreads + tid]);
      } else {
        for (int i = tid; i < tlen; i += kAThreads) gt[i] = acc[i];
      }
    }
    uint32_t word = touched[tid];
    while (word) {
      const int b = __ffs(word) - 1;
      word &= word - 1;
      const int slot = tid * 32 + b;
      const int64_t i = t0 + slot;
      wts[i] = __fsub_rn(wts[i], __fmul_rn(a.eta, acc[slot]));
    }
    __syncthreads();
  }
}

int64_t agg_tiles(int64_t n) { return (n + kATile - 1) / kATile; }

size_t agg_bytes(int32_t W, int32_t idx_format, int64_t n) {
  const int64_t nt = agg_tiles(n);
  size_t off = sizeof(WsHeader);
  off = round_up(off + (size_t)W * (nt + 1) * 8, 256);
  if (idx_format == EF_IDX_BITMAP) off = round_up(off + (size_t)W * nt * 4, 256);
  return off;
}

}  // namespace
}  // namespace ef

extern "C" ef_status ef_aggregate_workspace_size(int32_t W, int32_t idx_format, int64_t n,
                                                 size_t* bytes) {
  if (!bytes) return EF_ERR_NULL;
  if (W < 1 || W > EF_MAX_WORKERS) return EF_ERR_WORKERS;
  if (idx_format != EF_IDX_INT32 && idx_format != EF_IDX_BITMAP) return EF_ERR_ARG;
  if (n < 0) return EF_ERR_SIZE;
  *bytes = ef::agg_bytes(W, idx_format, n);
  return EF_OK;
}

extern "C" ef_status sparse_aggregate_apply(int32_t W, int32_t idx_format,
                                            const float* const* h_values,
                                            const int32_t* const* h_indices,
                                            const uint32_t* const* h_bitmaps, const int64_t* h_k,
                                            int64_t n, float eta, float* G, float* w,
                                            void* workspace, size_t workspace_bytes,
                                            void* stream) {
  using namespace ef;
  if (W < 1 || W > EF_MAX_WORKERS) return EF_ERR_WORKERS;
  if (idx_format != EF_IDX_INT32 && idx_format != EF_IDX_BITMAP) return EF_ERR_ARG;
  if (n < 0) return EF_ERR_SIZE;
  if (idx_format == EF_IDX_INT32 && n > (int64_t(1) << 31)) return EF_ERR_SIZE;
  if (!std::isfinite(eta)) return EF_ERR_ARG;
  if (!h_values || !h_k) return EF_ERR_NULL;
  const bool bitmap = idx_format == EF_IDX_BITMAP;
  if (bitmap ? !h_bitmaps : !h_indices) return EF_ERR_NULL;
  const size_t need = agg_bytes(W, idx_format, n);
  if (!workspace) return EF_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < need)
    return EF_ERR_WORKSPACE;
  if (n > 0 && !w) return EF_ERR_NULL;
  if ((w && !aligned4(w)) || (G && !aligned4(G))) return EF_ERR_ALIGN;
  const size_t fb = (size_t)n * 4, wb = (size_t)((n + 31) / 32) * 4;
  if (G && overlaps(G, fb, w, fb)) return EF_ERR_ALIAS;
  if (overlaps(workspace, need, w, fb) || (G && overlaps(workspace, need, G, fb)))
    return EF_ERR_ALIAS;
  AggArgs a{};
  a.W = W;
  a.bitmap = bitmap ? 1 : 0;
  a.n = n;
  a.ntiles = agg_tiles(n);
  a.eta = eta;
  a.kbase[0] = 0;
  for (int i = 0; i < W; ++i) {
    const int64_t k = h_k[i];
    if (k < 0 || k > n) return EF_ERR_K;
    if (k > 0 && !h_values[i]) return EF_ERR_NULL;
    if (h_values[i] && !aligned4(h_values[i])) return EF_ERR_ALIGN;
    const size_t kb = (size_t)k * 4;
    if (overlaps(h_values[i], kb, w, fb) || (G && overlaps(h_values[i], kb, G, fb)))
      return EF_ERR_ALIAS;
    if (bitmap) {
      if (n > 0 && !h_bitmaps[i]) return EF_ERR_NULL;
      if (h_bitmaps[i] && !aligned4(h_bitmaps[i])) return EF_ERR_ALIGN;
      if (overlaps(h_bitmaps[i], wb, w, fb) || (G && overlaps(h_bitmaps[i], wb, G, fb)))
        return EF_ERR_ALIAS;
      a.bitmaps[i] = h_bitmaps[i];
    } else {
      if (k > 0 && !h_indices[i]) return EF_ERR_NULL;
      if (h_indices[i] && !aligned4(h_indices[i])) return EF_ERR_ALIGN;
      if (overlaps(h_indices[i], kb, w, fb) || (G && overlaps(h_indices[i], kb, G, fb)))
        return EF_ERR_ALIAS;
      a.indices[i] = h_indices[i];
    }
    a.values[i] = h_values[i];
    a.k[i] = k;
    a.kbase[i + 1] = a.kbase[i] + k;
  }
  DeviceInfo dev;
  ef_status st = current_device(&dev);
  if (st != EF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  cudaError_t err = cudaMemsetAsync(ws, 0, sizeof(WsHeader), s);
  if (err != cudaSuccess) return cuda_fail(err);
  if (n == 0) return EF_OK;
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  int64_t* start = reinterpret_cast<int64_t*>(ws + sizeof(WsHeader));
  const int64_t nt = a.ntiles;
  if (!bitmap) {
    const int64_t work = std::max<int64_t>(a.kbase[W], (int64_t)W * (nt + 1));
    const int grid = (int)std::max<int64_t>(
        1, std::min<int64_t>((work + kAThreads - 1) / kAThreads, (int64_t)dev.sms * 8));
    agg_starts_int32<<<grid, kAThreads, 0, s>>>(a, start, status);
    if ((st = check_launch()) != EF_OK) return st;
  } else {
    uint32_t* counts = reinterpret_cast<uint32_t*>(
        ws + round_up(sizeof(WsHeader) + (size_t)W * (nt + 1) * 8, 256));
    const int grid = (int)std::max<int64_t>(
        1, std::min<int64_t>((int64_t)W * nt, (int64_t)dev.sms * 8));
    agg_count_bitmap<<<grid, kAThreads, 0, s>>>(a, counts);
    if ((st = check_launch()) != EF_OK) return st;
    agg_scan_bitmap<<<W, 1024, 0, s>>>(a, counts, start, status);
    if ((st = check_launch()) != EF_OK) return st;
  }
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(nt, (int64_t)dev.sms * 6));
  prof_begin(EF_KERNEL_SPARSE_APPLY, s);
  agg_apply<<<grid, kAThreads, 0, s>>>(a, start, G, w);
  if ((st = check_launch()) != EF_OK) return st;
  prof_end(EF_KERNEL_SPARSE_APPLY, s);
  return EF_OK;
}
