// Receive side for top-k packets ("梯度稀疏化：只传输重要的梯度元素",
// §梯度稀疏化的基本原理 receiver and §详细算法流程 steps 6-7):
//   G[i] = (((+0 + p_0[i]) + p_1[i]) + ...) in worker order over the packets
//          that contain i;  w[i] -= eta * G[i] where some packet contains i.
//
// The dense index space is cut into tiles of kWT = 1024 elements, one per
// warp.  Because every packet is sorted, the entries of worker w that fall in
// tile t form one run [start[w][t], start[w][t+1]):
//   * int32 packets: one pass over the packet entries writes the run
//     boundaries (each entry fills the starts of the tiles between its
//     predecessor's tile and its own);
//   * bitmap packets: per-tile population counts, then one exclusive scan
//     per worker.
// The apply kernel gives each tile to one warp (48 tiles in flight per SM,
// enough to cover the dependent loads of a tile): the warp loads the run
// bounds of all workers at once, then the runs' entries of up to 4 workers
// at once, adds them worker by worker into a shared-memory copy of the tile
// (no atomics on values; indices inside one packet are distinct), writes the
// dense tile of G with 16-byte stores, and updates w only where touched.
// Algorithmic traffic: 4 B per element for G, 8 B per packet entry (values +
// indices, or values + n/8 bitmap bytes per worker), 8 B per touched w.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "ef_common.cuh"

namespace ef {
namespace {

constexpr int kWT = 1024;            // elements per warp tile
constexpr int kAThreads = 256;
constexpr int kAWarps = kAThreads / 32;
constexpr int kPre = 4;              // workers whose run entries are loaded at once

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

__device__ __forceinline__ uint32_t* starts_of(uint32_t* start, const AggArgs& a, int w) {
  return start + (int64_t)w * (a.ntiles + 1);
}

__device__ __forceinline__ int64_t clamp_tile(int64_t idx, const AggArgs& a) {
  if (idx < 0) return -1;
  const int64_t t = idx / kWT;
  return t >= a.ntiles ? a.ntiles - 1 : t;
}

// Run boundaries for int32 packets; validates order and range.
__global__ void __launch_bounds__(kAThreads)
agg_starts_int32(AggArgs a, uint32_t* start, int32_t* status) {
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = a.kbase[a.W];
  for (int64_t x = tid; x < total; x += nthr) {
    int w = 0;
    while (w + 1 < a.W && a.kbase[w + 1] <= x) ++w;
    const int64_t j = x - a.kbase[w];
    const int32_t* ind = a.indices[w];
    uint32_t* st = starts_of(start, a, w);
    const int64_t idx = ind[j];
    const int64_t prev = j > 0 ? (int64_t)ind[j - 1] : -1;
    const bool ok = idx >= 0 && idx < a.n && (j == 0 || idx > prev);
    if (!ok) set_status(status, EF_ERR_PACKET);
    const int64_t t = clamp_tile(idx, a);
    const int64_t tp = j > 0 ? clamp_tile(prev, a) : -1;
    for (int64_t tt = tp + 1; tt <= t; ++tt) st[tt] = (uint32_t)j;
    if (j == a.k[w] - 1)
      for (int64_t tt = (t < 0 ? 0 : t + 1); tt <= a.ntiles; ++tt) st[tt] = (uint32_t)a.k[w];
  }
  const int64_t span = a.ntiles + 1;
  for (int64_t x = tid; x < (int64_t)a.W * span; x += nthr) {
    const int w = (int)(x / span);
    if (a.k[w] == 0) starts_of(start, a, w)[x % span] = 0;
  }
}

constexpr int kScanTiles = 2048;  // tiles per chunk of the bitmap run-boundary pass

// Run boundaries for bitmap packets in one pass: CTAs take chunks of
// kScanTiles tiles in ticket order (worker-major), count each tile's set bits
// with one warp per tile, scan the chunk in shared memory and get the
// chunk's offset from the bounded decoupled look-back.  The last chunk of a
// worker checks the total against k_w.
__global__ void __launch_bounds__(kAThreads)
agg_bitmap_starts(AggArgs a, uint32_t* start, uint64_t* cstate, uint32_t* ticket,
                  int32_t* status) {
  __shared__ uint32_t cnt[kScanTiles];
  __shared__ uint32_t scratch[64];
  __shared__ uint32_t s_t;
  __shared__ uint64_t s_excl;
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  const int64_t nchunks = (a.ntiles + kScanTiles - 1) / kScanTiles;
  const int64_t nwords = (a.n + 31) / 32;
  for (;;) {
    if (threadIdx.x == 0) s_t = atomicAdd(ticket, 1u);
    __syncthreads();
    const int64_t tk = s_t;
    if (tk >= (int64_t)a.W * nchunks) break;
    const int w = (int)(tk / nchunks);
    const int64_t c = tk % nchunks;
    const int64_t t0 = c * kScanTiles;
    const int ntl = (int)min((int64_t)kScanTiles, a.ntiles - t0);
    const uint32_t* bm = a.bitmaps[w];
    // A tile is 32 words; lane l of a warp reads words 4l..4l+3 of a 4-tile
    // group (16 bytes, when the bitmap is 16-byte aligned), so 8 lanes share
    // a tile.  Four groups are loaded before any is counted.
    const bool v16 = (reinterpret_cast<uintptr_t>(bm) & 15u) == 0;
    for (int i0 = warp * 16; i0 < ntl; i0 += kAWarps * 16) {
      uint32_t c[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int tile = i0 + u * 4 + (int)(lane >> 3);
        const int64_t wi = (t0 + tile) * (kWT / 32) + (lane & 7) * 4;
        c[u] = 0;
        if (tile < ntl) {
          if (v16 && wi + 4 <= nwords) {
            const uint4 q = __ldg(reinterpret_cast<const uint4*>(bm + wi));
            c[u] = __popc(q.x) + __popc(q.y) + __popc(q.z) + __popc(q.w);
          } else {
            for (int r = 0; r < 4; ++r)
              if (wi + r < nwords) c[u] += __popc(__ldg(bm + wi + r));
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint32_t v = c[u];
        v += __shfl_xor_sync(kFull, v, 1);
        v += __shfl_xor_sync(kFull, v, 2);
        v += __shfl_xor_sync(kFull, v, 4);
        const int tile = i0 + u * 4 + (int)(lane >> 3);
        if ((lane & 7) == 0 && tile < ntl) cnt[tile] = v;
      }
    }
    __syncthreads();
    // thread t scans tiles [t * per, (t + 1) * per) of the chunk
    constexpr int per = kScanTiles / kAThreads;
    uint32_t local = 0;
#pragma unroll
    for (int q = 0; q < per; ++q) {
      const int i = threadIdx.x * per + q;
      local += i < ntl ? cnt[i] : 0u;
    }
    uint32_t total;
    const uint32_t ex = block_excl_scan(local, scratch, &total);
    if (warp == 0) {
      const uint64_t e = lookback_warp(cstate, tk, (int64_t)w * nchunks, total, status);
      if (lane == 0) s_excl = e;
    }
    __syncthreads();
    uint32_t* st = starts_of(start, a, w);
    uint64_t run = s_excl + ex;
#pragma unroll
    for (int q = 0; q < per; ++q) {
      const int i = threadIdx.x * per + q;
      if (i < ntl) {
        st[t0 + i] = (uint32_t)run;
        run += cnt[i];
      }
    }
    if (c == nchunks - 1 && threadIdx.x == 0) {
      const uint64_t all = s_excl + total;
      st[a.ntiles] = (uint32_t)all;
      if ((int64_t)all != a.k[w]) set_status(status, EF_ERR_PACKET);
    }
    __syncthreads();
  }
}

// Run of worker w in tile t, clamped into [0, k_w] (k_w < 2^32).
__device__ __forceinline__ void run_of(const AggArgs& a, const uint32_t* start, int w, int64_t t,
                                       uint32_t* lo, uint32_t* hi) {
  const uint32_t* st = start + (int64_t)w * (a.ntiles + 1);
  const uint32_t kw = (uint32_t)a.k[w];
  uint32_t l = st[t], h = st[t + 1];
  l = l > kw ? kw : l;
  h = h < l ? l : (h > kw ? kw : h);
  *lo = l;
  *hi = h;
}

template <bool kBitmap>
__global__ void __launch_bounds__(kAThreads, 6)
agg_apply(AggArgs a, const uint32_t* start, float* __restrict__ G, float* __restrict__ wts) {
  __shared__ __align__(16) float acc_all[kAWarps][kWT];
  __shared__ uint32_t touched_all[kAWarps][kWT / 32];
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  float* acc = acc_all[warp];
  uint32_t* touched = touched_all[warp];
  const bool g_vec = (reinterpret_cast<uintptr_t>(G) & 15u) == 0;
  const int64_t nw = (int64_t)gridDim.x * kAWarps;
  for (int64_t t = (int64_t)blockIdx.x * kAWarps + warp; t < a.ntiles; t += nw) {
    const int64_t t0 = t * kWT;
    const int tlen = (int)min((int64_t)kWT, a.n - t0);
    // run bounds of workers `lane` and `lane + 32`
    uint32_t lo0 = 0, hi0 = 0, lo1 = 0, hi1 = 0;
    if ((int)lane < a.W) run_of(a, start, lane, t, &lo0, &hi0);
    if ((int)lane + 32 < a.W) run_of(a, start, lane + 32, t, &lo1, &hi1);
    const bool any = __any_sync(kFull, hi0 > lo0 || hi1 > lo1);
    // The dense tile of G is written as zeros first: those stores depend on
    // nothing, so they stream while the tile's entries are fetched.  The
    // touched slots are overwritten with their sums at the end.
    const bool g_full = G && g_vec && tlen == kWT;
    if (G) {
      float* gt = G + t0;
      if (g_full) {
#pragma unroll
        for (int r = 0; r < kWT / 128; ++r)
          __stcs(reinterpret_cast<float4*>(gt) + r * 32 + lane, make_float4(0.f, 0.f, 0.f, 0.f));
      } else {
        for (int i = lane; i < tlen; i += 32) gt[i] = 0.0f;
      }
    }
    if (!any) continue;
    float4* acc4 = reinterpret_cast<float4*>(acc);
#pragma unroll
    for (int r = 0; r < kWT / 128; ++r) acc4[r * 32 + lane] = make_float4(0.f, 0.f, 0.f, 0.f);
    touched[lane] = 0;
    __syncwarp();
    if (any) {
      for (int wb = 0; wb < a.W; wb += kPre) {
        if (!kBitmap) {
          // the first 32 entries of every worker's run, loaded at once
          int32_t ix[kPre];
          float vx[kPre];
          bool ok[kPre];
#pragma unroll
          for (int u = 0; u < kPre; ++u) {
            const int w = wb + u;
            const int src = w & 31;
            const uint32_t l = __shfl_sync(kFull, w < 32 ? lo0 : lo1, src);
            const uint32_t h = __shfl_sync(kFull, w < 32 ? hi0 : hi1, src);
            // int32 packets have k <= 2^31, so these sums cannot wrap
            const uint32_t j = l + lane;
            ok[u] = w < a.W && j < h;
            ix[u] = ok[u] ? a.indices[w][j] : 0;
            vx[u] = ok[u] ? a.values[w][j] : 0.0f;
          }
          // added strictly in worker order; a run longer than 32 entries is
          // finished before the next worker starts
#pragma unroll
          for (int u = 0; u < kPre; ++u) {
            const int w = wb + u;
            if (w >= a.W) break;  // warp-uniform
            const int64_t slot = (int64_t)ix[u] - t0;
            if (ok[u] && slot >= 0 && slot < tlen) {
              acc[slot] = __fadd_rn(acc[slot], vx[u]);
              atomicOr(&touched[slot >> 5], 1u << (slot & 31));
            }
            __syncwarp();
            const int src = w & 31;
            const uint32_t l = __shfl_sync(kFull, w < 32 ? lo0 : lo1, src);
            const uint32_t h = __shfl_sync(kFull, w < 32 ? hi0 : hi1, src);
            for (uint32_t off = 32; l + off < h; off += 32) {
              const uint32_t j = l + off + lane;
              if (j < h) {
                const int64_t sl = (int64_t)a.indices[w][j] - t0;
                if (sl >= 0 && sl < tlen) {
                  acc[sl] = __fadd_rn(acc[sl], a.values[w][j]);
                  atomicOr(&touched[sl >> 5], 1u << (sl & 31));
                }
              }
              __syncwarp();
            }
          }
        } else {
          uint32_t word[kPre];
          const int64_t wi = t0 / 32 + lane;
#pragma unroll
          for (int u = 0; u < kPre; ++u) {
            const int w = wb + u;
            word[u] = 0;
            if (w < a.W && (int)lane * 32 < tlen) {
              word[u] = __ldg(a.bitmaps[w] + wi);
              const int rem = tlen - (int)lane * 32;
              if (rem < 32) word[u] &= (1u << rem) - 1u;
            }
          }
#pragma unroll
          for (int u = 0; u < kPre; ++u) {
            const int w = wb + u;
            if (w >= a.W) break;  // warp-uniform
            const int src = w & 31;
            const int64_t l = __shfl_sync(kFull, w < 32 ? lo0 : lo1, src);
            const int64_t h = __shfl_sync(kFull, w < 32 ? hi0 : hi1, src);
            const uint32_t c = __popc(word[u]);
            int64_t j = l + (int64_t)(warp_incl_scan(c) - c);
            uint32_t wd = word[u];
            touched[lane] |= wd;
            while (wd) {
              const int bpos = __ffs(wd) - 1;
              wd &= wd - 1;
              if (j < h)
                acc[lane * 32 + bpos] = __fadd_rn(acc[lane * 32 + bpos], a.values[w][j]);
              ++j;
            }
            __syncwarp();
          }
        }
      }
    }
    __syncwarp();  // orders this warp's zero stores before the sums below
    uint32_t tw = touched[lane];
    while (tw) {
      const int bpos = __ffs(tw) - 1;
      tw &= tw - 1;
      const int slot = lane * 32 + bpos;
      const int64_t i = t0 + slot;
      if (G) G[i] = acc[slot];
      wts[i] = __fsub_rn(wts[i], __fmul_rn(a.eta, acc[slot]));
    }
    __syncwarp();
  }
}

int64_t agg_tiles(int64_t n) { return (n + kWT - 1) / kWT; }

int64_t agg_chunks(int64_t n) { return (agg_tiles(n) + kScanTiles - 1) / kScanTiles; }

// Workspace: status header | run boundaries uint32[W][tiles + 1] | (bitmap
// packets) ticket word, 256 bytes | look-back states uint64[W][chunks].
size_t agg_bytes(int32_t W, int32_t idx_format, int64_t n) {
  const int64_t nt = agg_tiles(n);
  size_t off = sizeof(WsHeader);
  off = round_up(off + (size_t)W * (nt + 1) * 4, 256);
  if (idx_format == EF_IDX_BITMAP) off = round_up(off + 256 + (size_t)W * agg_chunks(n) * 8, 256);
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
    if (k < 0 || k > n || k > (int64_t)0xFFFFFFFF) return EF_ERR_K;
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
  uint32_t* start = reinterpret_cast<uint32_t*>(ws + sizeof(WsHeader));
  const int64_t nt = a.ntiles;
  if (!bitmap) {
    const int64_t work = std::max<int64_t>(a.kbase[W], (int64_t)W * (nt + 1));
    const int grid = (int)std::max<int64_t>(
        1, std::min<int64_t>((work + kAThreads - 1) / kAThreads, (int64_t)dev.sms * 8));
    agg_starts_int32<<<grid, kAThreads, 0, s>>>(a, start, status);
    if ((st = check_launch()) != EF_OK) return st;
  } else {
    char* ctl = ws + round_up(sizeof(WsHeader) + (size_t)W * (nt + 1) * 4, 256);
    const size_t ctl_bytes = 256 + (size_t)W * agg_chunks(n) * 8;
    err = cudaMemsetAsync(ctl, 0, ctl_bytes, s);
    if (err != cudaSuccess) return cuda_fail(err);
    const int grid = (int)std::max<int64_t>(
        1, std::min<int64_t>((int64_t)W * agg_chunks(n), (int64_t)dev.sms * 4));
    agg_bitmap_starts<<<grid, kAThreads, 0, s>>>(a, start, reinterpret_cast<uint64_t*>(ctl + 256),
                                                 reinterpret_cast<uint32_t*>(ctl), status);
    if ((st = check_launch()) != EF_OK) return st;
  }
  const int grid = (int)std::max<int64_t>(
      1, std::min<int64_t>((nt + kAWarps - 1) / kAWarps, (int64_t)dev.sms * 6));
  prof_begin(EF_KERNEL_SPARSE_APPLY, s);
  if (bitmap)
    agg_apply<true><<<grid, kAThreads, 0, s>>>(a, start, G, w);
  else
    agg_apply<false><<<grid, kAThreads, 0, s>>>(a, start, G, w);
  if ((st = check_launch()) != EF_OK) return st;
  prof_end(EF_KERNEL_SPARSE_APPLY, s);
  return EF_OK;
}
