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
  pdl_wait();
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
  pdl_wait();
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
    // a tile.  Eight groups are loaded before any is counted.
    const bool v16 = (reinterpret_cast<uintptr_t>(bm) & 15u) == 0;
    for (int i0 = warp * 32; i0 < ntl; i0 += kAWarps * 32) {
      uint4 q[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int tile = i0 + u * 4 + (int)(lane >> 3);
        const int64_t wi = (t0 + tile) * (kWT / 32) + (lane & 7) * 4;
        q[u] = make_uint4(0u, 0u, 0u, 0u);
        if (tile < ntl) {
          if (v16 && wi + 4 <= nwords) {
            q[u] = __ldg(reinterpret_cast<const uint4*>(bm + wi));
          } else {
            if (wi < nwords) q[u].x = __ldg(bm + wi);
            if (wi + 1 < nwords) q[u].y = __ldg(bm + wi + 1);
            if (wi + 2 < nwords) q[u].z = __ldg(bm + wi + 2);
            if (wi + 3 < nwords) q[u].w = __ldg(bm + wi + 3);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint32_t v = __popc(q[u].x) + __popc(q[u].y) + __popc(q[u].z) + __popc(q[u].w);
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

// One tile by the general method: every worker's run bounds, the tile's
// zeros, then the runs' entries of up to kPre workers at once, added worker
// by worker into a shared dense copy of the tile (no atomics on values;
// indices inside one packet are distinct); touched slots get their sums in G
// and their SGD update in w.  Its loads wait on one another (bounds, then
// entries, then w).
template <bool kBitmap>
__device__ __forceinline__ void tile_general(const AggArgs& a, const uint32_t* start, int64_t t,
                                             float* G, float* wts, bool g_vec, float* acc,
                                             uint32_t* touched, unsigned lane) {
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
  if (!any) return;
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

// General apply: one tile per warp at a time (48 tiles in flight per SM).
template <bool kBitmap>
__global__ void __launch_bounds__(kAThreads, 6)
agg_apply(AggArgs a, const uint32_t* start, float* __restrict__ G, float* __restrict__ wts) {
  pdl_wait();
  __shared__ __align__(16) float acc_all[kAWarps][kWT];
  __shared__ uint32_t touched_all[kAWarps][kWT / 32];
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  const bool g_vec = (reinterpret_cast<uintptr_t>(G) & 15u) == 0;
  const int64_t nw = (int64_t)gridDim.x * kAWarps;
  for (int64_t t = (int64_t)blockIdx.x * kAWarps + warp; t < a.ntiles; t += nw)
    tile_general<kBitmap>(a, start, t, G, wts, g_vec, acc_all[warp], touched_all[warp], lane);
}

// ---------------------------------------------------------------------------
// Pipelined apply for the common case: few workers and at most 32 packet
// entries in a tile, so that lane e holds entry e of the tile (entries in
// worker-major order).  A warp walks its tiles j = 0, 1, ... and in step j
// issues the loads of later tiles while it finishes tile j:
//   int32 packets:  run bounds of tile j+3, entries of tile j+2 (from the
//                   bounds loaded in the previous step), w at the slots of
//                   tile j+1 (from the entries loaded in the previous step);
//   bitmap packets: run bounds and bitmap words of tile j+2, values and w of
//                   tile j+1;
// so no step waits on a load issued in the same step.  Finishing tile j
// stores its zeros, groups the lanes holding the same slot
// (__match_any_sync: at most one lane per worker, in worker order), and the
// lowest lane of each group adds the group's values in lane order onto +0
// and writes G and the SGD update of w.  A tile with more than 32 entries is
// done by tile_general instead.
// ---------------------------------------------------------------------------

constexpr int kPipeMaxW = 32;       // int32 packets: one lane per worker's run bounds
constexpr int kPipeMaxWBitmap = 4;  // bitmap packets: bitmap words of 4 workers per lane

struct Bounds {
  uint32_t lo, hi;  // run of worker `lane` in the tile (zero for lane >= W)
};

struct Entry {
  int32_t ix;    // packet index (int32 stages), then slot in the tile or -1
  float v;
  bool fast;     // warp-uniform: the tile has at most 32 entries
};

__device__ __forceinline__ Bounds pipe_bounds(const AggArgs& a, const uint32_t* start, int64_t t,
                                              bool valid, unsigned lane) {
  Bounds b{0u, 0u};
  if (valid && (int)lane < a.W) run_of(a, start, lane, t, &b.lo, &b.hi);
  return b;
}

// Entry `lane` of the tile from the run bounds: its worker is the last w
// whose list offset is <= lane (a worker with an empty run is never last).
__device__ __forceinline__ Entry pipe_entries_int32(const AggArgs& a, Bounds b, unsigned lane) {
  Entry e{0, 0.0f, true};
  const uint32_t len = min(b.hi - b.lo, 33u);
  const uint32_t incl = warp_incl_scan(len);
  const uint32_t E = __shfl_sync(kFull, incl, 31);
  e.fast = E <= 32u;
  if (!e.fast) return e;
  const uint32_t roff = incl - len;
  int myw = 0;
  for (int w = 1; w < a.W; ++w)
    if (__shfl_sync(kFull, roff, w) <= lane) myw = w;
  const uint32_t ro = __shfl_sync(kFull, roff, myw);
  const uint32_t lo = __shfl_sync(kFull, b.lo, myw);
  e.ix = -1;
  if (lane < E) {
    const uint32_t j = lo + (lane - ro);
    e.ix = a.indices[myw][j];
    e.v = a.values[myw][j];
  }
  return e;
}

// Turns the packet index into a slot of tile t (or -1) and loads w there.
__device__ __forceinline__ float pipe_w_int32(const AggArgs& a, const float* wts, int64_t t,
                                              Entry* e) {
  if (!e->fast) return 0.0f;
  const int64_t t0 = t * kWT;
  const int tlen = (int)min((int64_t)kWT, a.n - t0);
  const int64_t sl = (e->ix < 0) ? -1 : (int64_t)e->ix - t0;
  e->ix = (sl >= 0 && sl < tlen) ? (int32_t)sl : -1;
  return e->ix >= 0 ? wts[t0 + e->ix] : 0.0f;
}

struct BitmapStage {
  Bounds b;
  uint32_t word[kPipeMaxWBitmap];  // word `lane` of the tile, per worker
};

__device__ __forceinline__ BitmapStage pipe_bitmap_load(const AggArgs& a, const uint32_t* start,
                                                        int64_t t, bool valid, unsigned lane) {
  BitmapStage s;
  s.b = pipe_bounds(a, start, t, valid, lane);
  const int tlen = valid ? (int)min((int64_t)kWT, a.n - t * kWT) : 0;
#pragma unroll
  for (int w = 0; w < kPipeMaxWBitmap; ++w) {
    s.word[w] = 0u;
    if (w < a.W && (int)lane * 32 < tlen) {
      s.word[w] = __ldg(a.bitmaps[w] + t * (kWT / 32) + lane);
      const int rem = tlen - (int)lane * 32;
      if (rem < 32) s.word[w] &= (1u << rem) - 1u;
    }
  }
  return s;
}

// Entry `lane` of the tile from the bitmap words: the r-th set bit of worker
// w is entry r of its run (bits past the run's length, possible only in a
// malformed packet, are dropped); then its value and w at its slot.
__device__ __forceinline__ Entry pipe_bitmap_entries(const AggArgs& a, const float* wts,
                                                     const BitmapStage& s, int64_t t,
                                                     uint32_t* lst, unsigned lane, float* wv) {
  Entry e{-1, 0.0f, true};
  *wv = 0.0f;
  const uint32_t len = min(s.b.hi - s.b.lo, 33u);
  const uint32_t incl = warp_incl_scan(len);
  const uint32_t E = __shfl_sync(kFull, incl, 31);
  e.fast = E <= 32u;
  if (!e.fast) return e;
  const uint32_t roff = incl - len;
  lst[lane] = 0xFFFFFFFFu;
  __syncwarp();
#pragma unroll
  for (int w = 0; w < kPipeMaxWBitmap; ++w) {
    if (w >= a.W) break;  // warp-uniform
    const uint32_t c = __popc(s.word[w]);
    uint32_t r = warp_incl_scan(c) - c;
    const uint32_t base = __shfl_sync(kFull, roff, w), ln = __shfl_sync(kFull, len, w);
    uint32_t x = s.word[w];
    while (x) {
      const int bpos = __ffs(x) - 1;
      x &= x - 1;
      if (r < ln) lst[base + r] = (lane * 32u + (uint32_t)bpos) | ((uint32_t)w << 16);
      ++r;
    }
  }
  __syncwarp();
  const uint32_t code = lst[lane];
  const bool ok = lane < E && code != 0xFFFFFFFFu;
  const int myw = ok ? (int)(code >> 16) : 0;
  const uint32_t ro = __shfl_sync(kFull, roff, myw);
  const uint32_t lo = __shfl_sync(kFull, s.b.lo, myw);
  if (ok) {
    e.ix = (int32_t)(code & 0xFFFFu);
    e.v = a.values[myw][lo + (lane - ro)];
    *wv = wts[t * kWT + e.ix];
  }
  __syncwarp();
  return e;
}

// Finishes a tile whose entries, slots and w values are in the lanes.  The
// tile of G is assembled in the warp's shared copy (zeros, then each slot's
// sum) and stored once with 16-byte stores: no slot is written twice, so no
// partial sector ever reaches DRAM.
__device__ __forceinline__ void pipe_finish(const AggArgs& a, int64_t t, const Entry& e, float wv,
                                            float* G, float* wts, bool g_vec, float* vbuf,
                                            float* acc, unsigned lane) {
  const int64_t t0 = t * kWT;
  const int tlen = (int)min((int64_t)kWT, a.n - t0);
  float4* acc4 = reinterpret_cast<float4*>(acc);
  if (G) {
#pragma unroll
    for (int r = 0; r < kWT / 128; ++r) acc4[r * 32 + lane] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const unsigned grp = __match_any_sync(kFull, e.ix >= 0 ? e.ix : kWT + (int)lane);
  vbuf[lane] = e.v;
  __syncwarp();
  if (e.ix >= 0 && (int)lane == __ffs(grp) - 1) {
    float sum = __fadd_rn(0.0f, e.v);
    unsigned m = grp & (grp - 1);
    while (m) {
      const int i = __ffs(m) - 1;
      m &= m - 1;
      sum = __fadd_rn(sum, vbuf[i]);
    }
    if (G) acc[e.ix] = sum;
    wts[t0 + e.ix] = __fsub_rn(wv, __fmul_rn(a.eta, sum));
  }
  __syncwarp();
  if (G) {
    float* gt = G + t0;
    if (g_vec && tlen == kWT) {
#pragma unroll
      for (int r = 0; r < kWT / 128; ++r)
        __stcs(reinterpret_cast<float4*>(gt) + r * 32 + lane, acc4[r * 32 + lane]);
    } else {
      for (int i = lane; i < tlen; i += 32) gt[i] = acc[i];
    }
  }
  __syncwarp();  // the shared copy is reused by the next tile
}

template <bool kBitmap>
__global__ void __launch_bounds__(kAThreads, 5)
agg_apply_pipe(AggArgs a, const uint32_t* start, float* __restrict__ G, float* __restrict__ wts) {
  pdl_wait();
  __shared__ __align__(16) float acc_all[kAWarps][kWT];
  __shared__ uint32_t touched_all[kAWarps][kWT / 32];
  __shared__ float vbuf_all[kAWarps][32];
  __shared__ uint32_t lst_all[kAWarps][32];
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  const bool g_vec = (reinterpret_cast<uintptr_t>(G) & 15u) == 0;
  const int64_t first = (int64_t)blockIdx.x * kAWarps + warp;
  const int64_t nw = (int64_t)gridDim.x * kAWarps;
  if (first >= a.ntiles) return;
  const int64_t cnt = (a.ntiles - 1 - first) / nw + 1;  // tiles of this warp
  float* vbuf = vbuf_all[warp];
  auto finish = [&](int64_t j, const Entry& e, float wv) {
    const int64_t t = first + j * nw;
    if (e.fast)
      pipe_finish(a, t, e, wv, G, wts, g_vec, vbuf, acc_all[warp], lane);
    else
      tile_general<kBitmap>(a, start, t, G, wts, g_vec, acc_all[warp], touched_all[warp], lane);
  };
  if (!kBitmap) {
    const Bounds b0 = pipe_bounds(a, start, first, true, lane);
    Bounds b1 = pipe_bounds(a, start, first + nw, 1 < cnt, lane);
    Entry e0 = pipe_entries_int32(a, b0, lane);
    Bounds b2 = pipe_bounds(a, start, first + 2 * nw, 2 < cnt, lane);
    Entry e1 = pipe_entries_int32(a, b1, lane);
    float w0 = pipe_w_int32(a, wts, first, &e0);
    for (int64_t j = 0; j < cnt; ++j) {
      const Bounds b3 = pipe_bounds(a, start, first + (j + 3) * nw, j + 3 < cnt, lane);
      const Entry e2 = pipe_entries_int32(a, b2, lane);
      const float w1 = pipe_w_int32(a, wts, first + (j + 1) * nw, &e1);
      finish(j, e0, w0);
      e0 = e1;
      w0 = w1;
      e1 = e2;
      b2 = b3;
    }
  } else {
    uint32_t* lst = lst_all[warp];
    const BitmapStage s0 = pipe_bitmap_load(a, start, first, true, lane);
    BitmapStage s1 = pipe_bitmap_load(a, start, first + nw, 1 < cnt, lane);
    float w0;
    Entry e0 = pipe_bitmap_entries(a, wts, s0, first, lst, lane, &w0);
    for (int64_t j = 0; j < cnt; ++j) {
      const BitmapStage s2 = pipe_bitmap_load(a, start, first + (j + 2) * nw, j + 2 < cnt, lane);
      float w1;
      const Entry e1 = pipe_bitmap_entries(a, wts, s1, first + (j + 1) * nw, lst, lane, &w1);
      finish(j, e0, w0);
      e0 = e1;
      w0 = w1;
      s1 = s2;
    }
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
    launch_pdl(agg_starts_int32, grid, kAThreads, 0, s, a, start, status);
    if ((st = check_launch()) != EF_OK) return st;
  } else {
    char* ctl = ws + round_up(sizeof(WsHeader) + (size_t)W * (nt + 1) * 4, 256);
    const size_t ctl_bytes = 256 + (size_t)W * agg_chunks(n) * 8;
    err = cudaMemsetAsync(ctl, 0, ctl_bytes, s);
    if (err != cudaSuccess) return cuda_fail(err);
    const int grid = (int)std::max<int64_t>(
        1, std::min<int64_t>((int64_t)W * agg_chunks(n), (int64_t)dev.sms * 5));
    launch_pdl(agg_bitmap_starts, grid, kAThreads, 0, s, a, start, reinterpret_cast<uint64_t*>(ctl + 256),
                                                 reinterpret_cast<uint32_t*>(ctl), status);
    if ((st = check_launch()) != EF_OK) return st;
  }
  const bool pipe = bitmap ? W <= kPipeMaxWBitmap : W <= kPipeMaxW;
  const int grid = (int)std::max<int64_t>(
      1, std::min<int64_t>((nt + kAWarps - 1) / kAWarps, (int64_t)dev.sms * (pipe ? 5 : 6)));
  prof_begin(EF_KERNEL_SPARSE_APPLY, s);
  if (bitmap && pipe)
    launch_pdl(agg_apply_pipe<true>, grid, kAThreads, 0, s, a, start, G, w);
  else if (bitmap)
    launch_pdl(agg_apply<true>, grid, kAThreads, 0, s, a, start, G, w);
  else if (pipe)
    launch_pdl(agg_apply_pipe<false>, grid, kAThreads, 0, s, a, start, G, w);
  else
    launch_pdl(agg_apply<false>, grid, kAThreads, 0, s, a, start, G, w);
  if ((st = check_launch()) != EF_OK) return st;
  prof_end(EF_KERNEL_SPARSE_APPLY, s);
  return EF_OK;
}
