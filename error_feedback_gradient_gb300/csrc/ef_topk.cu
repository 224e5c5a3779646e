// Top-k error feedback, sender side ("梯度稀疏化：只传输重要的梯度元素",
// §详细算法流程 steps 2-5, per tensor as §分层自适应Top-k describes):
//   g = g_raw + e;  S = k largest |g| (ties -> lower index);
//   e' = g off S, +0 on S;  packet = (g[i], i) for i in S, ascending i.
//
// Segments of at most kSmallMax elements are finished by one CTA each with
// the whole segment in shared memory: compensate, one pass over the top 11
// key bits, then either a direct rank of the few keys at or above the k-th
// key's bin (at most kSmallRank of them) or the 3-digit radix select and
// the ordered emit.  Longer segments take the streaming path, batched over
// the streaming segments of a call:
//   1. sample   (up to 128 CTAs per segment): up to 4096 blocks of 64
//      contiguous elements (at most 1/16 of the segment, each in the middle
//      of one of as many equal slots) are compensated, and a histogram of
//      their keys gives a conservative lower threshold T_lo.  In a compact
//      batch (below) one pass over the top 13 key bits, T_lo = the lower
//      edge of the 13-bit bin holding the rank-th largest sampled key; in
//      other batches two short passes (top 11 bits, then the next 10 inside
//      the chosen bin), T_lo = the lower edge of that 21-bit bin.  Only a
//      speed-up: the result never depends on it.
//   2. fused    (the HBM pass, 12 B / element): g = g_raw + e written over e,
//      except that a key >= T_lo is written as +0 and appended, in index
//      order, to a per-segment candidate list (warp ballots and a bounded
//      decoupled look-back; in a compact batch the look-back reads 128 tile
//      states per round trip and publishes them by atomic exchange).  A
//      warp's span whose candidates overflow its staging buffer is rescanned
//      from L2 by the scan warp, so the list stays complete; a candidate past
//      the list's capacity keeps g in e.  Each list is then checked: between
//      k and its capacity -> select on the list; otherwise (T_lo too high,
//      or the list over capacity) -> select on the whole segment, which is
//      always correct, only slower, once g is back in e at the listed
//      candidates.  (In other batches the last CTA records this; in a
//      compact batch the finish derives it.)
// A compact batch (every list expected to fit kFinishCap entries, as for
// the tensors of a layerwise model) ends with
//   3c. finish  one thread-block cluster per segment selects on its list
//      and emits it, the list spread over the cluster's shared memory; the
//      select takes two digit passes counted from T_lo (d0 = (key - T_lo)
//      >> 11 capped at 1023, then the low 11 bits), or three from the top
//      bits if the k-th key lies far above T_lo.
// The call's small segments run as extra CTAs of the first batch's sampling
// launch, in the shadow of the sampling.
// Other batches end with
//   3. restore, then select (x3): radix select on 11/10/10-bit digits of the
//      keys of each list, shared-memory histograms merged into one per
//      segment; the last CTA of each pass fixes that digit (lists of at most
//      kSelSmall entries are resolved by one CTA first).  Result: the k-th
//      key T and need = k - #(key > T).
//   4. emit     ordered compaction of the list: an entry is taken when
//      key > T, or key == T and fewer than `need` equal keys precede it;
//      position = #(key > T before it) + min(#(key == T before it), need).
//      The look-back carries (#gt, #lt) prefixes: both stay below 2^31 for a
//      list of up to 2^31 entries (T itself is in the list), and the equal
//      count follows from the list position j as j - gt - lt.
//      Writes values, int32 indices or bitmap bits.  On a candidate list e
//      already holds +0 at every candidate, so emit writes g back at the
//      candidates not taken (with a tight T_lo far fewer than k scattered
//      writes); on a whole-segment list it writes e = +0 at the taken ones.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <climits>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <vector>

#include "ef_common.cuh"
#include "ef_lookback.cuh"
#include "ef_topk_internal.h"

namespace ef {
namespace {

// Segments of at most kSmallMax elements are finished by one CTA from the
// whole segment; longer ones are sampled and finished from their candidate
// list, which for a one-CTA finish costs far less than the segment itself
// (a 32768-element segment at k = 1 % lists about 500 candidates).
constexpr int kSmallMax = 4096;
constexpr int kSmallThreads = 1024;
constexpr int kStreamWarps = 8;                 // fused pass: warps that stream the tile
constexpr int kWarpSpan = 4096;                 // elements per streaming warp per tile
// The fused pass picks its tile per batch among 32768, 16384 and 8192
// elements: the one with the least rounds of the persistent grid times
// (tile + kTileCost), kTileCost standing for a tile's fixed cost (ticket,
// barriers, look-back) in elements; ties go to the longer tile.  (4096-element
// tiles measured slower wherever the rule would pick them: the 2^20-element
// call 42.8 against 38.8 us with 8192, their look-back chains twice as long.)
constexpr int kWarpSpanMid = 2048;
constexpr int kWarpSpanSmall = 1024;
constexpr int kTileSmall = kStreamWarps * kWarpSpanSmall;
constexpr int64_t kTileCost = 4096;
constexpr int kStreamThreads = kStreamWarps * 32;
constexpr int kFusedThreads = kStreamThreads + 32;  // + one scan warp
constexpr int kStageCap = 256;                  // staged candidates per warp per buffer
constexpr int kBatch = 4;                       // 128-element rounds loaded at once
constexpr int kFusedCtasPerSm = 4;
constexpr int kSampleBlock = 64;         // contiguous elements per sample block
constexpr int kSampleBlocksMax = 4096;  // sample blocks per segment (262 144 keys)
constexpr int kChunk = 4096;  // list entries per select / emit chunk
constexpr int kSelThreads = 512;
constexpr int kEmitThreads = 256;  // 8 warps x 16 rounds x 32 lanes = kChunk
constexpr int kMaxLarge = 128;     // segments per streaming batch
constexpr int kMaxSmall = 512;     // segments per small-path launch
constexpr uint32_t kNoCandidate = 0x80000000u;  // above every 31-bit key
constexpr int kSelSmall = 32768;  // lists up to this length are selected by one CTA
// Compact batches: every streaming segment is at most kCompactLen elements
// and its expected candidate list at most half of kFinishCap entries, so one
// CTA finishes it in shared memory (topk_finish) and the three digit passes
// and the look-back emit are not launched.
constexpr int kFinishCap = kSelSmall;
constexpr int64_t kCompactLen = int64_t(1) << 22;

static_assert(kWarpSpan % (128 * kBatch) == 0, "tile layout");
static_assert(kWarpSpanMid % (128 * kBatch) == 0, "tile layout");
static_assert(kWarpSpanSmall % (128 * kBatch) == 0, "tile layout");
static_assert(kEmitThreads / 32 * 16 * 32 == kChunk, "emit layout");
static_assert(kChunk % kSelThreads == 0, "select layout");

struct SmallSeg {
  int64_t off;
  int64_t out_off;
  int32_t len;
  int32_t k;
};

struct SmallBatch {
  SmallSeg seg[kMaxSmall];
};

struct LargeSeg {
  int64_t off, len, k, out_off;
  int64_t cand_base, cap;
  int64_t tile_base;  // global id of the segment's first fused tile
  int64_t q_first;    // index of that tile in aligned units of the pass's tile
  int64_t rank;       // sample rank for T_lo (0: no candidates, > samples: all)
};

struct LargeBatch {
  LargeSeg seg[kMaxLarge];
};

// CTAs of the two sampling passes: segment s owns CTAs [base[s], base[s+1]),
// enough for one round of sample loads per warp (kMaxLarge segments).
struct SampleGrid {
  int32_t base[kMaxLarge + 1];
};

struct SegState {
  LargeSeg d;
  uint32_t t_lo;
  uint32_t mode;  // 0: select on candidates, 1: select on the whole segment
  int64_t list_len;
  int64_t chunk_base;
  uint32_t prefix;  // radix-select digits fixed so far (= T after pass 3)
  uint32_t krem;    // rank still to find inside the prefix (= need)
  uint32_t gt;
  uint32_t overflow;  // a warp's staging area overflowed: the list is incomplete
  uint32_t resolved;  // T and need already found (list fitted in one CTA)
  uint32_t chunks_done[3];  // chunks of the list histogrammed per digit pass
  int64_t cand_count;       // candidates found by the fused pass (-1: unknown)
};

// Per-segment state of the sampling passes (in the cleared control area).
struct SampleState {
  uint32_t done[2];  // CTAs finished in the first / second pass
  uint32_t b0;       // two-pass form: top-11-bit bin holding the rank-th sampled key
  uint32_t r1;       // that key's rank inside the bin
};

// Sample blocks of a segment of `len` elements (> kSmallMax): at most 1/16
// of the segment, at most kSampleBlocksMax.
__host__ __device__ __forceinline__ int64_t sample_blocks(int64_t len) {
  const int64_t b = len / (16 * kSampleBlock);
  return b < kSampleBlocksMax ? b : kSampleBlocksMax;
}

// The segment is cut into nblk equal slots of spacing = floor(len / nblk)
// (>= 1024) elements; sample block b sits in the middle of slot b.
__host__ __device__ __forceinline__ int64_t sample_block_start(int64_t spacing, int64_t b) {
  return b * spacing + (spacing - kSampleBlock) / 2;
}

struct alignas(256) Ctl {
  uint32_t fused_ticket, fused_done;
  uint32_t emit_ticket;
  int64_t total_chunks;
};

struct IO {
  const float* g_raw;
  float* e;
  float* out_values;
  int32_t* out_indices;
  uint32_t* out_bitmap;
  int32_t* status;
  uint32_t* pos_out;  // optional: each packet entry's position inside its segment
};

// Writes packet entry `pos` (must lie below `limit`, the segment's packet end;
// anything else would be a library defect and is recorded, not written) for
// element gidx (local index lidx in its segment), and e = +0 at the element
// unless it already holds +0 (zero_e false).
__device__ __forceinline__ void emit_one(const IO& io, int64_t gidx, int64_t lidx, int64_t pos,
                                         int64_t limit, float v, bool zero_e) {
  if (pos >= limit) {
    set_status(io.status, EF_ERR_INTERNAL);
    return;
  }
  io.out_values[pos] = v;
  if (io.out_indices) io.out_indices[pos] = (int32_t)gidx;
  if (io.pos_out) io.pos_out[pos] = (uint32_t)lidx;
  if (io.out_bitmap) atomicOr(io.out_bitmap + (gidx >> 5), 1u << (gidx & 31));
  if (zero_e) io.e[gidx] = 0.0f;
}

// Ordered emit by one CTA over a list of n entries whose k-th key T and tie
// count `need` are known: an entry is taken when key > T, or key == T and
// fewer than `need` equal keys precede it; its packet position is
// #(key > T before it) + min(#(key == T before it), need).  Warp w owns the
// contiguous range [w * span, (w + 1) * span) of the CTA's entries.
// block_count: one pass counts (greater, equal) per warp into shm[0..31] and
// shm[32..63] and returns the CTA's totals.  block_emit: a scan of the warp
// counts, on top of `base_gt` / `base_eq` (the entries before this CTA's,
// when several CTAs share a list), gives each warp its offsets, and a second
// pass emits with ballots.  `bits_at(j)` gives entry j's float bits,
// `loc_at(j)` its local index in the segment.  On a candidate list
// (`on_list`) e already holds +0 at every entry, so the entries not taken get
// their value back in e; otherwise e is set to +0 at the taken entries.
// Eight entries per lane are loaded before any is counted.
constexpr int kRound = 8 * 32;

__device__ __forceinline__ void warp_span(int n, int* w0, int* w1) {
  const int nwarps = blockDim.x >> 5;
  const int span = ((n + nwarps - 1) / nwarps + kRound - 1) / kRound * kRound;
  *w0 = (int)min((int64_t)(threadIdx.x >> 5) * span, (int64_t)n);
  *w1 = (int)min((int64_t)*w0 + span, (int64_t)n);
}

template <typename BitsAt>
__device__ __forceinline__ uint2 block_count(int n, uint32_t T, uint32_t* shm, BitsAt bits_at) {
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  int w0, w1;
  warp_span(n, &w0, &w1);
  uint32_t cg = 0, ce = 0;
  for (int b = w0; b < w1; b += kRound) {
    uint32_t v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = b + u * 32 + (int)lane;
      v[u] = j < w1 ? bits_at(j) : 0u;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = b + u * 32 + (int)lane;
      const uint32_t key = v[u] & 0x7FFFFFFFu;
      cg += j < w1 && key > T;
      ce += j < w1 && key == T;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    cg += __shfl_xor_sync(kFull, cg, o);
    ce += __shfl_xor_sync(kFull, ce, o);
  }
  if (lane == 0) {
    shm[warp] = cg;
    shm[32 + warp] = ce;
  }
  __syncthreads();
  uint32_t tg = 0, te = 0;
  for (int w = 0; w < nwarps; ++w) {
    tg += shm[w];
    te += shm[32 + w];
  }
  return make_uint2(tg, te);
}

template <typename BitsAt, typename LocAt>
__device__ __forceinline__ void block_emit(const IO& io, int n, uint32_t T, uint32_t need,
                                           uint32_t base_gt, uint32_t base_eq, int64_t seg_off,
                                           int64_t out_off, int64_t k, bool on_list,
                                           uint32_t* shm, BitsAt bits_at, LocAt loc_at) {
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  int w0, w1;
  warp_span(n, &w0, &w1);
  __syncthreads();  // every thread has read the warp counts (block_count)
  uint32_t* wgt = shm;
  uint32_t* weq = shm + 32;
  if (warp == 0) {
    const uint32_t g = lane < (unsigned)nwarps ? wgt[lane] : 0u;
    const uint32_t q = lane < (unsigned)nwarps ? weq[lane] : 0u;
    const uint32_t ig = warp_incl_scan(g), iq = warp_incl_scan(q);
    if (lane < (unsigned)nwarps) {
      wgt[lane] = base_gt + ig - g;
      weq[lane] = base_eq + iq - q;
    }
  }
  __syncthreads();
  uint32_t run_gt = wgt[warp], run_eq = weq[warp];
  const unsigned lm = lanemask_lt();
  for (int b = w0; b < w1; b += kRound) {
    uint32_t v[8];
    int loc[8];  // every entry's location is loaded with its bits, before any is used
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = b + u * 32 + (int)lane;
      v[u] = j < w1 ? bits_at(j) : 0u;
      loc[u] = j < w1 ? loc_at(j) : 0;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = b + u * 32 + (int)lane;
      const uint32_t key = v[u] & 0x7FFFFFFFu;
      const bool gt = j < w1 && key > T;
      const bool eq = j < w1 && key == T;
      const unsigned bg = __ballot_sync(kFull, gt), bq = __ballot_sync(kFull, eq);
      const uint32_t gt_before = run_gt + __popc(bg & lm);
      const uint32_t eq_before = run_eq + __popc(bq & lm);
      if (gt || (eq && eq_before < need)) {
        const int64_t pos = out_off + gt_before + min(eq_before, need);
        emit_one(io, seg_off + loc[u], loc[u], pos, out_off + k, __uint_as_float(v[u]),
                 !on_list);
      } else if (on_list && j < w1) {
        io.e[seg_off + loc[u]] = __uint_as_float(v[u]);
      }
      run_gt += __popc(bg);
      run_eq += __popc(bq);
    }
  }
}

template <typename BitsAt, typename LocAt>
__device__ __forceinline__ void block_ordered_emit(const IO& io, int n, uint32_t T,
                                                   uint32_t need, int64_t seg_off,
                                                   int64_t out_off, int64_t k, bool on_list,
                                                   uint32_t* shm, BitsAt bits_at, LocAt loc_at) {
  (void)block_count(n, T, shm, bits_at);
  block_emit(io, n, T, need, 0u, 0u, seg_off, out_off, k, on_list, shm, bits_at, loc_at);
}

// ---------------------------------------------------------------------------
// small segments: one CTA holds the whole segment
// ---------------------------------------------------------------------------

// Shared memory of a one-CTA select: keys_words of keys, then these.
constexpr int kSubCap = 8192;  // keys kept for the last digit pass
constexpr int kSelectExtraWords = 2048 + 64 + kSubCap;  // histogram, scratch, sub

// Keys at or above the k-th key's first-digit bin that a small segment
// ranks directly (all pairs) instead of running the last two digit passes.
constexpr int kSmallRank = 256;

// One segment of at most kSmallMax elements by one CTA: g = g_raw + e into
// e and into shared memory, then the k largest keys.  A first pass counts
// the top 11 key bits; when at most kSmallRank keys lie at or above the
// bin of the k-th key (the usual case for a small k: a layerwise model's
// small tensors at 1 %), those keys are gathered with their indices and
// each one's rank (#greater keys, and equal keys at lower indices) and
// output position (#selected at lower indices) are counted over the
// gathered set: every key not gathered is smaller than every gathered one,
// so these are the ranks in the whole segment.  Otherwise the radix select
// and the ordered emit run over the whole segment.  `sm` holds keys_words +
// 2048 + 64 + sub_cap words of shared memory.
__device__ __forceinline__ void small_segment(const SmallSeg& sg, const IO& io, uint32_t* sm,
                                              int keys_words, int sub_cap = kSubCap) {
  uint32_t* gbits = sm;
  uint32_t* hist = sm + keys_words;
  uint32_t* scratch = hist + 2048;
  uint32_t* sub = scratch + 64;
  const int len = sg.len;
  const float* gr = io.g_raw + sg.off;
  float* e = io.e + sg.off;
  // eight elements of each array in flight per thread
  for (int i0 = threadIdx.x; i0 < len; i0 += 8 * blockDim.x) {
    float gv[8], ev[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * blockDim.x;
      gv[u] = i < len ? gr[i] : 0.0f;
      ev[u] = i < len ? e[i] : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < len) {
        const float x = __fadd_rn(gv[u], ev[u]);
        e[i] = x;
        gbits[i] = __float_as_uint(x);
      }
    }
  }
  __syncthreads();
  if (sg.k == 0) return;  // uniform across the CTA
  for (int b = threadIdx.x; b < 2048; b += blockDim.x) hist[b] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < len; i += blockDim.x) hist_add(hist, (gbits[i] & 0x7FFFFFFFu) >> 20, true);
  __syncthreads();
  uint32_t b0, above0;
  block_find_bin(hist, 2048, (uint32_t)sg.k, scratch, &b0, &above0);
  const uint32_t m = above0 + hist[b0];  // keys whose first digit is >= b0
  if (m <= (uint32_t)kSmallRank && 2 * (int)m <= sub_cap) {  // uniform across the CTA
    uint32_t* gcount = scratch + 40;
    if (threadIdx.x == 0) *gcount = 0;
    __syncthreads();
    // (key, index) of every key in or above bin b0, in no particular order
    for (int i0 = 0; i0 < len; i0 += blockDim.x) {  // warp-uniform trip count
      const int i = i0 + (int)threadIdx.x;
      const uint32_t key = i < len ? gbits[i] & 0x7FFFFFFFu : 0u;
      const bool in = i < len && (key >> 20) >= b0;
      const unsigned mk = __ballot_sync(kFull, in);
      if (mk != 0u) {
        const int first = __ffs(mk) - 1;
        uint32_t base = 0;
        if ((int)(threadIdx.x & 31u) == first) base = atomicAdd(gcount, (uint32_t)__popc(mk));
        base = __shfl_sync(kFull, base, first);
        if (in) {
          const uint32_t pos = base + __popc(mk & lanemask_lt());
          sub[2 * pos] = key;
          sub[2 * pos + 1] = (uint32_t)i;
        }
      }
    }
    __syncthreads();
    uint32_t* selected = hist;  // the histogram is no longer needed
    for (int j = threadIdx.x; j < (int)m; j += blockDim.x) {
      const uint32_t kj = sub[2 * j], ij = sub[2 * j + 1];
      uint32_t rank = 0;
      for (int q = 0; q < (int)m; ++q) {
        const uint32_t kq = sub[2 * q], iq = sub[2 * q + 1];
        rank += (kq > kj || (kq == kj && iq < ij)) ? 1u : 0u;
      }
      selected[j] = rank < (uint32_t)sg.k ? 1u : 0u;
    }
    __syncthreads();
    for (int j = threadIdx.x; j < (int)m; j += blockDim.x) {
      if (!selected[j]) continue;
      const uint32_t ij = sub[2 * j + 1];
      uint32_t pos = 0;
      for (int q = 0; q < (int)m; ++q) pos += (selected[q] && sub[2 * q + 1] < ij) ? 1u : 0u;
      emit_one(io, sg.off + ij, ij, sg.out_off + pos, sg.out_off + sg.k, __uint_as_float(gbits[ij]),
               true);
    }
    return;
  }
  __syncthreads();  // every thread has read hist[b0] before the select clears it
  const SelectResult r =
      block_radix_select(gbits, len, (uint32_t)sg.k, hist, scratch, sub, sub_cap);
  block_ordered_emit(io, len, r.T, r.need, sg.off, sg.out_off, sg.k, false, scratch,
                     [gbits](int i) { return gbits[i]; }, [](int i) { return i; });
}

__global__ void __launch_bounds__(kSmallThreads)
topk_small(SmallBatch b, IO io, int keys_words) {
  pdl_wait();
  extern __shared__ uint32_t sm[];
  small_segment(b.seg[blockIdx.x], io, sm, keys_words);
}

// ---------------------------------------------------------------------------
// streaming path
// ---------------------------------------------------------------------------

constexpr int kSampleCtasMax = 128;  // CTAs per segment in each sampling pass, at most
constexpr int kSampleThreads = 256;
constexpr int kSampleUnroll = 4;     // sample blocks per warp in flight
// rounds of kSampleUnroll blocks per warp: more rounds, fewer CTAs to pay
// for zeroing and merging the histogram
constexpr int kSampleRounds = 4;
// The sampled lower threshold T_lo is the lower edge of a bin of the top 13
// key bits (8 exponent + 5 mantissa bits): a bin spans at most 1/32 of its
// value, so T_lo sits at most that far below the sampled rank's key.
constexpr int kSampleBits = 13;
constexpr int kSampleShift = 31 - kSampleBits;
constexpr int kSampleBins = 1 << kSampleBits;
// the sampling kernel's shared words: its histogram, or the whole of a small
// segment run by the same launch (keys, histogram, scratch, last-pass keys)
constexpr int kSampleSmem = kSampleBins + 2048 + 64;
static_assert(kSampleBins % (4 * kSampleThreads) == 0, "sample histogram layout");

// Compensated keys of sample blocks `bi` .. of this warp: lane l holds
// elements l and l + 32 of each block.
__device__ __forceinline__ void sample_keys(const IO& io, const LargeSeg& d, int64_t nblk,
                                            int64_t spacing, int64_t b0, int64_t stride,
                                            unsigned lane, uint32_t (&key)[kSampleUnroll][2],
                                            bool (&ok)[kSampleUnroll]) {
  float gv[kSampleUnroll][2], ev[kSampleUnroll][2];
#pragma unroll
  for (int u = 0; u < kSampleUnroll; ++u) {
    const int64_t bi = b0 + u * stride;
    ok[u] = bi < nblk;
    if (ok[u]) {
      const int64_t p = d.off + sample_block_start(spacing, bi) + lane;
      gv[u][0] = io.g_raw[p];
      gv[u][1] = io.g_raw[p + 32];
      ev[u][0] = io.e[p];
      ev[u][1] = io.e[p + 32];
    }
  }
#pragma unroll
  for (int u = 0; u < kSampleUnroll; ++u) {
    key[u][0] = ok[u] ? abs_key(__fadd_rn(gv[u][0], ev[u][0])) : 0u;
    key[u][1] = ok[u] ? abs_key(__fadd_rn(gv[u][1], ev[u][1])) : 0u;
  }
}

// Whether the segment samples at all (rank 0: no candidates; rank above the
// sample count: every element is a candidate).
__device__ __forceinline__ bool samples_needed(const LargeSeg& d, int64_t nblk) {
  return d.rank > 0 && d.rank <= nblk * kSampleBlock;
}

// Segment and CTA rank within it of sampling CTA `blk`.
__device__ __forceinline__ int sample_seg(const SampleGrid& g, int nseg, int blk, int* q,
                                          int* ctas) {
  int lo = 0, hi = nseg - 1;  // last segment whose first CTA is <= blk
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (g.base[mid] <= blk) lo = mid;
    else hi = mid - 1;
  }
  *q = blk - g.base[lo];
  *ctas = g.base[lo + 1] - g.base[lo];
  return lo;
}

__device__ __forceinline__ void init_state(SegState* st, int s, const LargeSeg& d, uint32_t t_lo) {
  SegState v;
  v.d = d;
  v.t_lo = t_lo;
  v.mode = 0;
  v.list_len = 0;
  v.chunk_base = 0;
  v.prefix = 0;
  v.krem = (uint32_t)d.k;
  v.gt = 0;
  v.overflow = 0;
  v.resolved = 0;
  v.chunks_done[0] = v.chunks_done[1] = v.chunks_done[2] = 0;
  v.cand_count = -1;
  st[s] = v;
}

// The sampling pass: a histogram of the top kSampleBits key bits over all
// sample blocks of each streaming segment (the segment's CTAs of `grid`,
// merged in global memory).  The CTA that merges last sets T_lo = the lower
// edge of the bin holding the rank-th largest sampled key (so at least
// `rank` sampled keys are >= T_lo) and the segment's state for the later
// passes.  A segment that does not sample gets its state from its one CTA.
// Small segments ride in the same launch only when a call has them
// (kSmall): the launch without them keeps the shared memory to the
// histogram and the parameters to the segment table, so that it holds as
// little as possible of the SMs that other streams' streaming passes share.
struct NoSmall {};

template <bool kSmall, typename Smalls>
__global__ void __launch_bounds__(kSampleThreads)
topk_sample(LargeBatch b, SampleGrid grid, int nseg, IO io, uint32_t* hist0, SampleState* ss,
            SegState* st, Smalls sb) {
  pdl_wait();
  __shared__ __align__(16) uint32_t sh[kSmall ? kSampleSmem : kSampleBins];
  __shared__ uint32_t scratch[64];
  __shared__ int s_last;
  if constexpr (kSmall) {
    if ((int)blockIdx.x >= grid.base[nseg]) {
      // a small segment folded into this launch: keys, histogram, scratch
      // and the last pass's keys all in `sh`
      small_segment(sb.seg[blockIdx.x - grid.base[nseg]], io, sh, kSmallMax,
                    kSampleSmem - kSmallMax - 2048 - 64);
      return;
    }
  }
  int q, ctas;
  const int s = sample_seg(grid, nseg, blockIdx.x, &q, &ctas);
  const LargeSeg d = b.seg[s];
  const int64_t nblk = sample_blocks(d.len);
  if (!samples_needed(d, nblk)) {  // uniform across the CTA
    if (q == 0 && threadIdx.x == 0) init_state(st, s, d, d.rank <= 0 ? kNoCandidate : 0u);
    return;
  }
  const int64_t spacing = d.len / nblk;
  const unsigned lane = lane_id();
  const int64_t gw = (int64_t)q * (kSampleThreads / 32) + (threadIdx.x >> 5);
  const int64_t kWarps = (int64_t)ctas * (kSampleThreads / 32);
  uint4* sh4 = reinterpret_cast<uint4*>(sh);
#pragma unroll
  for (int r = 0; r < kSampleBins / 4 / kSampleThreads; ++r)
    sh4[r * kSampleThreads + threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  for (int64_t b0 = gw; b0 < nblk; b0 += kWarps * kSampleUnroll) {  // warp-uniform
    uint32_t key[kSampleUnroll][2];
    bool ok[kSampleUnroll];
    sample_keys(io, d, nblk, spacing, b0, kWarps, lane, key, ok);
#pragma unroll
    for (int u = 0; u < kSampleUnroll; ++u) {
#pragma unroll
      for (int h = 0; h < 2; ++h) hist_add(sh, key[u][h] >> kSampleShift, ok[u]);
    }
  }
  __syncthreads();
  // merge the nonzero bins into the segment's global histogram, four bins
  // per 16-byte read
  uint32_t* gh = hist0 + (int64_t)s * kSampleBins;
#pragma unroll
  for (int r = 0; r < kSampleBins / 4 / kSampleThreads; ++r) {
    const int i4 = r * kSampleThreads + threadIdx.x;
    const uint4 c = sh4[i4];
    if (c.x) atomicAdd(&gh[4 * i4], c.x);
    if (c.y) atomicAdd(&gh[4 * i4 + 1], c.y);
    if (c.z) atomicAdd(&gh[4 * i4 + 2], c.z);
    if (c.w) atomicAdd(&gh[4 * i4 + 3], c.w);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(&ss[s].done[0], 1u) == (uint32_t)ctas - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // the merged histogram, read from L2 (__ldcg: not from this SM's L1) with
  // all of a thread's loads in flight at once
  const uint4* gh4 = reinterpret_cast<const uint4*>(gh);
  uint4 v[kSampleBins / 4 / kSampleThreads];
#pragma unroll
  for (int r = 0; r < kSampleBins / 4 / kSampleThreads; ++r)
    v[r] = __ldcg(&gh4[r * kSampleThreads + threadIdx.x]);
#pragma unroll
  for (int r = 0; r < kSampleBins / 4 / kSampleThreads; ++r) sh4[r * kSampleThreads + threadIdx.x] = v[r];
  __syncthreads();
  uint32_t bin, above;
  block_find_bin(sh, kSampleBins, (uint32_t)d.rank, scratch, &bin, &above);
  // T_lo >= 1: zeros are never candidates (a mostly-zero segment then lists
  // its nonzeros instead of overflowing; with fewer than k of them the
  // whole-segment select takes over as for any T_lo above the k-th key)
  if (threadIdx.x == 0) init_state(st, s, d, max(bin << kSampleShift, 1u));
}

// The two-pass form of the sampling, for batches whose lists are long (a
// flat tensor of many million elements): one round of sample loads per warp
// and small histograms (2048, then 1024 bins) in two short launches.  T_lo
// is the lower edge of the 21-bit bin holding the rank-th largest sampled
// key.  With several such calls on concurrent streams (one per worker)
// this form keeps the streams' streaming passes overlapped: the one-pass
// 8192-bin form measured 452 against 475 G elements/s on the four-worker
// 2^31 step, though alone it is as fast.
constexpr int kCoarseBins = 2048;
constexpr int kFineBins = 1024;

__global__ void __launch_bounds__(kSampleThreads)
topk_sample_coarse(LargeBatch b, SampleGrid grid, int nseg, IO io, uint32_t* hist0,
                   SampleState* ss) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint32_t sh[kCoarseBins];
  __shared__ uint32_t scratch[64];
  __shared__ int s_last;
  int q, ctas;
  const int s = sample_seg(grid, nseg, blockIdx.x, &q, &ctas);
  const LargeSeg& d = b.seg[s];
  const int64_t nblk = sample_blocks(d.len);
  if (!samples_needed(d, nblk)) return;  // uniform across the CTA
  const int64_t spacing = d.len / nblk;
  const unsigned lane = lane_id();
  const int64_t gw = (int64_t)q * (kSampleThreads / 32) + (threadIdx.x >> 5);
  const int64_t kWarps = (int64_t)ctas * (kSampleThreads / 32);
  for (int i = threadIdx.x; i < kCoarseBins; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  for (int64_t b0 = gw; b0 < nblk; b0 += kWarps * kSampleUnroll) {  // warp-uniform
    uint32_t key[kSampleUnroll][2];
    bool ok[kSampleUnroll];
    sample_keys(io, d, nblk, spacing, b0, kWarps, lane, key, ok);
#pragma unroll
    for (int u = 0; u < kSampleUnroll; ++u) {
      hist_add(sh, key[u][0] >> 20, ok[u]);
      hist_add(sh, key[u][1] >> 20, ok[u]);
    }
  }
  __syncthreads();
  uint32_t* gh = hist0 + (int64_t)s * kSampleBins;
  for (int i = threadIdx.x; i < kCoarseBins; i += blockDim.x)
    if (sh[i]) atomicAdd(&gh[i], sh[i]);
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(&ss[s].done[0], 1u) == (uint32_t)ctas - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int i = threadIdx.x; i < kCoarseBins; i += blockDim.x) sh[i] = __ldcg(&gh[i]);
  __syncthreads();
  uint32_t bin, above;
  block_find_bin(sh, kCoarseBins, (uint32_t)d.rank, scratch, &bin, &above);
  if (threadIdx.x == 0) {
    ss[s].b0 = bin;
    ss[s].r1 = (uint32_t)d.rank - above;
  }
}

__global__ void __launch_bounds__(kSampleThreads)
topk_sample_fine(LargeBatch b, SampleGrid grid, int nseg, IO io, uint32_t* hist1,
                 SampleState* ss, SegState* st) {
  pdl_wait();
  __shared__ uint32_t sh[kFineBins];
  __shared__ uint32_t scratch[64];
  __shared__ int s_last;
  int q, ctas;
  const int s = sample_seg(grid, nseg, blockIdx.x, &q, &ctas);
  const LargeSeg d = b.seg[s];
  const int64_t nblk = sample_blocks(d.len);
  if (!samples_needed(d, nblk)) {
    if (q == 0 && threadIdx.x == 0) init_state(st, s, d, d.rank <= 0 ? kNoCandidate : 0u);
    return;
  }
  const int64_t spacing = d.len / nblk;
  const uint32_t b0 = __ldcg(&ss[s].b0);
  const unsigned lane = lane_id();
  const int64_t gw = (int64_t)q * (kSampleThreads / 32) + (threadIdx.x >> 5);
  const int64_t kWarps = (int64_t)ctas * (kSampleThreads / 32);
  for (int i = threadIdx.x; i < kFineBins; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  for (int64_t bb = gw; bb < nblk; bb += kWarps * kSampleUnroll) {  // warp-uniform
    uint32_t key[kSampleUnroll][2];
    bool ok[kSampleUnroll];
    sample_keys(io, d, nblk, spacing, bb, kWarps, lane, key, ok);
#pragma unroll
    for (int u = 0; u < kSampleUnroll; ++u) {
#pragma unroll
      for (int h = 0; h < 2; ++h)
        hist_add(sh, (key[u][h] >> 10) & (kFineBins - 1), ok[u] && (key[u][h] >> 20) == b0);
    }
  }
  __syncthreads();
  uint32_t* gh = hist1 + (int64_t)s * kFineBins;
  for (int i = threadIdx.x; i < kFineBins; i += blockDim.x)
    if (sh[i]) atomicAdd(&gh[i], sh[i]);
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(&ss[s].done[1], 1u) == (uint32_t)ctas - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int i = threadIdx.x; i < kFineBins; i += blockDim.x) sh[i] = __ldcg(&gh[i]);
  __syncthreads();
  uint32_t bin, above;
  block_find_bin(sh, kFineBins, __ldcg(&ss[s].r1), scratch, &bin, &above);
  // T_lo >= 1, as in the one-pass form
  if (threadIdx.x == 0) init_state(st, s, d, max((b0 << 20) | (bin << 10), 1u));
}

__device__ __forceinline__ int find_seg(const int64_t* base, int nseg, int64_t x) {
  int lo = 0, hi = nseg - 1;  // largest s with base[s] <= x
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void set4(float4& v, int c, float x) {
  if (c == 0) v.x = x; else if (c == 1) v.y = x; else if (c == 2) v.z = x; else v.w = x;
}
__device__ __forceinline__ float get4(const float4& v, int c) {
  return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}

// Named barriers of the fused pass (0 is __syncthreads).
constexpr int kBarFull0 = 1;    // + buffer: staging buffer filled (streaming -> scan)
constexpr int kBarEmpty0 = 3;   // + buffer: staging buffer drained (scan -> streaming)
constexpr int kBarStream = 5;   // streaming warps only

template <int kId>
__device__ __forceinline__ void bar_sync(int count) {
  asm volatile("bar.sync %0, %1;" ::"n"(kId), "r"(count) : "memory");
}
template <int kId>
__device__ __forceinline__ void bar_arrive(int count) {
  asm volatile("bar.arrive %0, %1;" ::"n"(kId), "r"(count) : "memory");
}
// Barrier of buffer b with compile-time ids (so only the ids in use are
// reserved, which keeps more CTAs resident per SM).
__device__ __forceinline__ void full_arrive(int b) {
  if (b == 0) bar_arrive<kBarFull0>(kFusedThreads); else bar_arrive<kBarFull0 + 1>(kFusedThreads);
}
__device__ __forceinline__ void full_sync(int b) {
  if (b == 0) bar_sync<kBarFull0>(kFusedThreads); else bar_sync<kBarFull0 + 1>(kFusedThreads);
}
__device__ __forceinline__ void empty_arrive(int b) {
  if (b == 0) bar_arrive<kBarEmpty0>(kFusedThreads); else bar_arrive<kBarEmpty0 + 1>(kFusedThreads);
}
__device__ __forceinline__ void empty_sync(int b) {
  if (b == 0) bar_sync<kBarEmpty0>(kFusedThreads); else bar_sync<kBarEmpty0 + 1>(kFusedThreads);
}

struct FusedStage {
  uint2 cand[2][kStreamWarps][kStageCap];  // (local index, float bits), index order
  uint32_t cnt[2][kStreamWarps];           // true candidate count per warp
  int64_t tile[2];                         // tile of the buffer; -1 ends the pass
  int32_t seg[2];
  int64_t next[2];                         // ticket broadcast to the streaming warps
};

// What the fused pass left for segment s: its candidate count c (-1 if the
// last tile's state holds no inclusive prefix: a reported error), and
// which list its select runs on (mode 0: the candidate list, of c entries;
// mode 1: the whole segment, when the list is short of k, over capacity or
// incomplete).  `last_tile_state` is the state word of its last tile.
struct SegOutcome {
  uint32_t mode;
  int64_t len, count;
};
__device__ __forceinline__ SegOutcome seg_outcome(const LargeSeg& d, uint64_t last_tile_state,
                                                  uint32_t overflow) {
  SegOutcome o;
  const uint64_t w = last_tile_state;
  o.count = (w >> 62) == 2 ? (int64_t)(w & kPayloadMask) : -1;
  o.mode = (o.count >= d.k && o.count <= d.cap && !overflow) ? 0u : 1u;
  o.len = o.mode == 0 ? o.count : d.len;
  if (d.k == 0) {
    o.mode = 0;
    o.len = 0;
  }
  return o;
}

// The HBM pass.  Warps 0..7 stream tiles (ticket order): g = g_raw + e is
// written over e, and every element with key >= T_lo of its segment is
// staged in shared memory in index order.  Warp 8 takes each filled staging
// buffer, resolves the tile's offset in its segment's candidate list with the
// bounded decoupled look-back, and writes the candidates out; two buffers let
// the streaming warps run one tile ahead of it.  For a general batch the
// last CTA to finish records each segment's outcome for the select passes;
// in a compact batch (kCompact) topk_finish derives it itself.  A warp loads
// kB rounds of 128 elements at once.
template <int kSpan, bool kCompact, int kB = kBatch>
__global__ void __launch_bounds__(kFusedThreads, kB == kBatch ? kFusedCtasPerSm : 2)
topk_fused(IO io, SegState* st, int nseg, int64_t total_tiles, uint64_t* tstate,
           uint2* cand, Ctl* ctl, int phase, int vec) {
  pdl_wait();
  __shared__ int64_t s_base[kMaxLarge + 1];
  // the segments' fields a tile needs, so that starting a tile reads no
  // global memory
  __shared__ int64_t s_off[kMaxLarge], s_len[kMaxLarge], s_qf[kMaxLarge];
  __shared__ uint32_t s_tlo[kMaxLarge];
  __shared__ FusedStage sg;
  __shared__ int s_last;
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < nseg; i += blockDim.x) {
    s_base[i] = st[i].d.tile_base;
    s_off[i] = st[i].d.off;
    s_len[i] = st[i].d.len;
    s_qf[i] = st[i].d.q_first;
    s_tlo[i] = st[i].t_lo;
  }
  if (threadIdx.x == 0) s_base[nseg] = total_tiles;
  __syncthreads();

  if (warp < kStreamWarps) {
    // The next tile's ticket is requested while the current tile's last
    // loads are in flight, so its round trip stays off the critical path.
    uint32_t ticket = 0;
    if (threadIdx.x == 0) ticket = atomicAdd(&ctl->fused_ticket, 1u);
    for (int it = 0;; ++it) {
      const int b = it & 1;
      if (threadIdx.x == 0) sg.next[b] = ticket;
      bar_sync<kBarStream>(kStreamThreads);
      const int64_t tile = sg.next[b];
      if (it >= 2) empty_sync(b);  // buffer b drained
      if (tile >= total_tiles) {
        if (threadIdx.x == 0) sg.tile[b] = -1;
        full_arrive(b);
        // consume the scan warp's last "drained" arrival so every barrier
        // completes (the scan warp then meets the end marker and stops)
        if (it >= 1) empty_sync(b ^ 1);
        break;
      }
      const int seg = find_seg(s_base, nseg, tile);
      const int64_t a = s_off[seg];
      const uint32_t t_lo = s_tlo[seg];
      // this warp's window, as pointers and 32-bit offsets
      const int64_t w0 = (s_qf[seg] + (tile - s_base[seg])) * (kStreamWarps * kSpan) +
                         (int64_t)warp * kSpan - phase;
      const float* gp = io.g_raw + w0;
      float* ep = io.e + w0;
      const int lo = (int)max((int64_t)-4, min(a - w0, (int64_t)kSpan));
      const int hi = (int)max((int64_t)-4, min(a + s_len[seg] - w0, (int64_t)kSpan + 4));
      const uint32_t loc0 = (uint32_t)(w0 - a);  // local index of window offset 0 (mod 2^32)
      uint2* stage = sg.cand[b][warp];
      uint32_t count = 0;
#pragma unroll 1
      for (int r0 = 0; r0 < kSpan / 128; r0 += kB) {
        float4 gr[kB], ee[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) {
          const int o = (r0 + u) * 128 + (int)lane * 4;
          if (vec && o >= lo && o + 4 <= hi) {
            gr[u] = __ldcs(reinterpret_cast<const float4*>(gp + o));
            ee[u] = __ldcs(reinterpret_cast<const float4*>(ep + o));
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const bool in = o + c >= lo && o + c < hi;
              set4(gr[u], c, in ? gp[o + c] : 0.0f);
              set4(ee[u], c, in ? ep[o + c] : 0.0f);
            }
          }
        }
        if (r0 + kB == kSpan / 128 && threadIdx.x == 0)
          ticket = atomicAdd(&ctl->fused_ticket, 1u);
#pragma unroll
        for (int u = 0; u < kB; ++u) {
          const int o = (r0 + u) * 128 + (int)lane * 4;
          float4 g;
          g.x = __fadd_rn(gr[u].x, ee[u].x);
          g.y = __fadd_rn(gr[u].y, ee[u].y);
          g.z = __fadd_rn(gr[u].z, ee[u].z);
          g.w = __fadd_rn(gr[u].w, ee[u].w);
          const bool full = vec && o >= lo && o + 4 <= hi;
          uint32_t nib = 0;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (full || (o + c >= lo && o + c < hi))
              nib |= (uint32_t)(abs_key(get4(g, c)) >= t_lo) << c;
          // staged candidates are written to e as +0 (emit puts g back at
          // the ones not taken); a candidate without a staging slot keeps g
          uint32_t zero = 0;
          if (__any_sync(kFull, nib != 0)) {
            const uint32_t n4 = __popc(nib);
            const uint32_t inc = warp_incl_scan(n4);
            uint32_t pos = count + inc - n4;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              if ((nib >> c) & 1u) {
                if (pos < kStageCap) {
                  stage[pos] = make_uint2(loc0 + (uint32_t)(o + c), __float_as_uint(get4(g, c)));
                  zero |= 1u << c;
                }
                ++pos;
              }
            }
            count += __shfl_sync(kFull, inc, 31);
          }
          g.x = (zero & 1u) ? 0.0f : g.x;
          g.y = (zero & 2u) ? 0.0f : g.y;
          g.z = (zero & 4u) ? 0.0f : g.z;
          g.w = (zero & 8u) ? 0.0f : g.w;
          if (full) {
            __stcs(reinterpret_cast<float4*>(ep + o), g);
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c)
              if (o + c >= lo && o + c < hi) ep[o + c] = get4(g, c);
          }
        }
      }
      if (lane == 0) sg.cnt[b][warp] = count;
      if (threadIdx.x == 0) {
        sg.tile[b] = tile;
        sg.seg[b] = seg;
      }
      full_arrive(b);
    }
  } else {
    // scan warp
    for (int it = 0;; ++it) {
      const int b = it & 1;
      full_sync(b);
      const int64_t tile = sg.tile[b];
      if (tile < 0) break;
      const int seg = sg.seg[b];
      const uint32_t c = lane < kStreamWarps ? sg.cnt[b][lane] : 0u;
      const uint32_t inc = warp_incl_scan(c);
      const uint32_t agg = __shfl_sync(kFull, inc, 31);
      uint64_t excl;
      if constexpr (kCompact)  // topk_finish reads the states after the kernel ends
        excl = lookback_warp_short<4>(tstate, tile, s_base[seg], agg, io.status);
      else
        excl = lookback_warp(tstate, tile, s_base[seg], agg, io.status);
      if (agg) {
        const int64_t cap = st[seg].d.cap;
        float* es = io.e + st[seg].d.off;
        uint2* out = cand + st[seg].d.cand_base;
        for (int w = 0; w < kStreamWarps; ++w) {
          const uint32_t ct = __shfl_sync(kFull, c, w);
          const uint32_t cw = min(ct, (uint32_t)kStageCap);
          const int64_t base = (int64_t)excl + __shfl_sync(kFull, inc - c, w);
          for (uint32_t j = lane; j < cw; j += 32) {
            const uint2 v = sg.cand[b][w][j];
            if (base + j < cap)
              out[base + j] = v;
            else
              es[v.x] = __uint_as_float(v.y);  // no room in the list: e keeps g
          }
          if (ct > kStageCap && base + kStageCap < cap) {  // warp-uniform
            // The candidates that found no staging slot (a span whose
            // candidates cluster) still hold g in e, after the last staged
            // one.  Staged candidates hold +0 and T_lo >= 1, so a rescan of
            // the rest of the span from L2 finds exactly them, in index
            // order: they fill list slots base + kStageCap on and get +0 in
            // e like every listed candidate (past the capacity they keep g).
            // Once the slots lie past the capacity there is nothing to fill:
            // the list is over capacity and the whole-segment select runs.
            const uint32_t t_lo = st[seg].t_lo;
            const int64_t w0 = (st[seg].d.q_first + (tile - s_base[seg])) *
                                   (int64_t)(kStreamWarps * kSpan) +
                               (int64_t)w * kSpan - phase;
            const int64_t end = min(w0 + kSpan, st[seg].d.off + st[seg].d.len) - st[seg].d.off;
            int64_t pos = base + kStageCap;
            uint32_t found = 0;
            for (int64_t i0 = (int64_t)sg.cand[b][w][kStageCap - 1].x + 1; i0 < end; i0 += 128) {
              float v[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int64_t i = i0 + u * 32 + lane;
                v[u] = i < end ? __ldcg(es + i) : 0.0f;
              }
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int64_t i = i0 + u * 32 + lane;
                const bool cnd = i < end && abs_key(v[u]) >= t_lo;
                const unsigned m = __ballot_sync(kFull, cnd);
                const int64_t p = pos + __popc(m & lanemask_lt());
                if (cnd && p < cap) {
                  out[p] = make_uint2((uint32_t)i, __float_as_uint(v[u]));
                  es[i] = 0.0f;
                }
                pos += __popc(m);
                found += __popc(m);
              }
            }
            // a count that does not match would leave the list incomplete:
            // the whole-segment select then takes over
            if (found != ct - kStageCap && lane == 0) atomicOr(&st[seg].overflow, 1u);
          }
        }
      }
      __syncwarp();
      empty_arrive(b);
    }
  }

  // The last CTA to finish decides, per segment, which list the select runs on.
  if (kCompact) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(&ctl->fused_done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int s = threadIdx.x; s < nseg; s += blockDim.x) {
    const SegOutcome o =
        seg_outcome(st[s].d, ld_acquire(&tstate[s_base[s + 1] - 1]),
                    *reinterpret_cast<volatile uint32_t*>(&st[s].overflow));
    st[s].mode = o.mode;
    st[s].list_len = o.len;
    st[s].cand_count = o.count;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int64_t acc = 0;
    for (int s = 0; s < nseg; ++s) {
      st[s].chunk_base = acc;
      acc += (st[s].list_len + kChunk - 1) / kChunk;
    }
    ctl->total_chunks = acc;
  }
}

// A segment's select list: the candidate list (mode 0: entries are
// (local index, float bits)) or the whole segment itself (mode 1).
struct ListRef {
  uint32_t mode;
  int64_t cand_base, off, len;
};

__device__ __forceinline__ ListRef list_ref(const SegState* st, int seg) {
  ListRef r;
  r.mode = st[seg].mode;
  r.cand_base = st[seg].d.cand_base;
  r.off = st[seg].d.off;
  r.len = st[seg].list_len;
  return r;
}

constexpr int kRestoreThreads = 256;

// A segment whose select runs on the whole segment (mode 1) reads its keys
// from e, which must then hold g everywhere: g is put back at the candidates
// the fused pass staged and wrote as +0, from the candidate list (its first
// min(candidates, capacity) slots, every one written by the fused pass).
// Segments selecting on their list are left alone.
// The segments' states are read in one parallel round into shared memory,
// so a batch without such a segment costs one load per thread.
__global__ void __launch_bounds__(kRestoreThreads)
topk_restore(IO io, const SegState* st, int nseg, const uint2* cand) {
  pdl_trigger();
  pdl_wait();
  __shared__ int64_t s_m[kMaxLarge];  // entries to restore per segment (0: none)
  for (int s = threadIdx.x; s < nseg; s += blockDim.x) {
    const int64_t c = st[s].cand_count;  // <= 0: no candidates, or a reported error
    s_m[s] = (st[s].mode == 1 && c > 0) ? min(c, st[s].d.cap) : 0;
  }
  __syncthreads();
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  for (int s = 0; s < nseg; ++s) {
    const int64_t m = s_m[s];
    if (m == 0) continue;  // uniform across the grid
    const int64_t len = st[s].d.len;
    const uint2* l = cand + st[s].d.cand_base;
    float* es = io.e + st[s].d.off;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < m; j += nthr) {
      const uint2 v = l[j];
      if ((int64_t)v.x < len) es[v.x] = __uint_as_float(v.y);
    }
  }
}

// Lists of at most kSelSmall entries: one CTA per segment loads the keys into
// shared memory and runs the 3-digit radix select there.
__global__ void __launch_bounds__(kSmallThreads)
topk_select_small(IO io, SegState* st, const uint2* cand) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ uint32_t sm[];
  uint32_t* keys = sm;
  uint32_t* hist = sm + kSelSmall;
  uint32_t* scratch = hist + 2048;
  uint32_t* sub = scratch + 64;
  const int seg = blockIdx.x;
  const ListRef l = list_ref(st, seg);
  const int64_t k = st[seg].d.k;
  if (k == 0 || l.len == 0 || l.len > kSelSmall) return;
  const int len = (int)l.len;
  // eight loads in flight per thread
  for (int j0 = 0; j0 < len; j0 += 8 * kSmallThreads) {
    uint32_t y[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u * kSmallThreads + (int)threadIdx.x;
      y[u] = j >= len ? 0u
                      : (l.mode == 0 ? cand[l.cand_base + j].y : __float_as_uint(io.e[l.off + j]));
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u * kSmallThreads + (int)threadIdx.x;
      if (j < len) keys[j] = y[u];
    }
  }
  __syncthreads();
  const SelectResult r = block_radix_select(keys, len, (uint32_t)k, hist, scratch, sub, kSubCap);
  if (threadIdx.x == 0) {
    st[seg].prefix = r.T;
    st[seg].krem = r.need;
    st[seg].gt = r.gt;
    st[seg].resolved = 1;
  }
}

// Longer lists: one digit pass over the chunks of every unresolved list.
// Each CTA builds a shared-memory histogram of a chunk and
// merges it into its segment's global histogram; the CTA that merges a
// segment's last chunk fixes that digit for the segment.  The segments'
// list descriptors and digit prefixes are read once per CTA (they do not
// change during a pass: a segment's prefix is extended only after all of
// its chunks are counted), and a chunk's keys are loaded all at once.
__global__ void __launch_bounds__(kSelThreads)
topk_select(IO io, SegState* st, int nseg, const uint2* cand, uint32_t* ghist, Ctl* ctl,
            int pass) {
  pdl_trigger();
  pdl_wait();
  constexpr int kPer = kChunk / kSelThreads;  // keys per thread per chunk
  __shared__ uint32_t sh[2048];
  __shared__ int64_t s_cb[kMaxLarge + 1];
  __shared__ ListRef s_list[kMaxLarge];
  __shared__ uint32_t s_prefix[kMaxLarge];
  __shared__ uint32_t s_resolved[kMaxLarge];
  __shared__ uint32_t scratch[64];
  __shared__ int s_last;
  const int shift = pass == 0 ? 20 : (pass == 1 ? 10 : 0);
  const int nb = pass == 0 ? 2048 : 1024;
  const int hi = shift + (pass == 0 ? 11 : 10);
  const int64_t total = *reinterpret_cast<volatile int64_t*>(&ctl->total_chunks);
  for (int i = threadIdx.x; i < nseg; i += blockDim.x) {
    s_cb[i] = st[i].chunk_base;
    s_list[i] = list_ref(st, i);
    s_prefix[i] = st[i].prefix;
    s_resolved[i] = st[i].resolved;
  }
  if (threadIdx.x == 0) s_cb[nseg] = total;
  for (int b = threadIdx.x; b < nb; b += blockDim.x) sh[b] = 0;
  __syncthreads();
  for (int64_t c = blockIdx.x; c < total; c += gridDim.x) {
    const int seg = find_seg(s_cb, nseg, c);
    if (s_resolved[seg]) continue;  // uniform across the CTA
    const ListRef l = s_list[seg];
    const uint32_t prefix = s_prefix[seg];
    const int64_t j0 = (c - s_cb[seg]) * kChunk;
    const int64_t j1 = min(j0 + (int64_t)kChunk, l.len);
    uint32_t bits[kPer];
    if (l.mode == 0) {
      const uint2* cl = cand + l.cand_base;
#pragma unroll
      for (int r = 0; r < kPer; ++r) {
        const int64_t j = j0 + r * kSelThreads + threadIdx.x;
        bits[r] = j < j1 ? cl[j].y : 0u;
      }
    } else {
      const float* el = io.e + l.off;
#pragma unroll
      for (int r = 0; r < kPer; ++r) {
        const int64_t j = j0 + r * kSelThreads + threadIdx.x;
        bits[r] = j < j1 ? __float_as_uint(el[j]) : 0u;
      }
    }
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int64_t j = j0 + r * kSelThreads + threadIdx.x;
      const uint32_t key = bits[r] & 0x7FFFFFFFu;
      hist_add(sh, (key >> shift) & (nb - 1),
                    j < j1 && (hi >= 31 || (key >> hi) == (prefix >> hi)));
    }
    __syncthreads();
    for (int b = threadIdx.x; b < nb; b += blockDim.x) {
      const uint32_t v = sh[b];
      if (v) {
        atomicAdd(&ghist[(int64_t)seg * 2048 + b], v);
        sh[b] = 0;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const int64_t nch = s_cb[seg + 1] - s_cb[seg];
      s_last = (int64_t)atomicAdd(&st[seg].chunks_done[pass], 1u) == nch - 1;
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      uint32_t* gh = ghist + (int64_t)seg * 2048;
      uint32_t v[2048 / kSelThreads];
#pragma unroll
      for (int r = 0; r < 2048 / kSelThreads; ++r) {
        const int b = r * kSelThreads + threadIdx.x;
        v[r] = b < nb ? __ldcg(&gh[b]) : 0u;
      }
#pragma unroll
      for (int r = 0; r < 2048 / kSelThreads; ++r) {
        const int b = r * kSelThreads + threadIdx.x;
        if (b < nb) {
          sh[b] = v[r];
          gh[b] = 0;
        }
      }
      __syncthreads();
      uint32_t bin, above;
      block_find_bin(sh, nb, st[seg].krem, scratch, &bin, &above);
      if (threadIdx.x == 0) {
        st[seg].prefix |= bin << shift;
        st[seg].krem -= above;
        st[seg].gt += above;
      }
      for (int b = threadIdx.x; b < nb; b += blockDim.x) sh[b] = 0;
      __syncthreads();
    }
  }
}

__global__ void __launch_bounds__(kEmitThreads)
topk_emit(IO io, SegState* st, int nseg, const uint2* cand, uint64_t* cstate, Ctl* ctl) {
  pdl_wait();
  __shared__ int64_t s_cb[kMaxLarge + 1];
  __shared__ uint32_t s_wgt[kEmitThreads / 32], s_wlt[kEmitThreads / 32];
  __shared__ uint32_t s_ogt[kEmitThreads / 32], s_olt[kEmitThreads / 32];
  __shared__ int64_t s_c;
  __shared__ uint64_t s_agg;
  __shared__ LookbackShared s_lb;
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  const int64_t total = *reinterpret_cast<volatile int64_t*>(&ctl->total_chunks);
  for (int i = threadIdx.x; i < nseg; i += blockDim.x) s_cb[i] = st[i].chunk_base;
  if (threadIdx.x == 0) s_cb[nseg] = total;
  for (;;) {
    if (threadIdx.x == 0) s_c = atomicAdd(&ctl->emit_ticket, 1u);
    __syncthreads();
    const int64_t c = s_c;
    if (c >= total) break;
    const int seg = find_seg(s_cb, nseg, c);
    const ListRef l = list_ref(st, seg);
    const uint32_t T = st[seg].prefix, need = st[seg].krem;
    const int64_t seg_off = st[seg].d.off, out_off = st[seg].d.out_off;
    const int64_t out_end = out_off + st[seg].d.k;
    const int64_t jw = (c - s_cb[seg]) * kChunk + warp * 512;
    uint32_t vb[16], loc[16];
    uint32_t gtm = 0, eqm = 0, ltm = 0;
    // The list kind is uniform per segment, so the branch sits outside the
    // unrolled loads.  (A per-entry branch inside this unrolled, predicated
    // loop produced wrong flags with this toolchain; this form does not.)
    if (l.mode == 0) {
      const uint2* cl = cand + l.cand_base;
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const int64_t j = jw + r * 32 + lane;
        uint2 v = make_uint2(0u, 0u);
        if (j < l.len) v = cl[j];
        vb[r] = v.y;
        loc[r] = v.x;
        const uint32_t key = v.y & 0x7FFFFFFFu;
        gtm |= (uint32_t)(j < l.len && key > T) << r;
        eqm |= (uint32_t)(j < l.len && key == T) << r;
        ltm |= (uint32_t)(j < l.len && key < T) << r;
      }
    } else {
      const float* el = io.e + l.off;
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const int64_t j = jw + r * 32 + lane;
        uint32_t v = 0u;
        if (j < l.len) v = __float_as_uint(el[j]);
        vb[r] = v;
        loc[r] = (uint32_t)j;
        const uint32_t key = v & 0x7FFFFFFFu;
        gtm |= (uint32_t)(j < l.len && key > T) << r;
        eqm |= (uint32_t)(j < l.len && key == T) << r;
        ltm |= (uint32_t)(j < l.len && key < T) << r;
      }
    }
    uint32_t cg = __popc(gtm), ce = __popc(eqm), cl = __popc(ltm);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      cg += __shfl_xor_sync(kFull, cg, o);
      ce += __shfl_xor_sync(kFull, ce, o);
      cl += __shfl_xor_sync(kFull, cl, o);
    }
    if (lane == 0) {
      s_wgt[warp] = cg;
      s_wlt[warp] = cl;
    }
    __syncthreads();
    if (warp == 0) {
      const uint32_t a = lane < kEmitThreads / 32 ? s_wgt[lane] : 0u;
      const uint32_t b = lane < kEmitThreads / 32 ? s_wlt[lane] : 0u;
      const uint32_t ia = warp_incl_scan(a), ib = warp_incl_scan(b);
      if (lane < kEmitThreads / 32) {
        s_ogt[lane] = ia - a;
        s_olt[lane] = ib - b;
      }
      const uint64_t agg = ((uint64_t)__shfl_sync(kFull, ia, 31) << 31) |
                           (uint64_t)__shfl_sync(kFull, ib, 31);
      if (lane == 0) s_agg = agg;
    }
    __syncthreads();
    const uint64_t excl = lookback_block(cstate, c, s_cb[seg], s_agg, io.status, s_lb);
    // On a candidate list (mode 0) e holds +0 at every entry: entries not
    // taken get g back.  On the whole segment (mode 1) taken entries get +0.
    const bool on_list = l.mode == 0;
    if (cg | ce | (on_list ? cl : 0u)) {  // warp-uniform
      int64_t run_gt = (int64_t)(excl >> 31) + s_ogt[warp];
      int64_t run_lt = (int64_t)(excl & 0x7FFFFFFFu) + s_olt[warp];
      const unsigned lm = lanemask_lt();
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const bool g = (gtm >> r) & 1u, q = (eqm >> r) & 1u, b = (ltm >> r) & 1u;
        const unsigned bg = __ballot_sync(kFull, g), bl = __ballot_sync(kFull, b);
        const int64_t j = jw + r * 32 + lane;
        const int64_t gt_before = run_gt + __popc(bg & lm);
        const int64_t eq_before = j - gt_before - (run_lt + __popc(bl & lm));
        if (g || (q && eq_before < (int64_t)need)) {
          const int64_t pos = out_off + gt_before + min(eq_before, (int64_t)need);
          emit_one(io, seg_off + loc[r], loc[r], pos, out_end, __uint_as_float(vb[r]), !on_list);
        } else if (on_list && (q || b)) {
          io.e[seg_off + loc[r]] = __uint_as_float(vb[r]);
        }
        run_gt += __popc(bg);
        run_lt += __popc(bl);
      }
    }
    __syncthreads();
  }
}

namespace cg = cooperative_groups;

constexpr int kFinishThreads = 512;  // per CTA; a cluster of C CTAs shares one item
constexpr uint32_t kNoDigit = 0xFFFFFFFFu;  // a key that a digit pass does not count

// Radix select over the entries of one item split across the C CTAs of a
// thread-block cluster (C = 1: one CTA).  Each CTA counts the keys of its
// own share (`key_at(i)`, i < n) into its histogram; after a cluster
// barrier every CTA sums the C histograms through distributed shared memory
// and finds the same bin, so all CTAs agree on T, gt and need.  Histograms
// alternate between two buffers: a CTA clears the buffer of pass p + 2 only
// after the barrier of pass p + 1, when every CTA has finished reading it.
// The second pass copies this CTA's keys that share the first digit with
// the k-th key into `sub` (room for sub_cap), and the third reads only them
// when they fit.  Shared memory: hist2 = 2 x 2048, tot = 2048, scratch = 64
// words.
template <int C, typename KeyAt>
__device__ __forceinline__ SelectResult cluster_radix_select(int n, uint32_t k, uint32_t* hist2,
                                                             uint32_t* tot, uint32_t* scratch,
                                                             uint32_t* sub, int sub_cap,
                                                             KeyAt key_at) {
  uint32_t prefix = 0, krem = k, gt = 0;
  uint32_t* sub_count = scratch + 40;
  int m = -1;  // keys in sub for the last pass (-1: read all n keys)
  for (int p = 0; p < 3; ++p) {
    // digits: bits 30..20, 19..10, 9..0
    const int shift = 20 - 10 * p, width = p == 0 ? 11 : 10;
    const int nb = 1 << width;
    const int hi = shift + width;  // bits above this digit are fixed
    uint32_t* hist = hist2 + (p & 1) * 2048;
    const bool collect = p == 1;
    for (int b = threadIdx.x; b < nb; b += blockDim.x) hist[b] = 0;
    if (collect && threadIdx.x == 0) *sub_count = 0;
    __syncthreads();
    const bool from_sub = p == 2 && m >= 0;
    const int len = from_sub ? m : n;
    for (int i0 = 0; i0 < len; i0 += 8 * (int)blockDim.x) {
      uint32_t key[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * (int)blockDim.x + (int)threadIdx.x;
        key[u] = i < len ? (from_sub ? sub[i] : key_at(i)) & 0x7FFFFFFFu : 0u;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * (int)blockDim.x + (int)threadIdx.x;
        const bool in = i < len && (hi >= 31 || (key[u] >> hi) == (prefix >> hi));
        hist_add(hist, (key[u] >> shift) & (nb - 1), in);
        if (collect) {
          const unsigned mk = __ballot_sync(kFull, in);
          if (mk != 0u) {  // warp-uniform
            const int first = __ffs(mk) - 1;
            uint32_t base = 0;
            if ((int)(threadIdx.x & 31u) == first) base = atomicAdd(sub_count, (uint32_t)__popc(mk));
            base = __shfl_sync(kFull, base, first);
            const uint32_t pos = base + __popc(mk & lanemask_lt());
            if (in && pos < (uint32_t)sub_cap) sub[pos] = key[u];
          }
        }
      }
    }
    __syncthreads();
    if (collect) m = *sub_count <= (uint32_t)sub_cap ? (int)*sub_count : -1;
    uint32_t* h = hist;
    if (C > 1) {
      // the C histograms summed through distributed shared memory, all of a
      // thread's remote loads in flight at once
      cg::cluster_group cl = cg::this_cluster();
      cl.sync();
      constexpr int kPer = 2048 / kFinishThreads;
      const uint32_t* rh[C];
#pragma unroll
      for (int q = 0; q < C; ++q) rh[q] = cl.map_shared_rank(hist, q);
      uint32_t v[kPer][C];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int b = u * kFinishThreads + (int)threadIdx.x;
#pragma unroll
        for (int q = 0; q < C; ++q) v[u][q] = b < nb ? rh[q][b] : 0u;
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int b = u * kFinishThreads + (int)threadIdx.x;
        uint32_t t = 0;
#pragma unroll
        for (int q = 0; q < C; ++q) t += v[u][q];
        if (b < nb) tot[b] = t;
      }
      __syncthreads();
      h = tot;
    }
    uint32_t bin, above;
    block_find_bin(h, nb, krem, scratch, &bin, &above);
    prefix |= bin << shift;
    gt += above;
    krem -= above;
  }
  return SelectResult{prefix, gt, krem};
}

// One cluster-wide digit pass: every CTA counts digit(i) of its keys (those
// that are not kNoDigit) into `hist` (2048 words, all zero on entry), the C
// histograms are summed through distributed shared memory into `tot`, and
// the bin holding rank krem is found.  Returns (bin, keys above it).
template <int C, typename DigitAt>
__device__ __forceinline__ uint2 cluster_digit_pass(int n, int nb, uint32_t krem, uint32_t* hist,
                                                    uint32_t* tot, uint32_t* scratch,
                                                    DigitAt digit_at) {
  for (int i0 = 0; i0 < n; i0 += 8 * (int)blockDim.x) {
    uint32_t dg[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * (int)blockDim.x + (int)threadIdx.x;
      dg[u] = i < n ? digit_at(i) : kNoDigit;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) hist_add(hist, dg[u], dg[u] != kNoDigit);
  }
  __syncthreads();
  cg::cluster_group cl = cg::this_cluster();
  cl.sync();
  constexpr int kPer = 2048 / kFinishThreads;
  const uint32_t* rh[C];
#pragma unroll
  for (int q = 0; q < C; ++q) rh[q] = cl.map_shared_rank(hist, q);
  uint32_t v[kPer][C];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int b = u * kFinishThreads + (int)threadIdx.x;
#pragma unroll
    for (int q = 0; q < C; ++q) v[u][q] = b < nb ? rh[q][b] : 0u;
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int b = u * kFinishThreads + (int)threadIdx.x;
    uint32_t t = 0;
#pragma unroll
    for (int q = 0; q < C; ++q) t += v[u][q];
    if (b < nb) tot[b] = t;
  }
  __syncthreads();
  uint32_t bin, above;
  block_find_bin(tot, nb, krem, scratch, &bin, &above);
  return make_uint2(bin, above);
}

// Select on a candidate list whose keys are all >= t_lo (the sampled lower
// threshold), in two cluster passes instead of three: the k-th key lies a
// little above t_lo, so the first digit is taken relative to it,
// d0 = min((key - t_lo) >> 11, kWinBins - 1) -- the top bin gathering every
// key at least (kWinBins - 1) * 2^11 above t_lo, about an eighth of an
// octave at the least -- and the second digit is the low 11 bits of
// key - t_lo.  If the k-th key falls in the top bin (t_lo far below it)
// the result is not usable and *ok is false on every CTA of the cluster
// (they all find the same bin).  Buffers as in cluster_radix_select; both
// histograms of hist2 are zero on entry (the caller clears them with its
// own loads, before the barrier it has anyway).
constexpr uint32_t kWinBins = 1024;  // first-digit bins of the two-pass select (the last: the rest)
template <int C, typename KeyAt>
__device__ __forceinline__ SelectResult cluster_window_select(int n, uint32_t k, uint32_t t_lo,
                                                              uint32_t* hist2, uint32_t* tot,
                                                              uint32_t* scratch, KeyAt key_at,
                                                              bool* ok) {
  const uint2 r0 = cluster_digit_pass<C>(n, kWinBins, k, hist2, tot, scratch, [&](int i) {
    const uint32_t off = (key_at(i) & 0x7FFFFFFFu) - t_lo;
    return min(off >> 11, kWinBins - 1u);
  });
  *ok = r0.x < kWinBins - 1u;
  if (!*ok) return SelectResult{0u, 0u, 0u};
  const uint32_t krem = k - r0.y;
  const uint2 r1 = cluster_digit_pass<C>(n, 2048, krem, hist2 + 2048, tot, scratch, [&](int i) {
    const uint32_t off = (key_at(i) & 0x7FFFFFFFu) - t_lo;
    return (off >> 11) == r0.x ? (off & 2047u) : kNoDigit;
  });
  return SelectResult{t_lo + (r0.x << 11) + r1.x, r0.y + r1.y, krem - r1.y};
}

// The (greater, equal) counts of the cluster's CTAs before this one, from
// each CTA's totals (`mine`, published in scratch[62..63]; block_count's
// warp counts use scratch[0..15] and [32..47] with kFinishThreads threads).
static_assert(kFinishThreads <= 512, "cluster totals sit above the warp counts");
static_assert(2048 % kFinishThreads == 0, "cluster histogram reduction layout");
template <int C>
__device__ __forceinline__ uint2 cluster_base(uint2 mine, uint32_t* scratch) {
  if (C == 1) return make_uint2(0u, 0u);
  cg::cluster_group cl = cg::this_cluster();
  if (threadIdx.x == 0) {
    scratch[62] = mine.x;
    scratch[63] = mine.y;
  }
  cl.sync();
  uint32_t bg = 0, be = 0;
  const unsigned r = cl.block_rank();
  for (unsigned q = 0; q < r; ++q) {
    const uint32_t* o = cl.map_shared_rank(scratch, q);
    bg += o[62];
    be += o[63];
  }
  // no CTA may leave while another still reads its totals: arrive here and
  // wait in cluster_leave() at the end of the kernel, so the emit runs while
  // the barrier completes
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
  return make_uint2(bg, be);
}

// The other half of cluster_base's last barrier; every thread calls it once
// before leaving.
template <int C>
__device__ __forceinline__ void cluster_leave() {
  if (C > 1) asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// The last kernel of a compact batch, whose every streaming segment has a
// candidate list that fits kFinishCap entries.  Segment i = blockIdx.x / C
// is finished by one cluster of C CTAs, each taking a contiguous share of
// its list: select on the list and ordered emit.  A segment whose fused pass
// fell back to the whole segment (list incomplete or T_lo above the k-th
// key) is finished from global memory: the cluster puts g back into e at
// the staged candidates, then selects and emits reading e directly (a
// correctness path; such a segment is at most kCompactLen elements long).
// Shared memory per CTA: part_words keys, the same again (at most kSubCap)
// for the last select pass, and the select's 6208 words of histograms and
// scratch.
template <int C>
__global__ void __launch_bounds__(kFinishThreads)
topk_finish(IO io, const SegState* st, int nseg, const uint64_t* tstate, int64_t total_tiles,
            const uint2* cand, int part_words) {
  pdl_wait();
  extern __shared__ uint32_t sm[];
  const int sub_cap = min(part_words, kSubCap);
  uint32_t* keys = sm;
  uint32_t* sub = keys + part_words;
  uint32_t* hist2 = sub + sub_cap;
  uint32_t* tot = hist2 + 2 * 2048;
  uint32_t* scratch = tot + 2048;
  const int item = (int)blockIdx.x / C, rank = (int)blockIdx.x % C;
  const LargeSeg d = st[item].d;
  const int64_t next_tile = item + 1 < nseg ? st[item + 1].d.tile_base : total_tiles;
  const SegOutcome o = seg_outcome(d, tstate[next_tile - 1], st[item].overflow);
  const uint32_t mode = o.mode;
  const int64_t list_len = o.len;
  if (d.k == 0 || list_len == 0) return;  // uniform across the cluster
  const uint2* cl = cand + d.cand_base;
  float* es = io.e + d.off;
  if (mode == 0) {
    // the candidate list: k <= len <= cap <= kFinishCap entries; this CTA's
    // share [lo, lo + n), loaded with eight loads in flight per thread
    const int len = (int)list_len;
    const int per = (len + C - 1) / C;
    const int lo = min(rank * per, len), n = min(per, len - lo);
    const uint2* my = cl + lo;
    for (int j0 = 0; j0 < n; j0 += 8 * kFinishThreads) {
      uint32_t y[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u * kFinishThreads + (int)threadIdx.x;
        y[u] = j < n ? my[j].y : 0u;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u * kFinishThreads + (int)threadIdx.x;
        if (j < n) keys[j] = y[u];
      }
    }
    // both histograms of the two-pass select start at zero
    for (int b = threadIdx.x; b < 2 * 2048; b += kFinishThreads) hist2[b] = 0;
    __syncthreads();
    auto key_at = [keys](int i) { return keys[i]; };
    // two passes relative to T_lo; three from the top bits if the k-th key
    // lies far above T_lo (every CTA takes the same branch)
    bool ok = false;
    SelectResult r;
    if (C > 1)
      r = cluster_window_select<C>(n, (uint32_t)d.k, st[item].t_lo, hist2, tot, scratch, key_at,
                                   &ok);
    if (!ok) {
      if (C > 1) cg::this_cluster().sync();  // no CTA still reads this one's histograms
      r = cluster_radix_select<C>(n, (uint32_t)d.k, hist2, tot, scratch, sub, sub_cap, key_at);
    }
    const uint2 mine = block_count(n, r.T, scratch, key_at);
    const uint2 base = cluster_base<C>(mine, scratch);
    block_emit(io, n, r.T, r.need, base.x, base.y, d.off, d.out_off, d.k, true, scratch, key_at,
               [my](int j) { return (int)my[j].x; });
    cluster_leave<C>();
    return;
  }
  // whole segment: this cluster's CTAs put g back at their share of the
  // staged candidates, then select and emit their share of the segment
  const int64_t c = o.count;  // <= 0: no candidates, or a reported error
  const int64_t mlist = c > 0 ? min(c, d.cap) : 0;
  for (int64_t j = (int64_t)rank * kFinishThreads + threadIdx.x; j < mlist;
       j += (int64_t)C * kFinishThreads) {
    const uint2 v = cl[j];
    if ((int64_t)v.x < d.len) es[v.x] = __uint_as_float(v.y);
  }
  __threadfence();
  if (C > 1) cg::this_cluster().sync();
  else __syncthreads();
  const int len = (int)d.len;  // at most kCompactLen
  const int per = (len + C - 1) / C;
  const int lo = min(rank * per, len), n = min(per, len - lo);
  const float* mine_e = es + lo;
  auto key_at = [mine_e](int i) { return __float_as_uint(mine_e[i]); };
  const SelectResult r = cluster_radix_select<C>(n, (uint32_t)d.k, hist2, tot, scratch, sub,
                                                 sub_cap, key_at);
  const uint2 mine = block_count(n, r.T, scratch, key_at);
  const uint2 base = cluster_base<C>(mine, scratch);
  block_emit(io, n, r.T, r.need, base.x, base.y, d.off, d.out_off, d.k, false, scratch, key_at,
             [lo](int i) { return lo + i; });
  cluster_leave<C>();
}

// Shared memory of a topk_finish<C> CTA for keys of up to part_words words,
// and the share of an item of up to `len` entries.
size_t finish_smem_words(int part_words) {
  return (size_t)part_words + (size_t)std::min(part_words, kSubCap) + 2 * 2048 + 2048 + 64;
}
int finish_part_words(int cluster, int len) { return ((len + cluster - 1) / cluster + 3) & ~3; }

// Cluster size of a finish launch over `items` items: wide clusters while
// the grid stays within about one round of the GPU's SMs.
int finish_cluster(int items, int sms) {
  if (items * 8 <= 2 * sms) return 8;
  if (items * 4 <= 2 * sms) return 4;
  return 2;
}

// ---------------------------------------------------------------------------
// host planning
// ---------------------------------------------------------------------------

struct Batch {
  std::vector<LargeSeg> segs;
  bool compact = false;    // finished by topk_finish (see kCompactLen)
  int64_t max_tiles = 0;   // upper bound over address phases
  int64_t max_chunks = 0;  // every list at its longest (whole segment)
  int64_t cand_total = 0;
};

struct Plan {
  std::vector<SmallSeg> small;  // longest first
  std::vector<Batch> batches;
  size_t small_folded = 0;  // small segments run by the first compact batch's sampling launch
  int64_t total_k = 0;
  // workspace regions (byte offsets); batches reuse the same regions
  size_t off_ctl = 0, off_st = 0, off_sstate = 0, off_hist0 = 0, off_hist1 = 0, off_hist = 0;
  size_t off_tiles = 0, off_chunks = 0, off_cand = 0;
  size_t ctl_clear_bytes = 0;  // bytes cleared from off_ctl before each batch
  size_t bytes = 0;
};

// Rank of T_lo among a segment's sampled keys: the expected number of
// sampled keys at or above the k-th largest key, m = k * S / len, plus five
// standard deviations and 10 (0: no candidates; > S: every element).
int64_t sample_rank(int64_t k, int64_t len) {
  if (k <= 0) return 0;
  const int64_t S = sample_blocks(len) * kSampleBlock;
  const double m = (double)k * (double)S / (double)len;
  const double r = std::ceil(m + 5.0 * std::sqrt(m) + 10.0);
  return r > (double)S ? S + 1 : (int64_t)r;
}

// Whether a streaming segment goes to a compact batch: its candidate list,
// expected at about rank * len / S entries, fills at most half of kFinishCap.
bool compact_segment(int64_t len, int64_t rank) {
  if (len > kCompactLen) return false;
  if (rank <= 0) return true;
  const int64_t S = sample_blocks(len) * kSampleBlock;
  if (rank > S) return false;
  return (double)rank * (double)len / (double)S <= 0.5 * kFinishCap;
}

ef_status make_plan(int64_t n, int32_t nseg, const int64_t* offs, const int64_t* ks,
                    int32_t idx_format, Plan* p) {
  if (n < 0) return EF_ERR_SIZE;
  if (nseg < 1) return EF_ERR_SEGMENTS;
  if (!offs || !ks) return EF_ERR_NULL;
  if (idx_format != EF_IDX_INT32 && idx_format != EF_IDX_BITMAP) return EF_ERR_ARG;
  if (idx_format == EF_IDX_INT32 && n > (int64_t(1) << 31)) return EF_ERR_SIZE;
  if (offs[0] != 0 || offs[nseg] != n) return EF_ERR_SEGMENTS;
  int64_t out_off = 0;
  Batch cur[2];  // [0]: general, [1]: compact
  cur[1].compact = true;
  for (int32_t s = 0; s < nseg; ++s) {
    const int64_t a = offs[s], b = offs[s + 1];
    if (b < a) return EF_ERR_SEGMENTS;
    const int64_t len = b - a;
    if (len > (int64_t(1) << 31)) return EF_ERR_SIZE;
    const int64_t k = ks[s];
    if (k < 0 || k > len) return EF_ERR_K;
    if (len == 0) continue;
    if (len <= kSmallMax) {
      p->small.push_back(SmallSeg{a, out_off, (int32_t)len, (int32_t)k});
    } else {
      LargeSeg d{};
      d.off = a;
      d.len = len;
      d.k = k;
      d.out_off = out_off;
      d.rank = sample_rank(k, len);
      const bool compact = compact_segment(len, d.rank);
      Batch& c = cur[compact ? 1 : 0];
      d.cap = compact ? std::min<int64_t>(len, kFinishCap) : std::min<int64_t>(len, 4 * k + 65536);
      d.cand_base = c.cand_total;
      c.cand_total += d.cap;
      c.max_tiles += (len + kTileSmall - 1) / kTileSmall + 1;  // any tile size
      c.max_chunks += (len + kChunk - 1) / kChunk;
      c.segs.push_back(d);
      if ((int)c.segs.size() == kMaxLarge) {
        p->batches.push_back(c);
        c = Batch();
        c.compact = compact;
      }
    }
    out_off += k;
  }
  // compact batches first; the first batch's sampling launch also runs the
  // longest small segments
  for (int i = 1; i >= 0; --i)
    if (!cur[i].segs.empty()) p->batches.push_back(cur[i]);
  std::stable_partition(p->batches.begin(), p->batches.end(),
                        [](const Batch& b) { return b.compact; });
  std::stable_sort(p->small.begin(), p->small.end(),
                   [](const SmallSeg& x, const SmallSeg& y) { return x.len > y.len; });
  if (!p->batches.empty() && p->batches[0].compact)
    p->small_folded = std::min<size_t>(p->small.size(), kMaxSmall);
  p->total_k = out_off;

  int64_t tiles = 0, chunks = 0, cands = 0, segs = 0;
  bool general = false;
  for (const Batch& b : p->batches) {
    segs = std::max(segs, (int64_t)b.segs.size());
    tiles = std::max(tiles, b.max_tiles);
    cands = std::max(cands, b.cand_total);
    if (!b.compact) {
      general = true;
      chunks = std::max(chunks, b.max_chunks);
    }
  }
  size_t off = sizeof(WsHeader);
  if (!p->batches.empty()) {
    p->off_ctl = off;
    off += sizeof(Ctl);
    p->off_st = off;
    off = round_up(off + sizeof(SegState) * segs, 256);
    p->off_sstate = off;
    off = round_up(off + sizeof(SampleState) * segs, 256);
    p->off_hist0 = off;
    off = round_up(off + (size_t)segs * kSampleBins * 4, 256);
    p->off_hist1 = off;
    if (general) off = round_up(off + (size_t)segs * kFineBins * 4, 256);
    p->off_hist = off;
    if (general) off = round_up(off + (size_t)segs * 2048 * 4, 256);
    p->off_tiles = off;
    off = round_up(off + (size_t)tiles * 8, 256);
    p->off_chunks = off;
    off = round_up(off + (size_t)chunks * 8, 256);
    p->ctl_clear_bytes = off - p->off_ctl;
    p->off_cand = off;
    off = round_up(off + (size_t)cands * 8, 256);
  }
  p->bytes = off;
  return EF_OK;
}

std::once_flag g_attr_once[64];
ef_status g_attr_status[64];

ef_status set_attributes(int dev) {
  if (dev < 0 || dev >= 64) return EF_ERR_ARCH;
  std::call_once(g_attr_once[dev], [&]() {
    const int small_smem = (kSmallMax + kSelectExtraWords) * 4;
    cudaError_t e1 = cudaFuncSetAttribute(topk_small, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          small_smem);
    const int sel_smem = (kSelSmall + kSelectExtraWords) * 4;
    cudaError_t e2 = cudaFuncSetAttribute(topk_select_small,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, sel_smem);
    cudaError_t bad = e1 != cudaSuccess ? e1 : e2;
    const int fin[3][2] = {{2, 0}, {4, 0}, {8, 0}};
    for (const auto& f : fin) {
      const int words = (int)finish_smem_words(finish_part_words(f[0], kFinishCap));
      cudaError_t e = cudaSuccess;
      if (f[0] == 2) e = cudaFuncSetAttribute(topk_finish<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, words * 4);
      if (f[0] == 4) e = cudaFuncSetAttribute(topk_finish<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, words * 4);
      if (f[0] == 8) e = cudaFuncSetAttribute(topk_finish<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, words * 4);
      if (bad == cudaSuccess) bad = e;
    }
    g_attr_status[dev] = bad == cudaSuccess ? EF_OK : cuda_fail(bad);
  });
  return g_attr_status[dev];
}

}  // namespace
}  // namespace ef

extern "C" ef_status ef_topk_workspace_size(int64_t n, int32_t nseg, const int64_t* h_seg_offsets,
                                            const int64_t* h_seg_k, int32_t idx_format,
                                            size_t* bytes) {
  if (!bytes) return EF_ERR_NULL;
  ef::Plan p;
  ef_status st = ef::make_plan(n, nseg, h_seg_offsets, h_seg_k, idx_format, &p);
  if (st != EF_OK) return st;
  *bytes = p.bytes;
  return EF_OK;
}

namespace ef {

ef_status topk_plan_info(int64_t n, int32_t nseg, const int64_t* h_seg_offsets,
                         const int64_t* h_seg_k, int32_t idx_format, size_t* bytes,
                         int64_t* total_k) {
  Plan p;
  ef_status st = make_plan(n, nseg, h_seg_offsets, h_seg_k, idx_format, &p);
  if (st != EF_OK) return st;
  *bytes = p.bytes;
  *total_k = p.total_k;
  return EF_OK;
}

ef_status topk_compress_impl(const float* g_raw, float* e, int64_t n, int32_t nseg,
                             const int64_t* h_seg_offsets, const int64_t* h_seg_k,
                             int32_t idx_format, float* out_values, int32_t* out_indices,
                             uint32_t* out_bitmap, uint32_t* pos_out, void* workspace,
                             size_t workspace_bytes, void* stream) {
  using namespace ef;
  Plan p;
  ef_status st = make_plan(n, nseg, h_seg_offsets, h_seg_k, idx_format, &p);
  if (st != EF_OK) return st;
  const bool bitmap = idx_format == EF_IDX_BITMAP;
  if (!workspace) return EF_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < p.bytes)
    return EF_ERR_WORKSPACE;
  if (n > 0 && (!g_raw || !e)) return EF_ERR_NULL;
  if (p.total_k > 0 && !out_values) return EF_ERR_NULL;
  if (!bitmap && p.total_k > 0 && !out_indices) return EF_ERR_NULL;
  if (bitmap && n > 0 && !out_bitmap) return EF_ERR_NULL;
  if (!bitmap && out_bitmap) return EF_ERR_ARG;
  if (bitmap && out_indices) return EF_ERR_ARG;
  if ((g_raw && !aligned4(g_raw)) || (e && !aligned4(e)) || (out_values && !aligned4(out_values)) ||
      (out_indices && !aligned4(out_indices)) || (out_bitmap && !aligned4(out_bitmap)))
    return EF_ERR_ALIGN;
  const size_t fb = (size_t)n * 4, kb = (size_t)p.total_k * 4, wb = (size_t)((n + 31) / 32) * 4;
  const void* outs[2] = {out_values, bitmap ? (const void*)out_bitmap : (const void*)out_indices};
  const size_t outb[2] = {kb, bitmap ? wb : kb};
  if (overlaps(g_raw, fb, e, fb)) return EF_ERR_ALIAS;
  for (int i = 0; i < 2; ++i) {
    if (overlaps(outs[i], outb[i], g_raw, fb) || overlaps(outs[i], outb[i], e, fb) ||
        overlaps(outs[i], outb[i], workspace, p.bytes))
      return EF_ERR_ALIAS;
  }
  if (overlaps(outs[0], outb[0], outs[1], outb[1])) return EF_ERR_ALIAS;
  if (overlaps(workspace, p.bytes, g_raw, fb) || overlaps(workspace, p.bytes, e, fb))
    return EF_ERR_ALIAS;

  DeviceInfo dev;
  if ((st = current_device(&dev)) != EF_OK) return st;
  int devid = 0;
  cudaGetDevice(&devid);
  if ((st = set_attributes(devid)) != EF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  // the status word, and with it a compact first batch's control region
  // (which follows it directly): one memset less in a short call (1.6 us
  // of a 2^20-element call), while calls that stream long lists on several
  // streams at once measured 0.15 % slower with the merged memset
  const bool merged = !p.batches.empty() && p.batches[0].compact;
  const size_t clear0 = merged ? p.off_ctl + p.ctl_clear_bytes : sizeof(WsHeader);
  cudaError_t err = cudaMemsetAsync(ws, 0, clear0, s);
  if (err != cudaSuccess) return cuda_fail(err);
  if (n == 0) return EF_OK;
  if (bitmap) {
    err = cudaMemsetAsync(out_bitmap, 0, wb, s);
    if (err != cudaSuccess) return cuda_fail(err);
  }
  IO io{g_raw, e, out_values, bitmap ? nullptr : out_indices, bitmap ? out_bitmap : nullptr,
        reinterpret_cast<int32_t*>(ws), pos_out};

  // small segments not folded into the first compact batch's sampling launch
  for (size_t i0 = p.small_folded; i0 < p.small.size(); i0 += kMaxSmall) {
    const size_t cnt = std::min<size_t>(kMaxSmall, p.small.size() - i0);
    SmallBatch sb;
    int maxlen = 0;
    for (size_t i = 0; i < cnt; ++i) {
      sb.seg[i] = p.small[i0 + i];
      maxlen = std::max(maxlen, sb.seg[i].len);
    }
    const int keys_words = (maxlen + 3) & ~3;
    const size_t smem = (size_t)(keys_words + kSelectExtraWords) * 4;
    launch_pdl(topk_small, (unsigned)cnt, kSmallThreads, smem, s, sb, io, keys_words);
    if ((st = check_launch()) != EF_OK) return st;
  }

  // streaming path
  const int phase_g = (int)((reinterpret_cast<uintptr_t>(g_raw) >> 2) & 3u);
  const int phase_e = (int)((reinterpret_cast<uintptr_t>(e) >> 2) & 3u);
  const int vec = phase_g == phase_e ? 1 : 0;
  const int phase = vec ? phase_g : 0;
  Ctl* ctl = reinterpret_cast<Ctl*>(ws + p.off_ctl);
  SegState* sst = reinterpret_cast<SegState*>(ws + p.off_st);
  uint32_t* ghist = reinterpret_cast<uint32_t*>(ws + p.off_hist);
  uint32_t* hist0 = reinterpret_cast<uint32_t*>(ws + p.off_hist0);
  SampleState* sstate = reinterpret_cast<SampleState*>(ws + p.off_sstate);
  uint64_t* tstate = reinterpret_cast<uint64_t*>(ws + p.off_tiles);
  uint64_t* cstate = reinterpret_cast<uint64_t*>(ws + p.off_chunks);
  uint2* cand = reinterpret_cast<uint2*>(ws + p.off_cand);
  bool first_batch = true;
  for (Batch& b : p.batches) {
    LargeBatch lb;
    const int nsg = (int)b.segs.size();
    auto count_tiles = [&](int64_t tile) {
      int64_t n_t = 0;
      for (int i = 0; i < nsg; ++i) {
        LargeSeg d = b.segs[i];
        const int64_t qa = d.off + phase, qb = d.off + d.len + phase;
        d.q_first = qa / tile;
        d.tile_base = n_t;
        n_t += (qb - 1) / tile - d.q_first + 1;
        lb.seg[i] = d;
      }
      return n_t;
    };
    const int64_t cap_ctas = (int64_t)dev.sms * kFusedCtasPerSm;
    int span = kWarpSpanSmall;
    int64_t best = INT64_MAX;
    for (int sp : {kWarpSpan, kWarpSpanMid, kWarpSpanSmall}) {
      const int64_t tile = (int64_t)kStreamWarps * sp;
      const int64_t cost = (count_tiles(tile) + cap_ctas - 1) / cap_ctas * (tile + kTileCost);
      if (cost < best) {
        best = cost;
        span = sp;
      }
    }
    const int64_t tiles = count_tiles((int64_t)kStreamWarps * span);
    if (!(first_batch && merged)) {
      err = cudaMemsetAsync(ws + p.off_ctl, 0, p.ctl_clear_bytes, s);
      if (err != cudaSuccess) return cuda_fail(err);
    }
    // sampling CTAs per segment: kSampleRounds rounds of sample loads per
    // warp in a compact batch, one otherwise (32 blocks per round per CTA),
    // at most kSampleCtasMax; one for a segment that does not sample (it
    // sets the segment's state).  A compact batch whose one-round grid still
    // fits one CTA per SM (a single tensor of a few million elements) takes
    // one round too: its CTAs then wait for one load round trip, not four.
    // (Two rounds for ResNet-50's 53 lists, 400 CTAs in one wave, measured
    // 0.5 us slower than four.)
    auto sample_grid = [&](int rounds) {
      SampleGrid g;
      g.base[0] = 0;
      for (int i = 0; i < nsg; ++i) {
        const LargeSeg& d = lb.seg[i];
        const int64_t nblk = sample_blocks(d.len);
        const int64_t per = (int64_t)(kSampleThreads / 32) * kSampleUnroll * rounds;
        const int64_t c = (d.rank > 0 && d.rank <= nblk * kSampleBlock)
                              ? std::min<int64_t>(kSampleCtasMax, (nblk + per - 1) / per)
                              : 1;
        g.base[i + 1] = g.base[i] + (int32_t)std::max<int64_t>(1, c);
      }
      return g;
    };
    SampleGrid sg = sample_grid(1);
    if (b.compact && sg.base[nsg] > dev.sms) sg = sample_grid(kSampleRounds);
    const size_t nsmall = first_batch ? p.small_folded : 0;
    if (!b.compact) {
      // long lists: the two short sampling passes
      uint32_t* hist1 = reinterpret_cast<uint32_t*>(ws + p.off_hist1);
      launch_pdl(topk_sample_coarse, (unsigned)sg.base[nsg], kSampleThreads, 0, s, lb, sg, nsg,
                 io, hist0, sstate);
      if ((st = check_launch()) != EF_OK) return st;
      launch_pdl(topk_sample_fine, (unsigned)sg.base[nsg], kSampleThreads, 0, s, lb, sg, nsg, io,
                 hist1, sstate, sst);
    } else if (nsmall > 0) {
      // the first compact batch's sampling launch also runs the folded small segments
      SmallBatch sb;
      for (size_t i = 0; i < nsmall; ++i) sb.seg[i] = p.small[i];
      launch_pdl(topk_sample<true, SmallBatch>, (unsigned)(sg.base[nsg] + nsmall), kSampleThreads,
                 0, s, lb, sg, nsg, io, hist0, sstate, sst, sb);
    } else {
      launch_pdl(topk_sample<false, NoSmall>, (unsigned)sg.base[nsg], kSampleThreads, 0, s, lb, sg,
                 nsg, io, hist0, sstate, sst, NoSmall{});
    }
    if ((st = check_launch()) != EF_OK) return st;
    const int fgrid = (int)std::min<int64_t>(tiles, (int64_t)dev.sms * kFusedCtasPerSm);
    prof_begin(EF_KERNEL_TOPK_FUSED, s);
    auto fused = [&](auto kernel) {
      launch_pdl(kernel, fgrid, kFusedThreads, 0, s, io, sst, nsg, tiles, tstate, cand, ctl, phase,
                 vec);
    };
    if (b.compact) {
      // a batch of at most two CTAs per SM of the smallest tiles (a single
      // tensor of a million elements): each warp loads its whole span at
      // once, one round trip instead of two (96 registers, two CTAs per
      // SM; the 2^20-element call 30.9 -> 29.5 us)
      if (span == kWarpSpanSmall && tiles <= (int64_t)dev.sms * 2)
        fused(topk_fused<kWarpSpanSmall, true, kWarpSpanSmall / 128>);
      else if (span == kWarpSpanSmall) fused(topk_fused<kWarpSpanSmall, true>);
      else if (span == kWarpSpanMid) fused(topk_fused<kWarpSpanMid, true>);
      else fused(topk_fused<kWarpSpan, true>);
    } else {
      if (span == kWarpSpanSmall) fused(topk_fused<kWarpSpanSmall, false>);
      else if (span == kWarpSpanMid) fused(topk_fused<kWarpSpanMid, false>);
      else fused(topk_fused<kWarpSpan, false>);
    }
    if ((st = check_launch()) != EF_OK) return st;
    prof_end(EF_KERNEL_TOPK_FUSED, s);
    if (b.compact) {
      // one cluster per segment
      const int cl = finish_cluster(nsg, dev.sms);
      const int part = finish_part_words(cl, kFinishCap);
      const size_t smem = finish_smem_words(part) * 4;
      const unsigned grid = (unsigned)(nsg * cl);
      if (cl == 8)
        launch_cluster_pdl(topk_finish<8>, 8, grid, kFinishThreads, smem, s, io, sst, nsg,
                           tstate, tiles, cand, part);
      else if (cl == 4)
        launch_cluster_pdl(topk_finish<4>, 4, grid, kFinishThreads, smem, s, io, sst, nsg,
                           tstate, tiles, cand, part);
      else
        launch_cluster_pdl(topk_finish<2>, 2, grid, kFinishThreads, smem, s, io, sst, nsg,
                           tstate, tiles, cand, part);
      if ((st = check_launch()) != EF_OK) return st;
    } else {
      launch_pdl(topk_restore, dev.sms * 2, kRestoreThreads, 0, s, io, sst, nsg, cand);
      if ((st = check_launch()) != EF_OK) return st;
      launch_pdl(topk_select_small, nsg, kSmallThreads, (size_t)(kSelSmall + kSelectExtraWords) * 4, s,
                 io, sst, cand);
      if ((st = check_launch()) != EF_OK) return st;
      const int sgrid =
          (int)std::max<int64_t>(1, std::min<int64_t>(b.max_chunks, (int64_t)dev.sms * 3));
      for (int pass = 0; pass < 3; ++pass) {
        launch_pdl(topk_select, sgrid, kSelThreads, 0, s, io, sst, nsg, cand, ghist, ctl, pass);
        if ((st = check_launch()) != EF_OK) return st;
      }
      const int egrid =
          (int)std::max<int64_t>(1, std::min<int64_t>(b.max_chunks, (int64_t)dev.sms * 4));
      launch_pdl(topk_emit, egrid, kEmitThreads, 0, s, io, sst, nsg, cand, cstate, ctl);
      if ((st = check_launch()) != EF_OK) return st;
    }
    first_batch = false;
  }
  return EF_OK;
}

}  // namespace ef

extern "C" ef_status ef_topk_compress(const float* g_raw, float* e, int64_t n, int32_t nseg,
                                      const int64_t* h_seg_offsets, const int64_t* h_seg_k,
                                      int32_t idx_format, float* out_values,
                                      int32_t* out_indices, uint32_t* out_bitmap,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  return ef::topk_compress_impl(g_raw, e, n, nseg, h_seg_offsets, h_seg_k, idx_format,
                                out_values, out_indices, out_bitmap, nullptr, workspace,
                                workspace_bytes, stream);
}

// ---------------------------------------------------------------------------
// Allocation-free entry point: the same computation as ef_topk_compress with
// a library-owned scratch array in place of the caller's workspace.
// ---------------------------------------------------------------------------

namespace ef {
namespace {

// Scratch for ef_topk_compress_noalloc; holds EF_NOALLOC_SCRATCH_BYTES on
// every device that loads the library.  In host code this name is only a
// stand-in for the device array; its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[EF_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current).
ef_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err);
  if (dev < 0 || dev >= 64) return EF_ERR_ARCH;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess) return cuda_fail(err);
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return EF_OK;
}

}  // namespace
}  // namespace ef

extern "C" ef_status ef_topk_compress_noalloc(const float* g_raw, float* e, int64_t n,
                                              int32_t nseg, const int64_t* h_seg_offsets,
                                              const int64_t* h_seg_k, int32_t idx_format,
                                              float* out_values, int32_t* out_indices,
                                              uint32_t* out_bitmap, void* stream) {
  size_t need = 0;
  ef_status st = ef_topk_workspace_size(n, nseg, h_seg_offsets, h_seg_k, idx_format, &need);
  if (st != EF_OK) return st;
  if (need > (size_t)EF_NOALLOC_SCRATCH_BYTES) return EF_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((st = ef::noalloc_scratch(&scratch)) != EF_OK) return st;
  return ef_topk_compress(g_raw, e, n, nseg, h_seg_offsets, h_seg_k, idx_format, out_values,
                          out_indices, out_bitmap, scratch, (size_t)EF_NOALLOC_SCRATCH_BYTES,
                          stream);
}

extern "C" ef_status ef_topk_noalloc_status(void* stream, int32_t* device_status) {
  if (!device_status) return EF_ERR_NULL;
  void* scratch = nullptr;
  ef_status st = ef::noalloc_scratch(&scratch);
  if (st != EF_OK) return st;
  cudaError_t err = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return ef::cuda_fail(err);
  int32_t v = 0;
  err = cudaMemcpy(&v, scratch, sizeof(v), cudaMemcpyDeviceToHost);
  if (err != cudaSuccess) return ef::cuda_fail(err);
  *device_status = v;
  return EF_OK;
}
