// Random magnitude-proportional sparsification with error feedback
// ("梯度稀疏化：只传输重要的梯度元素", §随机稀疏化, in place of step 3 of
// §详细算法流程): each element is kept with probability proportional to |g|,
// normalised so that the expected count is k:
//   S = exact sum of |g| over a segment's finite elements, rounded once to
//       float64;  c = RN32(k / S)  (0 when S = 0);
//   p_i = min(1, RN32(c |g_i|)), 1 for non-finite g_i;
//   u_i = (w_i >> 8) / 2^24, w_i = word i % 4 of Philox4x32-10 at counter
//         (i / 4 low, i / 4 high, step low, step high), key (seed low, high);
//   kept iff u_i < p_i;  the packet lists kept (g_i, i), ascending, unscaled,
//   up to its capacity; e = g - g~ (+0 where sent, g elsewhere).
// Philox4x32-10 follows its published definition (Salmon, Moraes, Dror,
// Shaw, SC 2011): ten rounds of two 32x32->64 multiplies by 0xD2511F53 and
// 0xCD9E8D57, the key bumped by 0x9E3779B9 / 0xBB67AE85 between rounds.
//
// Pass 1 (rk_sum, 12 B / element) writes g = g_raw + e over e and sums |g|
// exactly: a float32 magnitude is m * 2^(sh - 149) with m < 2^24 and
// 0 <= sh <= 253, so each thread keeps four 128-bit integer accumulators,
// one per 64-bit-aligned group of sh, and a CTA flushes them as 40-bit
// carry-save chunks with one atomicAdd per chunk when it leaves a segment
// (sums of at most 2^14 flushes of 2^50 fit in 64 bits).  rk_finalize turns
// each segment's chunks into the float64 nearest the exact sum and forms c.
// Pass 2 (rk_select, 4 B / element + 8 B per kept element) stages each
// 8192-element tile of g in shared memory, draws one Philox call per four
// elements, and compacts the kept elements in ticket order with the bounded
// decoupled look-back (the running offset carries across launches).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "ef_common.cuh"

namespace ef {
namespace {

constexpr int kRT = 256;                // threads per CTA
constexpr int kRPer = 32;               // elements per thread per tile
constexpr int kRTile = kRT * kRPer;     // 8192 elements per tile
constexpr int kRBatch = 128;            // segments per launch
constexpr int kChunks = 8;              // 40-bit chunks of an exact sum (320 bits)
constexpr uint64_t kMask40 = (1ull << 40) - 1;

struct RSeg {
  int64_t off, len, k;
  int64_t tile_a;  // first tile of the segment in pass 1
  int64_t tile_b;  // first tile in pass 2 (segments with k = 0 have none)
  int32_t id;      // segment number in the whole call
};

struct RBatch {
  RSeg seg[kRBatch];
  int64_t tiles_a[kRBatch + 1];  // prefix of pass-1 tiles; [nseg] = total
  int64_t tiles_b[kRBatch + 1];
  int32_t nseg;
};

struct RCtl {
  uint32_t ticket;
  uint32_t pad;
  int64_t base[2];  // kept elements before a launch: launch b reads [b % 2], its
                    // last tile writes [(b + 1) % 2] (never the word being read)
};

__device__ __forceinline__ int find_tile_seg(const int64_t* base, int nseg, int64_t t) {
  int lo = 0, hi = nseg - 1;  // last segment whose first tile is <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// ---------------------------------------------------------------- exact sum

struct Acc {
  uint64_t lo[4], hi[4];
};

__device__ __forceinline__ void acc_clear(Acc& a) {
#pragma unroll
  for (int q = 0; q < 4; ++q) a.lo[q] = a.hi[q] = 0;
}

// 128-bit add hi:lo += ah:al with the carry chain in four 32-bit
// add-with-carry instructions.
__device__ __forceinline__ void add128(uint64_t& lo, uint64_t& hi, uint64_t al, uint64_t ah) {
  asm("{\n\t"
      ".reg .u32 l0, l1, h0, h1, a0, a1, b0, b1;\n\t"
      "mov.b64 {l0, l1}, %0;\n\t"
      "mov.b64 {h0, h1}, %1;\n\t"
      "mov.b64 {a0, a1}, %2;\n\t"
      "mov.b64 {b0, b1}, %3;\n\t"
      "add.cc.u32 l0, l0, a0;\n\t"
      "addc.cc.u32 l1, l1, a1;\n\t"
      "addc.cc.u32 h0, h0, b0;\n\t"
      "addc.u32 h1, h1, b1;\n\t"
      "mov.b64 %0, {l0, l1};\n\t"
      "mov.b64 %1, {h0, h1};\n\t"
      "}"
      : "+l"(lo), "+l"(hi)
      : "l"(al), "l"(ah));
}

// Adds |x| given as its bit pattern (finite, sign cleared): m * 2^(sh - 149)
// goes into group sh / 64 as m << (sh % 64).  Magnitudes in [2^-62, 4)
// (group 1) take the short path.
__device__ __forceinline__ void acc_add(Acc& a, uint32_t bits) {
  const uint32_t E = bits >> 23;
  const uint64_t m = E ? (uint64_t)((bits & 0x7FFFFFu) | 0x800000u) : (uint64_t)(bits & 0x7FFFFFu);
  const uint32_t sh = E ? E - 1 : 0;
  const uint32_t g = sh >> 6, off = sh & 63u;
  const uint64_t l = m << off;
  const uint64_t h = off > 40 ? m >> (64 - off) : 0ull;
  if (g == 1) {
    add128(a.lo[1], a.hi[1], l, h);
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (q != 1 && q == (int)g) add128(a.lo[q], a.hi[q], l, h);
  }
}

// Bits [pos, pos + 40) of the 128-bit value hi:lo (pos may be negative).
__device__ __forceinline__ uint64_t bits40(uint64_t hi, uint64_t lo, int pos) {
  if (pos <= -40 || pos >= 128) return 0;
  if (pos < 0) return (lo << (-pos)) & kMask40;
  uint64_t v;
  if (pos == 0) v = lo;
  else if (pos < 64) v = (lo >> pos) | (hi << (64 - pos));
  else v = hi >> (pos - 64);
  return v & kMask40;
}

// CTA-wide flush of every thread's accumulator into the segment's chunks.
__device__ void acc_flush(const Acc& a, uint64_t* chunks, uint64_t (*red)[kChunks]) {
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    uint64_t v = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) v += bits40(a.hi[q], a.lo[q], 40 * c - 64 * q);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    if (lane == 0) red[warp][c] = v;
  }
  __syncthreads();
  if (threadIdx.x < kChunks) {
    uint64_t v = 0;
    for (int w = 0; w < kRT / 32; ++w) v += red[w][threadIdx.x];
    if (v) atomicAdd(reinterpret_cast<unsigned long long*>(&chunks[threadIdx.x]), v);
  }
  __syncthreads();
}

// Pass 1: g = g_raw + e written over e; exact sum of the finite |g|.
__global__ void __launch_bounds__(kRT)
rk_sum(RBatch b, const float* __restrict__ g_raw, float* __restrict__ e, uint64_t* acc) {
  __shared__ int64_t s_base[kRBatch + 1];
  __shared__ uint64_t red[kRT / 32][kChunks];
  for (int i = threadIdx.x; i <= b.nseg; i += blockDim.x) s_base[i] = b.tiles_a[i];
  __syncthreads();
  const int64_t tiles = s_base[b.nseg];
  Acc a;
  acc_clear(a);
  int cur = -1;
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int s = find_tile_seg(s_base, b.nseg, t);
    if (s != cur) {  // uniform across the CTA
      if (cur >= 0) {
        acc_flush(a, acc + (int64_t)cur * kChunks, red);
        acc_clear(a);
      }
      cur = s;
    }
    const RSeg& d = b.seg[s];
    const int64_t j0 = (t - s_base[s]) * kRTile;
    const int64_t len = min((int64_t)kRTile, d.len - j0);
    const float* gp = g_raw + d.off + j0;
    float* ep = e + d.off + j0;
#pragma unroll 1
    for (int r0 = 0; r0 < kRPer; r0 += 8) {
      float gv[8], ev[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t j = (int64_t)(r0 + u) * kRT + threadIdx.x;
        gv[u] = j < len ? __ldcs(gp + j) : 0.0f;
        ev[u] = j < len ? __ldcs(ep + j) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t j = (int64_t)(r0 + u) * kRT + threadIdx.x;
        if (j < len) {
          const float g = __fadd_rn(gv[u], ev[u]);
          __stcs(ep + j, g);
          const uint32_t bits = __float_as_uint(g) & 0x7FFFFFFFu;
          if (bits < 0x7F800000u) acc_add(a, bits);
        }
      }
    }
  }
  if (cur >= 0) acc_flush(a, acc + (int64_t)cur * kChunks, red);
}

// float64 nearest (ties to even) to the exact sum sum_c chunks[c] * 2^(40c)
// times 2^-149.
__device__ double exact_to_double(const uint64_t* chunks) {
  uint64_t L[6] = {0, 0, 0, 0, 0, 0};
  for (int c = 0; c < kChunks; ++c) {
    // add chunks[c] << 40c into L
    const int bit = 40 * c, w = bit >> 6, o = bit & 63;
    const uint64_t v = chunks[c];
    uint64_t add0 = v << o, add1 = o ? v >> (64 - o) : 0ull;
    uint64_t carry = 0;
    for (int i = w; i < 6; ++i) {
      const uint64_t x = i == w ? add0 : (i == w + 1 ? add1 : 0ull);
      const uint64_t s1 = L[i] + x;
      const uint64_t c1 = s1 < L[i] ? 1ull : 0ull;
      const uint64_t s2 = s1 + carry;
      const uint64_t c2 = s2 < s1 ? 1ull : 0ull;
      L[i] = s2;
      carry = c1 + c2;
      if (i > w + 1 && !carry) break;
    }
  }
  int top = -1;
  for (int i = 5; i >= 0 && top < 0; --i)
    if (L[i]) top = 64 * i + 63 - __clzll((long long)L[i]);
  if (top < 0) return 0.0;
  // 53-bit mantissa from bits [top - 52, top], rounded to nearest even
  auto bit_at = [&](int p) -> uint64_t {
    return p < 0 ? 0ull : (L[p >> 6] >> (p & 63)) & 1ull;
  };
  uint64_t mant = 0;
  for (int p = top; p >= top - 52; --p) mant = (mant << 1) | bit_at(p);
  int shift = top - 52;  // value = mant * 2^shift * 2^-149 before rounding
  if (shift > 0) {
    const uint64_t guard = bit_at(shift - 1);
    bool sticky = false;
    for (int p = shift - 2; p >= 0 && !sticky; --p) sticky = bit_at(p) != 0;
    if (guard && (sticky || (mant & 1ull))) {
      ++mant;
      if (mant >> 53) {
        mant >>= 1;
        ++shift;
      }
    }
  }
  // mant in [2^52, 2^53): biased exponent of mant * 2^(shift - 149)
  const int64_t be = (int64_t)shift - 149 + 52 + 1023;
  return __longlong_as_double((long long)(((uint64_t)be << 52) | (mant & ((1ull << 52) - 1))));
}

__global__ void rk_finalize(RBatch b, const uint64_t* acc, float* coef) {
  const int s = threadIdx.x;
  if (s >= b.nseg) return;
  const double S = exact_to_double(acc + (int64_t)s * kChunks);
  coef[s] = S > 0.0 ? __double2float_rn(__ddiv_rn((double)b.seg[s].k, S)) : 0.0f;
}

// ---------------------------------------------------------------- pass 2

__device__ __forceinline__ void philox4x32_10(uint32_t& c0, uint32_t& c1, uint32_t& c2,
                                              uint32_t& c3, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
}

struct RSelectArgs {
  const float* coef;
  float* e;
  float* out_values;
  int32_t* out_indices;
  int64_t capacity;
  unsigned long long* counts;  // [nseg + 1] of the whole call
  int32_t nseg_total;
  uint64_t seed, step;
  uint64_t* tstate;
  RCtl* ctl;
  int32_t* status;
  int parity;  // launch number % 2
};

// Pass 2: keep draws and the ordered packet.  A tile of 8192 elements per
// ticket; warp w owns elements [1024 w, 1024 (w + 1)) in 32 rounds of 32
// consecutive elements (lane l: element 32 r + l of the slice), four rounds
// at a time: the 32 lanes first compute one Philox call each for the quads
// the four rounds touch (33 when the slice is not quad-aligned) and leave
// the words in a per-warp buffer, then every lane tests its element.  A
// round's keep ballot gives the ranks inside the slice; one block scan over
// the warps and the bounded look-back over tiles give the packet offset, and
// each warp then writes its kept elements (values re-read from e, an L2 hit).
constexpr int kRWarps = kRT / 32;
constexpr int kRSlice = kRTile / kRWarps;   // 1024 elements per warp
constexpr int kRRounds = kRSlice / 32;      // 32 rounds

__global__ void __launch_bounds__(kRT, 8)
rk_select(RBatch b, RSelectArgs a) {
  __shared__ int64_t s_base[kRBatch + 1];
  __shared__ uint32_t words[kRWarps][33 * 4];
  __shared__ uint32_t s_wtot[kRWarps], s_woff[kRWarps];
  __shared__ uint32_t s_t;
  __shared__ uint64_t s_excl;
  __shared__ int64_t s_prev;
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i <= b.nseg; i += blockDim.x) s_base[i] = b.tiles_b[i];
  if (threadIdx.x == 0) s_prev = *reinterpret_cast<volatile int64_t*>(&a.ctl->base[a.parity]);
  __syncthreads();
  const int64_t tiles = s_base[b.nseg];
  const int64_t prev = s_prev;
  const uint32_t k0 = (uint32_t)a.seed, k1 = (uint32_t)(a.seed >> 32);
  const uint32_t st0 = (uint32_t)a.step, st1 = (uint32_t)(a.step >> 32);
  uint32_t* wb = words[warp];
  for (;;) {
    if (threadIdx.x == 0) s_t = atomicAdd(&a.ctl->ticket, 1u);
    __syncthreads();
    const int64_t t = s_t;
    if (t >= tiles) break;
    const int s = find_tile_seg(s_base, b.nseg, t);
    const RSeg& d = b.seg[s];
    const float c = a.coef[s];
    const int64_t j0 = (t - s_base[s]) * kRTile;
    const int64_t len = min((int64_t)kRTile, d.len - j0);
    const int64_t i0 = d.off + j0 + (int64_t)warp * kRSlice;  // global index of the slice start
    const int64_t slen = max((int64_t)0, min((int64_t)kRSlice, len - (int64_t)warp * kRSlice));
    const float* ep = a.e + i0;
    // keep ballots of this slice: lane x holds round x's ballot and the
    // number of kept elements before round x
    uint32_t my_ballot = 0, my_before = 0, run = 0;
    // the next group's values are loaded while this group's draws compute
    float nxt[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int jl = u * 32 + (int)lane;
      nxt[u] = jl < slen ? ep[jl] : 0.0f;
    }
    for (int r0 = 0; r0 < kRRounds; r0 += 4) {
      float gv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) gv[u] = nxt[u];
      if (r0 + 4 < kRRounds) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int jl = (r0 + 4 + u) * 32 + (int)lane;
          nxt[u] = jl < slen ? ep[jl] : 0.0f;
        }
      }
      // quads of rounds r0 .. r0 + 3: from (i0 + 32 r0) / 4, at most 33
      const int64_t first = i0 + (int64_t)r0 * 32;
      const uint64_t q0 = (uint64_t)first >> 2;
      __syncwarp();
      {
        uint64_t q = q0 + lane;
        uint32_t w0 = (uint32_t)q, w1 = (uint32_t)(q >> 32), w2 = st0, w3 = st1;
        philox4x32_10(w0, w1, w2, w3, k0, k1);
        wb[lane * 4 + 0] = w0;
        wb[lane * 4 + 1] = w1;
        wb[lane * 4 + 2] = w2;
        wb[lane * 4 + 3] = w3;
        if ((first & 3) != 0 && lane == 0) {  // the 33rd quad
          q = q0 + 32;
          w0 = (uint32_t)q;
          w1 = (uint32_t)(q >> 32);
          w2 = st0;
          w3 = st1;
          philox4x32_10(w0, w1, w2, w3, k0, k1);
          wb[128] = w0;
          wb[129] = w1;
          wb[130] = w2;
          wb[131] = w3;
        }
      }
      __syncwarp();
      // element o of the group (o = 32 u + lane) is word (f + o) of the
      // buffer, f = first % 4; u < min(1, x) is !(u >= x) for every x,
      // since u < 1 (x >= 1, +Inf and a NaN product all keep)
      const int f = (int)(first & 3);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int jl = (r0 + u) * 32 + (int)lane;
        bool keep = false;
        if (jl < slen) {
          const uint32_t w = wb[f + u * 32 + (int)lane];
          const float x = __fmul_rn(c, fabsf(gv[u]));
          keep = !(__uint2float_rn(w >> 8) * 0x1p-24f >= x);
        }
        const uint32_t bal = __ballot_sync(kFull, keep);
        if (lane == (unsigned)(r0 + u)) {
          my_ballot = bal;
          my_before = run;
        }
        run += __popc(bal);
      }
    }
    if (lane == 0) s_wtot[warp] = run;
    __syncthreads();
    if (warp == 0) {
      const uint32_t v = lane < kRWarps ? s_wtot[lane] : 0u;
      const uint32_t incl = warp_incl_scan(v);
      if (lane < kRWarps) s_woff[lane] = incl - v;
      const uint32_t total = __shfl_sync(kFull, incl, 31);
      const uint64_t ex = lookback_warp(a.tstate, t, 0, total, a.status);
      if (lane == 0) {
        s_excl = ex;
        const int64_t tile_off = prev + (int64_t)ex;
        const int64_t sent = max((int64_t)0, min((int64_t)total, a.capacity - tile_off));
        if (sent) atomicAdd(&a.counts[d.id], (unsigned long long)sent);
        if (tile_off + (int64_t)total > a.capacity) set_status(a.status, EF_ERR_CAPACITY);
        if (t == tiles - 1) {
          const int64_t all = tile_off + (int64_t)total;
          a.ctl->base[a.parity ^ 1] = all;
          a.counts[a.nseg_total] = (unsigned long long)min(all, a.capacity);
        }
      }
    }
    __syncthreads();
    const int64_t slice_off = prev + (int64_t)s_excl + s_woff[warp];
    if (run) {  // warp-uniform
      const unsigned lm = lanemask_lt();
      for (int x = 0; x < kRRounds; ++x) {
        const uint32_t bal = __shfl_sync(kFull, my_ballot, x);
        if (!bal) continue;  // warp-uniform
        const uint32_t before = __shfl_sync(kFull, my_before, x);
        if ((bal >> lane) & 1u) {
          const int64_t pos = slice_off + before + __popc(bal & lm);
          const int64_t jl = (int64_t)x * 32 + lane;
          if (pos < a.capacity) {
            a.out_values[pos] = ep[jl];
            a.out_indices[pos] = (int32_t)(i0 + jl);
            a.e[i0 + jl] = 0.0f;
          }
        }
      }
    }
    __syncthreads();
  }
}

struct RPlan {
  std::vector<RBatch> batches;
  int64_t max_tiles_b = 0;
  size_t off_acc = 0, off_coef = 0, off_ctl = 0, off_tiles = 0, clear_bytes = 0, bytes = 0;
};

ef_status rk_plan(int64_t n, int32_t nseg, const int64_t* offs, const int64_t* ks, RPlan* p) {
  if (n < 0 || n > (int64_t(1) << 31)) return EF_ERR_SIZE;
  if (nseg < 1) return EF_ERR_SEGMENTS;
  if (!offs || !ks) return EF_ERR_NULL;
  if (offs[0] != 0 || offs[nseg] != n) return EF_ERR_SEGMENTS;
  RBatch cur{};
  auto flush = [&]() {
    if (cur.nseg == 0) return;
    p->max_tiles_b = std::max(p->max_tiles_b, cur.tiles_b[cur.nseg]);
    p->batches.push_back(cur);
    cur = RBatch{};
  };
  for (int32_t i = 0; i < nseg; ++i) {
    const int64_t a = offs[i], b = offs[i + 1];
    if (b < a) return EF_ERR_SEGMENTS;
    const int64_t len = b - a, k = ks[i];
    if (k < 0 || k > len) return EF_ERR_K;
    if (len == 0) continue;
    const int t = cur.nseg;
    const int64_t tiles = (len + kRTile - 1) / kRTile;
    cur.seg[t] = RSeg{a, len, k, cur.tiles_a[t], cur.tiles_b[t], i};
    cur.tiles_a[t + 1] = cur.tiles_a[t] + tiles;
    cur.tiles_b[t + 1] = cur.tiles_b[t] + (k > 0 ? tiles : 0);
    if (++cur.nseg == kRBatch) flush();
  }
  flush();
  size_t off = sizeof(WsHeader);
  p->off_ctl = off;
  off = round_up(off + sizeof(RCtl), 256);
  p->off_acc = off;
  off = round_up(off + (size_t)kRBatch * kChunks * 8, 256);
  p->off_coef = off;
  off = round_up(off + (size_t)kRBatch * 4, 256);
  p->off_tiles = off;
  off = round_up(off + (size_t)std::max<int64_t>(p->max_tiles_b, 1) * 8, 256);
  p->bytes = off;
  return EF_OK;
}

}  // namespace
}  // namespace ef

extern "C" ef_status ef_randk_workspace_size(int64_t n, int32_t nseg,
                                             const int64_t* h_seg_offsets,
                                             const int64_t* h_seg_k, size_t* bytes) {
  if (!bytes) return EF_ERR_NULL;
  ef::RPlan p;
  ef_status st = ef::rk_plan(n, nseg, h_seg_offsets, h_seg_k, &p);
  if (st != EF_OK) return st;
  *bytes = p.bytes;
  return EF_OK;
}

extern "C" ef_status ef_randk_compress(const float* g_raw, float* e, int64_t n, int32_t nseg,
                                       const int64_t* h_seg_offsets, const int64_t* h_seg_k,
                                       uint64_t seed, uint64_t step, float* out_values,
                                       int32_t* out_indices, int64_t capacity,
                                       int64_t* d_counts, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  using namespace ef;
  RPlan p;
  ef_status st = rk_plan(n, nseg, h_seg_offsets, h_seg_k, &p);
  if (st != EF_OK) return st;
  if (!workspace) return EF_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < p.bytes)
    return EF_ERR_WORKSPACE;
  if (capacity < 0) return EF_ERR_ARG;
  if (!d_counts || (n > 0 && (!g_raw || !e)) || (capacity > 0 && (!out_values || !out_indices)))
    return EF_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(d_counts) & 7u) != 0 || (g_raw && !aligned4(g_raw)) ||
      (e && !aligned4(e)) || (out_values && !aligned4(out_values)) ||
      (out_indices && !aligned4(out_indices)))
    return EF_ERR_ALIGN;
  const size_t fb = (size_t)n * 4, cb = (size_t)capacity * 4, nb = (size_t)(nseg + 1) * 8;
  const void* bufs[6] = {g_raw, e, out_values, out_indices, d_counts, workspace};
  const size_t sizes[6] = {fb, fb, cb, cb, nb, p.bytes};
  for (int i = 0; i < 6; ++i)
    for (int j = i + 1; j < 6; ++j)
      if (overlaps(bufs[i], sizes[i], bufs[j], sizes[j])) return EF_ERR_ALIAS;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != EF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  cudaError_t err = cudaMemsetAsync(ws, 0, p.off_acc, s);  // status word and control block
  if (err == cudaSuccess) err = cudaMemsetAsync(d_counts, 0, nb, s);
  if (err != cudaSuccess) return cuda_fail(err);
  RCtl* ctl = reinterpret_cast<RCtl*>(ws + p.off_ctl);
  uint64_t* acc = reinterpret_cast<uint64_t*>(ws + p.off_acc);
  float* coef = reinterpret_cast<float*>(ws + p.off_coef);
  uint64_t* tstate = reinterpret_cast<uint64_t*>(ws + p.off_tiles);
  RSelectArgs a{coef, e, out_values, out_indices, capacity,
                reinterpret_cast<unsigned long long*>(d_counts), nseg, seed, step, tstate, ctl,
                reinterpret_cast<int32_t*>(ws), 0};
  int parity = 0;
  for (const RBatch& b : p.batches) {
    a.parity = parity;
    parity ^= 1;
    err = cudaMemsetAsync(acc, 0, (size_t)kRBatch * kChunks * 8, s);
    if (err == cudaSuccess) err = cudaMemsetAsync(tstate, 0, (size_t)std::max<int64_t>(b.tiles_b[b.nseg], 1) * 8, s);
    if (err == cudaSuccess) err = cudaMemsetAsync(&ctl->ticket, 0, 4, s);
    if (err != cudaSuccess) return cuda_fail(err);
    const int64_t ta = b.tiles_a[b.nseg], tb = b.tiles_b[b.nseg];
    const int ga = (int)std::max<int64_t>(1, std::min<int64_t>(ta, (int64_t)dev.sms * 4));
    rk_sum<<<ga, kRT, 0, s>>>(b, g_raw, e, acc);
    if ((st = check_launch()) != EF_OK) return st;
    rk_finalize<<<1, kRBatch, 0, s>>>(b, acc, coef);
    if ((st = check_launch()) != EF_OK) return st;
    if (tb > 0) {
      const int gb = (int)std::max<int64_t>(1, std::min<int64_t>(tb, (int64_t)dev.sms * 6));
      rk_select<<<gb, kRT, 0, s>>>(b, a);
      if ((st = check_launch()) != EF_OK) return st;
    }
  }
  return EF_OK;
}
