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
// Pass 2 draws and packs in three launches with no wait between warps:
// rk_draw (4 B / element + 1/8 B of keep bits) walks the aligned
// 4096-element blocks of each segment, a warp per block and each lane taking
// one quad of four elements (one Philox call, one 16-byte load), and writes
// the block's keep bits and count; rk_offsets turns the counts into packet
// offsets (the running offset carries across launches); rk_pack re-reads the
// keep bits and writes the kept elements in index order (8 B per kept
// element, + its residual write).
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
  int64_t base[2];  // kept elements before a launch: launch b reads [b % 2], its
                    // offsets kernel writes [(b + 1) % 2] (never the word being read)
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

// Group 1 of a thread's accumulator (magnitudes in [2^-62, 4), where
// gradients live) is held in registers; groups 0, 2 and 3 in the thread's
// own shared-memory slots.
struct AccSlow {
  uint64_t v[3][2][kRT];  // [group 0, 2, 3][lo, hi][thread]
};

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

// Adds |x| given as its bit pattern (sign cleared; nothing for Inf / NaN):
// m * 2^(sh - 149) goes into group sh / 64 as m << (sh % 64).
__device__ __forceinline__ void acc_add(uint64_t& lo1, uint64_t& hi1, AccSlow& slow,
                                        uint32_t bits) {
  if (bits >= 0x7F800000u) return;
  const uint32_t E = bits >> 23;
  const uint64_t m = E ? (uint64_t)((bits & 0x7FFFFFu) | 0x800000u) : (uint64_t)bits;
  const uint32_t sh = E ? E - 1 : 0;
  const uint32_t g = sh >> 6, off = sh & 63u;
  const uint64_t l = m << off;
  const uint64_t h = off > 40 ? m >> (64 - off) : 0ull;
  if (g == 1) {
    add128(lo1, hi1, l, h);
  } else {
    const int x = g == 0 ? 0 : (int)g - 1;
    uint64_t lo = slow.v[x][0][threadIdx.x], hi = slow.v[x][1][threadIdx.x];
    add128(lo, hi, l, h);
    slow.v[x][0][threadIdx.x] = lo;
    slow.v[x][1][threadIdx.x] = hi;
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

// CTA-wide flush of every thread's accumulator into the segment's chunks;
// clears the accumulator.
__device__ void acc_flush(uint64_t& lo1, uint64_t& hi1, AccSlow& slow, uint64_t* chunks,
                          uint64_t (*red)[kChunks]) {
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  uint64_t lo[4], hi[4];
  lo[1] = lo1;
  hi[1] = hi1;
#pragma unroll
  for (int x = 0; x < 3; ++x) {
    const int q = x == 0 ? 0 : x + 1;
    lo[q] = slow.v[x][0][threadIdx.x];
    hi[q] = slow.v[x][1][threadIdx.x];
    slow.v[x][0][threadIdx.x] = 0;
    slow.v[x][1][threadIdx.x] = 0;
  }
  lo1 = hi1 = 0;
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    uint64_t v = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) v += bits40(hi[q], lo[q], 40 * c - 64 * q);
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

// Pass 1: g = g_raw + e written over e; exact sum of the finite |g|.  Tiles
// are the aligned 8192-element blocks of the whole tensor cut to one
// segment, strided over the grid; a whole tile with 16-byte aligned buffers
// moves as float4 quads (thread x takes quads x + 256 u), four quads of each
// array in flight per thread; other tiles go element by element.
template <bool kVec>
__global__ void __launch_bounds__(kRT, 4)
rk_sum(RBatch b, const float* __restrict__ g_raw, float* __restrict__ e, uint64_t* acc) {
  __shared__ int64_t s_base[kRBatch + 1];
  __shared__ uint64_t red[kRT / 32][kChunks];
  __shared__ AccSlow slow;
  for (int i = threadIdx.x; i <= b.nseg; i += blockDim.x) s_base[i] = b.tiles_a[i];
#pragma unroll
  for (int x = 0; x < 3; ++x) slow.v[x][0][threadIdx.x] = slow.v[x][1][threadIdx.x] = 0;
  __syncthreads();
  const int64_t tiles = s_base[b.nseg];
  uint64_t lo1 = 0, hi1 = 0;
  int cur = -1;
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int s = find_tile_seg(s_base, b.nseg, t);
    if (s != cur) {  // uniform across the CTA
      if (cur >= 0) acc_flush(lo1, hi1, slow, acc + (int64_t)cur * kChunks, red);
      cur = s;
    }
    const RSeg& d = b.seg[s];
    const int64_t sa = (d.off / kRTile + (t - s_base[s])) * kRTile;
    const uint32_t lo = (uint32_t)max(d.off, sa), hi = (uint32_t)min(d.off + d.len, sa + kRTile);
    const uint32_t a0 = (uint32_t)sa;
    if (kVec && lo == a0 && hi == a0 + kRTile) {
      const float4* g4 = reinterpret_cast<const float4*>(g_raw) + (a0 >> 2);
      float4* e4 = reinterpret_cast<float4*>(e) + (a0 >> 2);
#pragma unroll 1
      for (int r0 = 0; r0 < kRTile / 4 / kRT; r0 += 4) {
        float4 gv[4], ev[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          gv[u] = __ldcs(g4 + (r0 + u) * kRT + threadIdx.x);
          ev[u] = __ldcs(e4 + (r0 + u) * kRT + threadIdx.x);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float4 o;
          o.x = __fadd_rn(gv[u].x, ev[u].x);
          o.y = __fadd_rn(gv[u].y, ev[u].y);
          o.z = __fadd_rn(gv[u].z, ev[u].z);
          o.w = __fadd_rn(gv[u].w, ev[u].w);
          __stcs(e4 + (r0 + u) * kRT + threadIdx.x, o);
          acc_add(lo1, hi1, slow, __float_as_uint(o.x) & 0x7FFFFFFFu);
          acc_add(lo1, hi1, slow, __float_as_uint(o.y) & 0x7FFFFFFFu);
          acc_add(lo1, hi1, slow, __float_as_uint(o.z) & 0x7FFFFFFFu);
          acc_add(lo1, hi1, slow, __float_as_uint(o.w) & 0x7FFFFFFFu);
        }
      }
    } else {
#pragma unroll 1
      for (int r0 = 0; r0 < kRTile / kRT; r0 += 8) {
        float gv[8], ev[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t i = a0 + (uint32_t)((r0 + u) * kRT) + threadIdx.x;
          gv[u] = i >= lo && i < hi ? __ldcs(g_raw + i) : 0.0f;
          ev[u] = i >= lo && i < hi ? __ldcs(e + i) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t i = a0 + (uint32_t)((r0 + u) * kRT) + threadIdx.x;
          if (i >= lo && i < hi) {
            const float g = __fadd_rn(gv[u], ev[u]);
            __stcs(e + i, g);
            acc_add(lo1, hi1, slow, __float_as_uint(g) & 0x7FFFFFFFu);
          }
        }
      }
    }
  }
  if (cur >= 0) acc_flush(lo1, hi1, slow, acc + (int64_t)cur * kChunks, red);
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

// Round keys of Philox4x32-10 for one key: key word 0 and 1 of round r are
// (seed low + r 0x9E3779B9, seed high + r 0xBB67AE85) mod 2^32.  Passed by
// value to the kernels, so a round reads them as constant operands.
struct PhiloxKeys {
  uint32_t k0[10], k1[10];
};

PhiloxKeys philox_keys(uint64_t seed) {
  PhiloxKeys k;
  uint32_t a = (uint32_t)seed, b = (uint32_t)(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    k.k0[r] = a;
    k.k1[r] = b;
    a += 0x9E3779B9u;
    b += 0xBB67AE85u;
  }
  return k;
}

// Two independent Philox4x32-10 calls, round by round.
__device__ __forceinline__ void philox4x32_10x2(uint32_t& a0, uint32_t& a1, uint32_t& a2,
                                                uint32_t& a3, uint32_t& b0, uint32_t& b1,
                                                uint32_t& b2, uint32_t& b3, const PhiloxKeys& k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t pa0 = (uint64_t)0xD2511F53u * a0, pa1 = (uint64_t)0xCD9E8D57u * a2;
    const uint64_t pb0 = (uint64_t)0xD2511F53u * b0, pb1 = (uint64_t)0xCD9E8D57u * b2;
    a0 = (uint32_t)(pa1 >> 32) ^ a1 ^ k.k0[r];
    a1 = (uint32_t)pa1;
    a2 = (uint32_t)(pa0 >> 32) ^ a3 ^ k.k1[r];
    a3 = (uint32_t)pa0;
    b0 = (uint32_t)(pb1 >> 32) ^ b1 ^ k.k0[r];
    b1 = (uint32_t)pb1;
    b2 = (uint32_t)(pb0 >> 32) ^ b3 ^ k.k1[r];
    b3 = (uint32_t)pb0;
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
  PhiloxKeys keys;
  uint32_t st0, st1;  // step low, high: counter words 2 and 3
  uint32_t* kw;      // keep words: 128 per tile, word 32 j + l = lane l's word j
  uint32_t* cnt;     // kept elements per tile
  uint32_t* csum;    // kept elements per chunk of kOffChunk tiles
  int64_t* off;      // [tiles + 1] packet position of each tile's first kept element
  RCtl* ctl;
  int32_t* status;
  int parity;  // launch number % 2
};

// Pass-2 tiles are the aligned 4096-element blocks of the whole tensor
// (global index / 4096) cut to one segment, so every quad of four elements
// that shares a Philox counter lies in one tile.  A warp walks a tile's 1024
// quads in 32 rounds of 32: in a round lane l takes quad 32 r + l, loads its
// four elements at once (16 bytes when e is 16-byte aligned), computes its
// one Philox call and sets four keep bits (bit 4 (r % 8) + u of word r / 8
// for element u of the quad).
constexpr int kRWarps = kRT / 32;
constexpr int kRSelTile = 4096;                 // elements per pass-2 tile (one warp)
constexpr int kRWords = kRSelTile / 1024;       // 4 keep words per lane
constexpr int kDrawCtas = 5;                    // rk_draw CTAs per SM (48 registers)
constexpr int kOffChunk = 8192;                 // tiles per rk_offsets CTA
constexpr int kOffPer = kOffChunk / kRT;        // 32 tiles per thread

// The four elements of quad q; with kAll every one of them is in the tile.
// Element indices are below 2^31, so quads and elements fit 32 bits.
template <bool kVec, bool kAll>
__device__ __forceinline__ float4 rk_load_quad(const float* e, uint32_t q, uint32_t lo,
                                               uint32_t hi) {
  const uint32_t i = 4 * q;
  if (kAll) {
    if (kVec) return reinterpret_cast<const float4*>(e)[q];
    return make_float4(e[i], e[i + 1], e[i + 2], e[i + 3]);
  }
  float4 v;
  v.x = (i >= lo && i < hi) ? e[i] : 0.0f;
  v.y = (i + 1 >= lo && i + 1 < hi) ? e[i + 1] : 0.0f;
  v.z = (i + 2 >= lo && i + 2 < hi) ? e[i + 2] : 0.0f;
  v.w = (i + 3 >= lo && i + 3 < hi) ? e[i + 3] : 0.0f;
  return v;
}

// u < min(1, x) is !(u >= x) for every x, since u < 1 (x >= 1, +Inf and a
// NaN product all keep).
__device__ __forceinline__ bool rk_keep(uint32_t w, float c, float g) {
  const float x = __fmul_rn(c, fabsf(g));
  return !(__uint2float_rn(w >> 8) * 0x1p-24f >= x);
}

// Keep bits of quad q (element u at bit u).
template <bool kAll>
__device__ __forceinline__ uint32_t rk_quad_bits(uint32_t q, const float4& v, float c,
                                                 uint32_t w0, uint32_t w1, uint32_t w2,
                                                 uint32_t w3, uint32_t lo, uint32_t hi) {
  bool k[4] = {rk_keep(w0, c, v.x), rk_keep(w1, c, v.y), rk_keep(w2, c, v.z),
               rk_keep(w3, c, v.w)};
  uint32_t bits = 0;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    if (!kAll) k[u] = k[u] && 4 * q + u >= lo && 4 * q + u < hi;
    if (k[u]) bits |= 1u << u;
  }
  return bits;
}

// Keep words of one tile starting at quad q0, written to kwt[32 j + lane];
// returns the number of kept elements of this lane.  Two rounds at a time,
// so that two independent Philox calls interleave.  The counter's high word
// (quad index / 2^32) is 0 for every quad of an int32-indexed tensor.
template <bool kVec, bool kAll>
__device__ __forceinline__ uint32_t rk_slice(const float* e, uint32_t q0, uint32_t lo, uint32_t hi,
                                             float c, const PhiloxKeys& keys, uint32_t st0,
                                             uint32_t st1, uint32_t* kwt) {
  const unsigned lane = lane_id();
  uint32_t cnt = 0;
#pragma unroll 1
  for (int j = 0; j < kRWords; ++j) {
    uint32_t kb = 0;
#pragma unroll
    for (int r = 0; r < 8; r += 2) {
      const uint32_t qa = q0 + 32u * (8 * j + r) + lane, qb = qa + 32;
      const float4 va = rk_load_quad<kVec, kAll>(e, qa, lo, hi);
      const float4 vb = rk_load_quad<kVec, kAll>(e, qb, lo, hi);
      uint32_t a0 = qa, a1 = 0, a2 = st0, a3 = st1;
      uint32_t b0 = qb, b1 = 0, b2 = st0, b3 = st1;
      philox4x32_10x2(a0, a1, a2, a3, b0, b1, b2, b3, keys);
      kb |= rk_quad_bits<kAll>(qa, va, c, a0, a1, a2, a3, lo, hi) << (4 * r);
      kb |= rk_quad_bits<kAll>(qb, vb, c, b0, b1, b2, b3, lo, hi) << (4 * r + 4);
    }
    kwt[32 * j + lane] = kb;
    cnt += __popc(kb);
  }
  return cnt;
}

// Tile t's segment and the bounds [lo, hi) of its elements; returns the
// first quad of its aligned block.
__device__ __forceinline__ int64_t rk_tile(const RBatch& b, const int64_t* s_base, int64_t t,
                                           int* seg, int64_t* lo, int64_t* hi) {
  const int s = find_tile_seg(s_base, b.nseg, t);
  const RSeg& d = b.seg[s];
  const int64_t sa = (d.off / kRSelTile + (t - s_base[s])) * kRSelTile;
  *seg = s;
  *lo = max(d.off, sa);
  *hi = min(d.off + d.len, sa + kRSelTile);
  return sa >> 2;
}

// Pass 2a: keep bits and counts, one warp per tile, tiles strided over the
// grid's warps.
template <bool kVec>
__global__ void __launch_bounds__(kRT, kDrawCtas)
rk_draw(RBatch b, RSelectArgs a) {
  __shared__ int64_t s_base[kRBatch + 1];
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i <= b.nseg; i += blockDim.x) s_base[i] = b.tiles_b[i];
  __syncthreads();
  const int64_t tiles = s_base[b.nseg];
  for (int64_t t = (int64_t)blockIdx.x * kRWarps + warp; t < tiles;
       t += (int64_t)gridDim.x * kRWarps) {
    int s;
    int64_t lo, hi;
    const int64_t q0 = rk_tile(b, s_base, t, &s, &lo, &hi);
    const float c = a.coef[s];
    uint32_t* kwt = a.kw + t * (32 * kRWords);
    const uint32_t q = (uint32_t)q0, l = (uint32_t)lo, h = (uint32_t)hi;
    const uint32_t cnt = (l == 4 * q && h == 4 * q + kRSelTile)
                             ? rk_slice<kVec, true>(a.e, q, l, h, c, a.keys, a.st0, a.st1, kwt)
                             : rk_slice<kVec, false>(a.e, q, l, h, c, a.keys, a.st0, a.st1, kwt);
    const uint32_t run = __reduce_add_sync(kFull, cnt);
    if (lane == 0) {
      a.cnt[t] = run;
      if (run) atomicAdd(&a.csum[t / kOffChunk], run);
    }
  }
}

// Pass 2b: packet offsets.  CTA c scans the counts of tiles
// [c kOffChunk, (c + 1) kOffChunk) on top of the kept elements before the
// launch and of the earlier chunks; the last CTA closes the launch (total,
// capacity status, base of the next launch).
__global__ void __launch_bounds__(kRT)
rk_offsets(int64_t tiles, RSelectArgs a) {
  __shared__ uint32_t scratch[40];
  __shared__ int64_t s_pre;
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  const int64_t c = blockIdx.x;
  if (warp == 0) {
    uint64_t v = 0;
    for (int64_t x = lane; x < c; x += 32) v += a.csum[x];
    v = warp_sum_u64(v);
    if (lane == 0)
      s_pre = *reinterpret_cast<volatile int64_t*>(&a.ctl->base[a.parity]) + (int64_t)v;
  }
  const int64_t t0 = c * kOffChunk + (int64_t)threadIdx.x * kOffPer;
  uint32_t v[kOffPer];
  uint32_t mine = 0;
  if (t0 + kOffPer <= tiles) {  // 128-byte aligned: the array is, and t0 % 32 == 0
#pragma unroll
    for (int x = 0; x < kOffPer; x += 4) {
      const uint4 q = *reinterpret_cast<const uint4*>(a.cnt + t0 + x);
      v[x] = q.x;
      v[x + 1] = q.y;
      v[x + 2] = q.z;
      v[x + 3] = q.w;
    }
  } else {
#pragma unroll
    for (int x = 0; x < kOffPer; ++x) v[x] = t0 + x < tiles ? a.cnt[t0 + x] : 0u;
  }
#pragma unroll
  for (int x = 0; x < kOffPer; ++x) mine += v[x];
  uint32_t total;
  const uint32_t ex = block_excl_scan(mine, scratch, &total);  // synchronises s_pre too
  int64_t pos = s_pre + (int64_t)ex;
#pragma unroll
  for (int x = 0; x < kOffPer; ++x) {
    if (t0 + x < tiles) a.off[t0 + x] = pos;
    pos += v[x];
  }
  if (c == gridDim.x - 1 && threadIdx.x == 0) {
    const int64_t all = s_pre + (int64_t)total;
    a.off[tiles] = all;
    a.ctl->base[a.parity ^ 1] = all;
    a.counts[a.nseg_total] = (unsigned long long)min(all, a.capacity);
    if (all > a.capacity) set_status(a.status, EF_ERR_CAPACITY);
  }
}

// Pass 2c: the ordered packet.  One warp per tile with kept elements: ranks
// from a warp scan of the lanes' counts round by round, values re-read from
// e and e set to +0 at every element that fits the packet.  The first
// threads of CTA 0 write the per-segment counts.
__global__ void __launch_bounds__(kRT)
rk_pack(RBatch b, RSelectArgs a) {
  __shared__ int64_t s_base[kRBatch + 1];
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i <= b.nseg; i += blockDim.x) s_base[i] = b.tiles_b[i];
  __syncthreads();
  const int64_t tiles = s_base[b.nseg];
  if (blockIdx.x == 0 && threadIdx.x < b.nseg) {
    const int64_t lo = min(a.off[s_base[threadIdx.x]], a.capacity);
    const int64_t hi = min(a.off[s_base[threadIdx.x + 1]], a.capacity);
    a.counts[b.seg[threadIdx.x].id] = (unsigned long long)(hi - lo);
  }
  for (int64_t t = (int64_t)blockIdx.x * kRWarps + warp; t < tiles;
       t += (int64_t)gridDim.x * kRWarps) {
    if (a.cnt[t] == 0) continue;  // warp-uniform
    int64_t pos = a.off[t];
    if (pos >= a.capacity) continue;
    int s;
    int64_t lo, hi;
    const int64_t q0 = rk_tile(b, s_base, t, &s, &lo, &hi);
    const uint32_t* kwt = a.kw + t * (32 * kRWords);
    uint32_t kbs[kRWords];
#pragma unroll
    for (int j = 0; j < kRWords; ++j) kbs[j] = kwt[32 * j + lane];
#pragma unroll
    for (int j = 0; j < kRWords; ++j) {
      const uint32_t kb = kbs[j];
      // rounds with a kept element anywhere in the warp, lowest first
      const uint32_t any = __reduce_or_sync(kFull, kb);
      uint32_t rounds = 0;
#pragma unroll
      for (int r = 0; r < 8; ++r) rounds |= ((any >> (4 * r)) & 0xFu) ? 1u << r : 0u;
      while (rounds) {
        const int r = __ffs(rounds) - 1;
        rounds &= rounds - 1;
        const uint32_t nib = (kb >> (4 * r)) & 0xFu;
        const uint32_t n4 = __popc(nib);
        const uint32_t incl = warp_incl_scan(n4);
        int64_t p = pos + (incl - n4);
        const int64_t i = 4 * (q0 + 32 * (8 * j + r) + lane);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if ((nib >> u) & 1u) {
            if (p < a.capacity) {
              a.out_values[p] = a.e[i + u];
              a.out_indices[p] = (int32_t)(i + u);
              a.e[i + u] = 0.0f;
            }
            ++p;
          }
        }
        pos += __shfl_sync(kFull, incl, 31);
      }
    }
  }
}

struct RPlan {
  std::vector<RBatch> batches;
  int64_t max_tiles_b = 0;
  size_t off_acc = 0, off_coef = 0, off_ctl = 0, off_kw = 0, off_cnt = 0, off_csum = 0,
         off_off = 0, bytes = 0;
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
    // aligned blocks the segment meets, in each pass
    const int64_t blocks_a = (b - 1) / kRTile - a / kRTile + 1;
    const int64_t blocks_b = (b - 1) / kRSelTile - a / kRSelTile + 1;
    cur.seg[t] = RSeg{a, len, k, cur.tiles_a[t], cur.tiles_b[t], i};
    cur.tiles_a[t + 1] = cur.tiles_a[t] + blocks_a;
    cur.tiles_b[t + 1] = cur.tiles_b[t] + (k > 0 ? blocks_b : 0);
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
  const size_t tb = (size_t)std::max<int64_t>(p->max_tiles_b, 1);
  p->off_kw = off;
  off = round_up(off + tb * 4 * 32 * kRWords, 256);
  p->off_cnt = off;
  off = round_up(off + tb * 4, 256);
  p->off_csum = off;
  off = round_up(off + (tb + kOffChunk - 1) / kOffChunk * 4, 256);
  p->off_off = off;
  off = round_up(off + (tb + 1) * 8, 256);
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
  RSelectArgs a{coef,
                e,
                out_values,
                out_indices,
                capacity,
                reinterpret_cast<unsigned long long*>(d_counts),
                nseg,
                philox_keys(seed),
                (uint32_t)step,
                (uint32_t)(step >> 32),
                reinterpret_cast<uint32_t*>(ws + p.off_kw),
                reinterpret_cast<uint32_t*>(ws + p.off_cnt),
                reinterpret_cast<uint32_t*>(ws + p.off_csum),
                reinterpret_cast<int64_t*>(ws + p.off_off),
                ctl,
                reinterpret_cast<int32_t*>(ws),
                0};
  // 16-byte accesses: pass 1 needs both arrays aligned, pass 2 only e
  const bool vec_e = (reinterpret_cast<uintptr_t>(e) & 15u) == 0;
  const bool vec = vec_e && (reinterpret_cast<uintptr_t>(g_raw) & 15u) == 0;
  int parity = 0;
  for (const RBatch& b : p.batches) {
    a.parity = parity;
    parity ^= 1;
    const int64_t ta = b.tiles_a[b.nseg], tb = b.tiles_b[b.nseg];
    const int64_t nchunks = std::max<int64_t>(1, (tb + kOffChunk - 1) / kOffChunk);
    err = cudaMemsetAsync(acc, 0, (size_t)kRBatch * kChunks * 8, s);
    if (err == cudaSuccess) err = cudaMemsetAsync(a.csum, 0, (size_t)nchunks * 4, s);
    if (err != cudaSuccess) return cuda_fail(err);
    const int ga = (int)std::max<int64_t>(1, std::min<int64_t>(ta, (int64_t)dev.sms * 4));
    if (vec) rk_sum<true><<<ga, kRT, 0, s>>>(b, g_raw, e, acc);
    else rk_sum<false><<<ga, kRT, 0, s>>>(b, g_raw, e, acc);
    if ((st = check_launch()) != EF_OK) return st;
    rk_finalize<<<1, kRBatch, 0, s>>>(b, acc, coef);
    if ((st = check_launch()) != EF_OK) return st;
    const int64_t warps = (tb + kRWarps - 1) / kRWarps;
    if (tb > 0) {
      const int gd =
          (int)std::max<int64_t>(1, std::min<int64_t>(warps, (int64_t)dev.sms * kDrawCtas));
      if (vec_e) rk_draw<true><<<gd, kRT, 0, s>>>(b, a);
      else rk_draw<false><<<gd, kRT, 0, s>>>(b, a);
      if ((st = check_launch()) != EF_OK) return st;
    }
    // always: it carries the running offset to the next launch
    rk_offsets<<<(unsigned)nchunks, kRT, 0, s>>>(tb, a);
    if ((st = check_launch()) != EF_OK) return st;
    if (tb > 0) {
      const int gp = (int)std::max<int64_t>(1, std::min<int64_t>(warps, (int64_t)dev.sms * 8));
      rk_pack<<<gp, kRT, 0, s>>>(b, a);
      if ((st = check_launch()) != EF_OK) return st;
    }
  }
  return EF_OK;
}
