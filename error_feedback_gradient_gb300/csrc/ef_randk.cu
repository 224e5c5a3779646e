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
// The draws u_i do not depend on g, and RN32(c |g_i|) never decreases as c
// grows, so for any c_max >= c every kept element passes the keep test at
// c_max.  The passes use that to read g once:
//   rk_sample sums |g| over a block sample of each long segment; c_max is
//     twice the coefficient that sum predicts (+Inf for short segments);
//   rk_sum (12 B / element + 1/8 B of candidate bits) writes g = g_raw + e
//     over e, sums |g| exactly and, with one Philox call per quad of four
//     elements, sets a candidate bit where u_i < RN32(c_max |g_i|);
//   rk_finalize rounds the exact sum, forms c and checks c <= c_max;
//   rk_refine re-tests the candidates at c (every element of a segment where
//     c > c_max or c_max is +Inf) and leaves the exact keep bits and counts;
//   rk_offsets turns the counts into packet offsets (the running offset
//     carries across launches) and rk_pack writes the packet in index order.
// The exact sum: a float32 magnitude is m * 2^(sh - 149) with m < 2^24 and
// 0 <= sh <= 253; each thread keeps a 128-bit integer accumulator per
// 64-bit-aligned group of sh, and a CTA flushes them as 40-bit carry-save
// chunks with one atomicAdd per chunk when it leaves a segment (sums of at
// most 2^14 flushes of 2^50 fit in 64 bits).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "ef_common.cuh"

namespace ef {
namespace {

constexpr int kRT = 256;                   // threads per CTA
constexpr int kRTile = 8192;               // elements per tile (aligned blocks of the tensor)
constexpr int kRTileWords = kRTile / 32;   // 256 keep words per tile
constexpr int kRBatch = 128;               // segments per launch
constexpr int kChunks = 8;                 // 40-bit chunks of an exact sum (320 bits)
constexpr uint64_t kMask40 = (1ull << 40) - 1;
constexpr int kSampleBlock = 64;           // elements per sampled block
constexpr int kSampleBlocksMax = 2048;     // sampled blocks per segment
constexpr int64_t kSampleMinLen = 65536;   // shorter segments test every element at c
constexpr int kOffChunk = 8192;            // tiles per rk_offsets CTA
constexpr int kOffPer = kOffChunk / kRT;   // 32 tiles per thread

struct RSeg {
  int64_t off, len, k;
  int64_t sblk;   // first sample block of the segment in the launch
  int32_t nsamp;  // sampled blocks (0: c_max = +Inf)
  int32_t id;     // segment number in the whole call
};

// Tiles are the aligned 8192-element blocks of the tensor cut to one
// segment: tile t of segment s covers [max(off, B), min(off + len, B + 8192))
// with B = (off / 8192 + t - tiles[s]) * 8192, so every quad of four
// elements (one Philox counter) lies in one tile.  Keep word x (0..255) of a
// tile holds quads B / 4 + x + 256 u (u = 0..7), element j of quad u at bit
// 4 u + j.
struct RBatch {
  RSeg seg[kRBatch];
  int64_t tiles[kRBatch + 1];  // prefix of tiles; [nseg] = total
  int64_t samp[kRBatch + 1];   // prefix of sampled blocks
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

// First element of tile t's aligned block, and the tile's bounds [lo, hi).
__device__ __forceinline__ uint32_t tile_bounds(const RSeg& d, int64_t first_tile, int64_t t,
                                                uint32_t* lo, uint32_t* hi) {
  const int64_t sa = (d.off / kRTile + (t - first_tile)) * kRTile;
  *lo = (uint32_t)max(d.off, sa);
  *hi = (uint32_t)min(d.off + d.len, sa + kRTile);
  return (uint32_t)sa;
}

// ---------------------------------------------------------------- draws

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

// The four words of Philox4x32-10 at counter (q, 0, st0, st1): the counter's
// high word (quad index / 2^32) is 0 for every quad of an int32-indexed
// tensor.
__device__ __forceinline__ void philox_quad(uint32_t q, uint32_t st0, uint32_t st1,
                                            const PhiloxKeys& k, uint32_t w[4]) {
  uint32_t c0 = q, c1 = 0, c2 = st0, c3 = st1;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c0;  // one 32x32->64 multiply each
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    c0 = (uint32_t)(p1 >> 32) ^ c1 ^ k.k0[r];
    c1 = (uint32_t)p1;
    c2 = (uint32_t)(p0 >> 32) ^ c3 ^ k.k1[r];
    c3 = (uint32_t)p0;
  }
  w[0] = c0;
  w[1] = c1;
  w[2] = c2;
  w[3] = c3;
}

// u < min(1, x) is !(u >= x) for every x, since u < 1 (x >= 1, +Inf and a
// NaN product all keep).
__device__ __forceinline__ bool rk_keep(uint32_t w, float c, float g) {
  const float x = __fmul_rn(c, fabsf(g));
  return !(__uint2float_rn(w >> 8) * 0x1p-24f >= x);
}

// Keep bits of one quad at coefficient c, element j at bit j, restricted to
// `mask`.
__device__ __forceinline__ uint32_t quad_keep(const float v[4], const uint32_t w[4], float c,
                                              uint32_t mask) {
  uint32_t bits = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (((mask >> j) & 1u) && rk_keep(w[j], c, v[j])) bits |= 1u << j;
  return bits;
}

// c_max of a segment from its sampled sum: twice the coefficient the sample
// predicts, rounded up; +Inf when the segment is not sampled or its sample
// sums to 0.  rk_sum and rk_finalize evaluate the same expression.
__device__ __forceinline__ float seg_cmax(const RSeg& d, double ssum) {
  if (d.nsamp == 0 || !(ssum > 0.0)) return __int_as_float(0x7F800000);
  const double m = (double)d.nsamp * kSampleBlock;
  return __double2float_ru(__ddiv_rn(2.0 * (double)d.k * m, (double)d.len * ssum));
}

struct RSelectArgs {
  float* coef;
  int32_t* mode;     // per segment: 1 = candidate bits hold every kept element
  const double* ssum;
  float* e;
  float* out_values;
  int32_t* out_indices;
  int64_t capacity;
  unsigned long long* counts;  // [nseg + 1] of the whole call
  int32_t nseg_total;
  PhiloxKeys keys;
  uint32_t st0, st1;  // step low, high: counter words 2 and 3
  uint32_t* kw;       // keep words, kRTileWords per tile
  uint32_t* cnt;      // kept elements per tile
  uint32_t* csum;     // kept elements per chunk of kOffChunk tiles
  int64_t* off;       // [tiles + 1] packet position of each tile's first kept element
  RCtl* ctl;
  int32_t* status;
  int parity;  // launch number % 2
};

// Sampled sum of |g_raw + e| over the finite elements of up to 2048 blocks
// of 64 per long segment (block b starts b * (len / nsamp) into it), one
// warp per block, added into ssum[s] in float64.  It only sets c_max.
__global__ void __launch_bounds__(kRT)
rk_sample(RBatch b, const float* __restrict__ g_raw, const float* __restrict__ e,
          double* ssum) {
  pdl_wait();
  __shared__ int64_t s_base[kRBatch + 1];
  for (int i = threadIdx.x; i <= b.nseg; i += blockDim.x) s_base[i] = b.samp[i];
  __syncthreads();
  const unsigned lane = lane_id();
  const int64_t total = s_base[b.nseg];
  for (int64_t blk = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; blk < total;
       blk += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int s = find_tile_seg(s_base, b.nseg, blk);
    const RSeg& d = b.seg[s];
    const int64_t i0 = d.off + (blk - s_base[s]) * (d.len / d.nsamp);
    float a = 0.0f;
#pragma unroll
    for (int u = 0; u < kSampleBlock / 32; ++u) {
      const int64_t i = i0 + 32 * u + lane;
      const float m = fabsf(__fadd_rn(g_raw[i], e[i]));
      if (m < __int_as_float(0x7F800000)) a += m;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(kFull, a, o);
    if (lane == 0 && a > 0.0f) atomicAdd(&ssum[s], (double)a);
  }
}

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

// Magnitudes with biased exponent E in [97, 129) (|x| in [2^-30, 4): sh in
// [96, 128), bits 32..63 of group 1) are added as M << (E - 97) into a
// 64-bit window accumulator; at most 32 of them (< 2^60) between folds.
// Others take acc_add.
__device__ __forceinline__ void acc_add_window(uint64_t& win, uint64_t& lo1, uint64_t& hi1,
                                               AccSlow& slow, uint32_t bits) {
  const uint32_t d = (bits >> 23) - 97u;
  if (d < 32u) win += (uint64_t)((bits & 0x7FFFFFu) | 0x800000u) << d;
  else acc_add(lo1, hi1, slow, bits);
}

// Folds the window accumulator into group 1 (at bit 32) and clears it.
__device__ __forceinline__ void acc_fold_window(uint64_t& win, uint64_t& lo1, uint64_t& hi1) {
  add128(lo1, hi1, win << 32, win >> 32);
  win = 0;
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

// Pass 1: g = g_raw + e written over e; exact sum of the finite |g|; the
// candidate bits at c_max.  A CTA takes whole tiles, strided over the grid:
// thread x takes quads x + 256 u of the tile (u = 0..7), so it writes keep
// word x.  A whole tile with 16-byte aligned buffers moves as float4 quads,
// four quads of each array in flight per thread; other tiles go element by
// element.
template <bool kVec>
__global__ void __launch_bounds__(kRT, 3)
rk_sum(RBatch b, const float* __restrict__ g_raw, float* __restrict__ e, uint64_t* acc,
       RSelectArgs a) {
  pdl_wait();
  __shared__ int64_t s_base[kRBatch + 1];
  __shared__ uint64_t red[kRT / 32][kChunks];
  __shared__ AccSlow slow;
  for (int i = threadIdx.x; i <= b.nseg; i += blockDim.x) s_base[i] = b.tiles[i];
#pragma unroll
  for (int x = 0; x < 3; ++x) slow.v[x][0][threadIdx.x] = slow.v[x][1][threadIdx.x] = 0;
  __syncthreads();
  const int64_t tiles = s_base[b.nseg];
  uint64_t lo1 = 0, hi1 = 0;
  int cur = -1;
  float cmax = 0.0f;
  bool draw = false;
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int s = find_tile_seg(s_base, b.nseg, t);
    if (s != cur) {  // uniform across the CTA
      if (cur >= 0) acc_flush(lo1, hi1, slow, acc + (int64_t)cur * kChunks, red);
      cur = s;
      cmax = seg_cmax(b.seg[s], a.ssum[s]);
      draw = b.seg[s].k > 0 && cmax < __int_as_float(0x7F800000);
    }
    const RSeg& d = b.seg[s];
    uint32_t lo, hi;
    const uint32_t a0 = tile_bounds(d, s_base[s], t, &lo, &hi);
    const uint32_t q0 = a0 >> 2;
    uint32_t word = 0;
    uint64_t win = 0;
    if (kVec && lo == a0 && hi == a0 + kRTile) {
      const float4* g4 = reinterpret_cast<const float4*>(g_raw) + q0;
      float4* e4 = reinterpret_cast<float4*>(e) + q0;
#pragma unroll 1
      for (int r0 = 0; r0 < 8; r0 += 4) {
        float4 gv[4], ev[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          gv[u] = __ldcs(g4 + (r0 + u) * kRT + threadIdx.x);
          ev[u] = __ldcs(e4 + (r0 + u) * kRT + threadIdx.x);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float o[4];
          o[0] = __fadd_rn(gv[u].x, ev[u].x);
          o[1] = __fadd_rn(gv[u].y, ev[u].y);
          o[2] = __fadd_rn(gv[u].z, ev[u].z);
          o[3] = __fadd_rn(gv[u].w, ev[u].w);
          __stcs(e4 + (r0 + u) * kRT + threadIdx.x, make_float4(o[0], o[1], o[2], o[3]));
#pragma unroll
          for (int j = 0; j < 4; ++j)
            acc_add_window(win, lo1, hi1, slow, __float_as_uint(o[j]) & 0x7FFFFFFFu);
          if (draw) {
            uint32_t w[4];
            philox_quad(q0 + (uint32_t)((r0 + u) * kRT) + threadIdx.x, a.st0, a.st1, a.keys, w);
            word |= quad_keep(o, w, cmax, 0xFu) << (4 * (r0 + u));
          }
        }
      }
    } else {
#pragma unroll 1
      for (int u = 0; u < 8; ++u) {
        const uint32_t q = q0 + (uint32_t)(u * kRT) + threadIdx.x;
        float o[4];
        uint32_t mask = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t i = 4 * q + j;
          o[j] = 0.0f;
          if (i >= lo && i < hi) {
            o[j] = __fadd_rn(__ldcs(g_raw + i), __ldcs(e + i));
            __stcs(e + i, o[j]);
            acc_add_window(win, lo1, hi1, slow, __float_as_uint(o[j]) & 0x7FFFFFFFu);
            mask |= 1u << j;
          }
        }
        if (draw && mask) {
          uint32_t w[4];
          philox_quad(q, a.st0, a.st1, a.keys, w);
          word |= quad_keep(o, w, cmax, mask) << (4 * u);
        }
      }
    }
    acc_fold_window(win, lo1, hi1);
    if (draw) a.kw[t * kRTileWords + threadIdx.x] = word;
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

__global__ void rk_finalize(RBatch b, const uint64_t* acc, RSelectArgs a) {
  pdl_trigger();
  pdl_wait();
  const int s = threadIdx.x;
  if (s >= b.nseg) return;
  const double S = exact_to_double(acc + (int64_t)s * kChunks);
  const float c = S > 0.0 ? __double2float_rn(__ddiv_rn((double)b.seg[s].k, S)) : 0.0f;
  const float cmax = seg_cmax(b.seg[s], a.ssum[s]);
  a.coef[s] = c;
  a.mode[s] = (b.seg[s].k > 0 && cmax < __int_as_float(0x7F800000) && c <= cmax) ? 1 : 0;
}

// Candidate bits of keep word x: every element of the tile in [lo, hi).
__device__ __forceinline__ uint32_t all_word(uint32_t q0, uint32_t x, uint32_t lo, uint32_t hi,
                                             bool whole) {
  if (whole) return 0xFFFFFFFFu;
  uint32_t w = 0;
#pragma unroll
  for (int u = 0; u < 8; ++u)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t i = 4 * (q0 + x + 256u * u) + j;
      if (i >= lo && i < hi) w |= 1u << (4 * u + j);
    }
  return w;
}

// Nonzero nibbles of w, as bit 4u for nibble u.
__device__ __forceinline__ uint32_t nz_nibbles(uint32_t w) {
  w |= w >> 1;
  w |= w >> 2;
  return w & 0x11111111u;
}

constexpr int kRefineList = 256;  // candidate quads a warp re-tests lane-parallel per tile

// The candidates of quad q given as nibble `nib` at coefficient c: their
// values from e (a 16-byte load for a whole quad when e is 16-byte
// aligned), one Philox call, the keep test.
template <bool kVec>
__device__ __forceinline__ uint32_t refine_quad(const RSelectArgs& a, uint32_t q, uint32_t nib,
                                                float c) {
  float v[4];
  if (kVec && nib == 0xFu) {
    const float4 f = reinterpret_cast<const float4*>(a.e)[q];
    v[0] = f.x;
    v[1] = f.y;
    v[2] = f.z;
    v[3] = f.w;
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = ((nib >> j) & 1u) ? a.e[4 * q + j] : 0.0f;
  }
  uint32_t w[4];
  philox_quad(q, a.st0, a.st1, a.keys, w);
  return quad_keep(v, w, c, nib);
}

// Pass 2a: exact keep bits and counts, one warp per tile, tiles strided over
// the grid's warps.  Lane l holds the tile's words l + 32 m.  With few
// candidate quads the warp lists them in shared memory and re-tests them one
// per lane (one Philox round for up to 32 quads); otherwise, and where
// every element is tested, each lane walks its own words.
template <bool kVec>
__global__ void __launch_bounds__(kRT, 4)
rk_refine(RBatch b, RSelectArgs a) {
  pdl_trigger();
  pdl_wait();
  constexpr int kM = kRTileWords / 32;
  __shared__ int64_t s_base[kRBatch + 1];
  __shared__ uint32_t s_in[kRT / 32][kRTileWords], s_out[kRT / 32][kRTileWords];
  __shared__ uint16_t s_list[kRT / 32][kRefineList];
  for (int i = threadIdx.x; i <= b.nseg; i += blockDim.x) s_base[i] = b.tiles[i];
  __syncthreads();
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  const int64_t tiles = s_base[b.nseg];
  const int64_t stride = ((int64_t)gridDim.x * blockDim.x) >> 5;
  int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  // the words of the warp's next tile are loaded while it works on this one
  uint32_t nxt[kM];
#pragma unroll
  for (int m = 0; m < kM; ++m) nxt[m] = t < tiles ? a.kw[t * kRTileWords + lane + 32 * m] : 0u;
  for (; t < tiles; t += stride) {
    uint32_t wd[kM];
#pragma unroll
    for (int m = 0; m < kM; ++m) {
      wd[m] = nxt[m];
      nxt[m] = t + stride < tiles ? a.kw[(t + stride) * kRTileWords + lane + 32 * m] : 0u;
    }
    const int s = find_tile_seg(s_base, b.nseg, t);
    const RSeg& d = b.seg[s];
    uint32_t cnt = 0;
    if (d.k > 0) {  // warp-uniform
      const float c = a.coef[s];
      const bool cand = a.mode[s] != 0;
      uint32_t lo, hi;
      const uint32_t a0 = tile_bounds(d, s_base[s], t, &lo, &hi);
      const uint32_t q0 = a0 >> 2;
      const bool whole = lo == a0 && hi == a0 + kRTile;
      uint32_t* kwt = a.kw + t * kRTileWords;
      uint32_t nq = 0;
#pragma unroll
      for (int m = 0; m < kM; ++m) {
        if (!cand) wd[m] = all_word(q0, lane + 32u * m, lo, hi, whole);
        nq += __popc(nz_nibbles(wd[m]));
      }
      const uint32_t incl = warp_incl_scan(nq);
      const uint32_t total = __shfl_sync(kFull, incl, 31);
      if (total <= (uint32_t)kRefineList) {
        uint32_t p = incl - nq;
#pragma unroll
        for (int m = 0; m < kM; ++m) {
          const uint32_t x = lane + 32u * m;
          s_in[warp][x] = wd[m];
          s_out[warp][x] = 0;
          uint32_t z = nz_nibbles(wd[m]);
          while (z) {
            const uint32_t bpos = __ffs(z) - 1;
            z &= z - 1;
            s_list[warp][p++] = (uint16_t)((x << 3) | (bpos >> 2));
          }
        }
        __syncwarp();
        for (uint32_t i = lane; i < total; i += 32) {
          const uint32_t ent = s_list[warp][i];
          const uint32_t x = ent >> 3, u = ent & 7u;
          const uint32_t nib = (s_in[warp][x] >> (4 * u)) & 0xFu;
          const uint32_t bits = refine_quad<kVec>(a, q0 + x + 256u * u, nib, c);
          if (bits) atomicOr(&s_out[warp][x], bits << (4 * u));
        }
        __syncwarp();
#pragma unroll
        for (int m = 0; m < kM; ++m) {
          const uint32_t out = s_out[warp][lane + 32 * m];
          kwt[lane + 32 * m] = out;
          cnt += __popc(out);
        }
        __syncwarp();
      } else {
#pragma unroll
        for (int m = 0; m < kM; ++m) {
          const uint32_t x = lane + 32u * m;
          uint32_t word = wd[m], out = 0;
          while (word) {
            const int u = (__ffs(word) - 1) >> 2;
            const uint32_t nib = (word >> (4 * u)) & 0xFu;
            word &= ~(0xFu << (4 * u));
            out |= refine_quad<kVec>(a, q0 + x + 256u * u, nib, c) << (4 * u);
          }
          kwt[x] = out;
          cnt += __popc(out);
        }
      }
    }
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
  pdl_trigger();
  pdl_wait();
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

// Pass 2c: the ordered packet.  One warp per tile with kept elements.  With
// at most 32 of them the warp lists their offsets in the tile in shared
// memory, one per lane, and ranks each by counting the smaller ones.
// Otherwise it walks the tile in index order, quad group u, then word, then
// lane, so a round (u, m) takes nibble u of the lanes' words l + 32 m, with
// ranks from a warp scan of the lanes' counts.  Values are re-read from e
// and e is set to +0 at every element that fits the packet.  The first
// threads of CTA 0 write the per-segment counts.
__global__ void __launch_bounds__(kRT)
rk_pack(RBatch b, RSelectArgs a) {
  pdl_wait();
  constexpr int kM = kRTileWords / 32;
  __shared__ int64_t s_base[kRBatch + 1];
  __shared__ uint16_t s_keys[kRT / 32][32];
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i <= b.nseg; i += blockDim.x) s_base[i] = b.tiles[i];
  __syncthreads();
  const int64_t tiles = s_base[b.nseg];
  if (blockIdx.x == 0 && threadIdx.x < b.nseg) {
    const int64_t lo = min(a.off[s_base[threadIdx.x]], a.capacity);
    const int64_t hi = min(a.off[s_base[threadIdx.x + 1]], a.capacity);
    a.counts[b.seg[threadIdx.x].id] = (unsigned long long)(hi - lo);
  }
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < tiles;
       t += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const uint32_t total = a.cnt[t];
    if (total == 0) continue;  // warp-uniform
    int64_t pos = a.off[t];
    if (pos >= a.capacity) continue;
    const int s = find_tile_seg(s_base, b.nseg, t);
    uint32_t lo, hi;
    const uint32_t a0 = tile_bounds(b.seg[s], s_base[s], t, &lo, &hi);
    const uint32_t q0 = a0 >> 2;
    const uint32_t* kwt = a.kw + t * kRTileWords;
    uint32_t wd[kM];
    uint32_t mine = 0;
#pragma unroll
    for (int m = 0; m < kM; ++m) {
      wd[m] = kwt[lane + 32 * m];
      mine += __popc(wd[m]);
    }
    if (total <= 32) {
      const uint32_t incl = warp_incl_scan(mine);
      uint32_t p = incl - mine;
#pragma unroll
      for (int m = 0; m < kM; ++m) {
        uint32_t w = wd[m];
        while (w) {
          const uint32_t bpos = __ffs(w) - 1;
          w &= w - 1;
          // offset in the tile of element bpos % 4 of quad (lane + 32 m) + 256 (bpos / 4)
          s_keys[warp][p++] = (uint16_t)(4 * (lane + 32 * m + 256 * (bpos >> 2)) + (bpos & 3u));
        }
      }
      __syncwarp();
      const uint32_t key = lane < total ? s_keys[warp][lane] : 0xFFFFu;
      uint32_t rank = 0;
#pragma unroll
      for (int l2 = 0; l2 < 32; ++l2) rank += __shfl_sync(kFull, key, l2) < key ? 1u : 0u;
      __syncwarp();
      if (lane < total) {
        const int64_t p2 = pos + rank;
        const uint32_t i = a0 + key;
        if (p2 < a.capacity) {
          a.out_values[p2] = a.e[i];
          a.out_indices[p2] = (int32_t)i;
          a.e[i] = 0.0f;
        }
      }
      continue;
    }
    uint32_t any = 0;
#pragma unroll
    for (int m = 0; m < kM; ++m) any |= wd[m];
    any = __reduce_or_sync(kFull, any);
#pragma unroll 1
    for (int u = 0; u < 8; ++u) {
      if (((any >> (4 * u)) & 0xFu) == 0) continue;  // warp-uniform
#pragma unroll
      for (int m = 0; m < kM; ++m) {
        const uint32_t nib = (wd[m] >> (4 * u)) & 0xFu;
        if (!__any_sync(kFull, nib != 0)) continue;
        const uint32_t n4 = __popc(nib);
        const uint32_t incl = warp_incl_scan(n4);
        int64_t p = pos + (incl - n4);
        const uint32_t i = 4 * (q0 + lane + 32u * m + 256u * u);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if ((nib >> j) & 1u) {
            if (p < a.capacity) {
              a.out_values[p] = a.e[i + j];
              a.out_indices[p] = (int32_t)(i + j);
              a.e[i + j] = 0.0f;
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
  int64_t max_tiles = 0;
  size_t off_acc = 0, off_coef = 0, off_mode = 0, off_ssum = 0, off_ctl = 0, off_kw = 0,
         off_cnt = 0, off_csum = 0, off_off = 0, bytes = 0;
};

ef_status rk_plan(int64_t n, int32_t nseg, const int64_t* offs, const int64_t* ks, RPlan* p) {
  if (n < 0 || n > (int64_t(1) << 31)) return EF_ERR_SIZE;
  if (nseg < 1) return EF_ERR_SEGMENTS;
  if (!offs || !ks) return EF_ERR_NULL;
  if (offs[0] != 0 || offs[nseg] != n) return EF_ERR_SEGMENTS;
  RBatch cur{};
  auto flush = [&]() {
    if (cur.nseg == 0) return;
    p->max_tiles = std::max(p->max_tiles, cur.tiles[cur.nseg]);
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
    const int64_t blocks = (b - 1) / kRTile - a / kRTile + 1;  // aligned blocks it meets
    const int32_t nsamp =
        (k > 0 && len >= kSampleMinLen)
            ? (int32_t)std::min<int64_t>(kSampleBlocksMax, len / (16 * kSampleBlock))
            : 0;
    cur.seg[t] = RSeg{a, len, k, cur.samp[t], nsamp, i};
    cur.tiles[t + 1] = cur.tiles[t] + blocks;
    cur.samp[t + 1] = cur.samp[t] + nsamp;
    if (++cur.nseg == kRBatch) flush();
  }
  flush();
  size_t off = sizeof(WsHeader);
  p->off_ctl = off;
  off = round_up(off + sizeof(RCtl), 256);
  p->off_acc = off;
  off = round_up(off + (size_t)kRBatch * kChunks * 8, 256);
  p->off_ssum = off;
  off = round_up(off + (size_t)kRBatch * 8, 256);
  p->off_coef = off;
  off = round_up(off + (size_t)kRBatch * 4, 256);
  p->off_mode = off;
  off = round_up(off + (size_t)kRBatch * 4, 256);
  const size_t tb = (size_t)std::max<int64_t>(p->max_tiles, 1);
  p->off_kw = off;
  off = round_up(off + tb * 4 * kRTileWords, 256);
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
  double* ssum = reinterpret_cast<double*>(ws + p.off_ssum);
  RSelectArgs a{reinterpret_cast<float*>(ws + p.off_coef),
                reinterpret_cast<int32_t*>(ws + p.off_mode),
                ssum,
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
    const int64_t tiles = b.tiles[b.nseg], sblocks = b.samp[b.nseg];
    const int64_t nchunks = std::max<int64_t>(1, (tiles + kOffChunk - 1) / kOffChunk);
    err = cudaMemsetAsync(acc, 0, (size_t)kRBatch * kChunks * 8, s);
    if (err == cudaSuccess) err = cudaMemsetAsync(ssum, 0, (size_t)kRBatch * 8, s);
    if (err == cudaSuccess) err = cudaMemsetAsync(a.csum, 0, (size_t)nchunks * 4, s);
    if (err != cudaSuccess) return cuda_fail(err);
    const int64_t warps = (tiles + kRT / 32 - 1) / (kRT / 32);
    if (sblocks > 0) {
      const int gs = (int)std::min<int64_t>((sblocks + kRT / 32 - 1) / (kRT / 32),
                                            (int64_t)dev.sms * 8);
      launch_pdl(rk_sample, gs, kRT, 0, s, b, g_raw, e, ssum);
      if ((st = check_launch()) != EF_OK) return st;
    }
    const int ga = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, (int64_t)dev.sms * 3));
    if (vec) launch_pdl(rk_sum<true>, ga, kRT, 0, s, b, g_raw, e, acc, a);
    else launch_pdl(rk_sum<false>, ga, kRT, 0, s, b, g_raw, e, acc, a);
    if ((st = check_launch()) != EF_OK) return st;
    launch_pdl(rk_finalize, 1, kRBatch, 0, s, b, acc, a);
    if ((st = check_launch()) != EF_OK) return st;
    // rk_refine: 4 CTAs per SM (58 registers), one wave; rk_pack: 8
    const int gr = (int)std::max<int64_t>(1, std::min<int64_t>(warps, (int64_t)dev.sms * 4));
    const int gw = (int)std::max<int64_t>(1, std::min<int64_t>(warps, (int64_t)dev.sms * 8));
    if (vec_e) launch_pdl(rk_refine<true>, gr, kRT, 0, s, b, a);
    else launch_pdl(rk_refine<false>, gr, kRT, 0, s, b, a);
    if ((st = check_launch()) != EF_OK) return st;
    // always: it carries the running offset to the next launch
    launch_pdl(rk_offsets, (unsigned)nchunks, kRT, 0, s, tiles, a);
    if ((st = check_launch()) != EF_OK) return st;
    launch_pdl(rk_pack, gw, kRT, 0, s, b, a);
    if ((st = check_launch()) != EF_OK) return st;
  }
  return EF_OK;
}
