// Shared internals of libefgrad: device helpers (scans, bounded decoupled
// look-back, block radix select) and host helpers (status, profiling hook,
// device properties).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "efgrad.h"

namespace ef {

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

struct DeviceInfo {
  int sms = 0;
  int major = 0, minor = 0;
  size_t max_smem_optin = 0;
};

// Properties of the current device (cached per device).  Returns EF_OK,
// EF_ERR_ARCH (not compute capability 10.3) or EF_ERR_CUDA.
ef_status current_device(DeviceInfo* out);

// Record the failing CUDA error for ef_last_cuda_error() and map to a status.
ef_status cuda_fail(cudaError_t err);

// Count one kernel launch and check it; returns EF_OK or EF_ERR_CUDA.
ef_status check_launch();

// Launches `kernel` on `s` with programmatic stream serialization: it may be
// scheduled while the kernel before it in the stream is still running, and
// every kernel of the library calls pdl_wait() before it touches memory, so
// the order of effects is the stream order.  Errors surface through
// check_launch().
template <typename... P, typename... A>
inline void launch_pdl(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       A&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  (void)cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// launch_pdl for a kernel whose CTAs form thread-block clusters of
// `cluster` CTAs along x (the grid a multiple of it).
template <typename... P, typename... A>
inline void launch_cluster_pdl(void (*kernel)(P...), int cluster, dim3 grid, dim3 block,
                               size_t smem, cudaStream_t s, A&&... args) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  (void)cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// Profiling hook: record the thread's start/stop event for `kernel_id`
// around a launch, if set.
void prof_begin(int kernel_id, cudaStream_t s);
void prof_end(int kernel_id, cudaStream_t s);

inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool overlaps(const void* a, size_t abytes, const void* b, size_t bbytes) {
  if (!a || !b || abytes == 0 || bbytes == 0) return false;
  uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bbytes && y < x + abytes;
}
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Every workspace starts with this header; `status` is what
// ef_workspace_status() reports.
struct alignas(256) WsHeader {
  int32_t status;
  uint32_t reserved[63];
};

// ---------------------------------------------------------------------------
// device side
// ---------------------------------------------------------------------------

constexpr unsigned kFull = 0xffffffffu;

// Programmatic dependent launch.  pdl_wait() returns once every kernel this
// one depends on in the stream has completed and its writes are visible (at
// once for a kernel launched without the attribute); every kernel calls it
// before its first memory access.  pdl_trigger() lets the next kernel in the
// stream be scheduled early, to wait in its own pdl_wait().  Short kernels
// whose successor is short call it first thing; the long streaming passes,
// the kernels before them and the last kernel of a call leave it to their
// exit, so that no waiting CTA holds SM resources a streaming pass on
// another stream could use.  (Triggering early in a layerwise top-k call,
// from its sampling launch or its streaming pass, measured slower: 110
// against 101 us for the ResNet-50 call.)
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t abs_key(float x) {
  return __float_as_uint(x) & 0x7FFFFFFFu;
}

__device__ __forceinline__ unsigned lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
  atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint64_t ld_acquire(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint64_t ld_relaxed(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ int32_t ld_volatile(const int32_t* p) {
  return *reinterpret_cast<const volatile int32_t*>(p);
}

// Warp inclusive scan of a uint32.
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
  const unsigned lane = lane_id();
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t t = __shfl_up_sync(kFull, v, o);
    if (lane >= (unsigned)o) v += t;
  }
  return v;
}

// Shared-memory histogram update: every lane with `valid` set counts one
// key in hist[bin].  All 32 lanes call it together (the callers keep their
// trip counts warp-uniform).  It is a plain shared-memory atomicAdd per key:
// a warp-aggregated form (one atomicAdd of the lane count per distinct bin,
// the lanes grouped with __match_any_sync) measured slower on GB300 in every
// case tried, ties included -- the ResNet-50 layerwise call 0.156 against
// 0.126 ms, an all-equal 2^29-element tensor 8.21 against 7.26 ms, the 2^20
// top-k call 79.8 against 57.5 us -- and so did aggregating only when the
// whole warp shares one bin (0.133 ms, 8.55 ms, 62.7 us).
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin, bool valid) {
  if (valid) atomicAdd(&hist[bin], 1u);
}

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Block exclusive scan of a uint32 (blockDim.x a multiple of 32, <= 1024).
// `scratch` holds >= 33 words of shared memory.  Returns the exclusive prefix;
// *total receives the block sum.  Contains __syncthreads().
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* scratch,
                                                    uint32_t* total) {
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  const unsigned nwarps = blockDim.x >> 5;
  uint32_t incl = warp_incl_scan(v);
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < nwarps ? scratch[lane] : 0u;
    uint32_t wi = warp_incl_scan(w);
    if (lane < nwarps) scratch[lane] = wi - w;
    if (lane == 31) scratch[32] = wi;
  }
  __syncthreads();
  uint32_t res = scratch[warp] + incl - v;
  *total = scratch[32];
  __syncthreads();
  return res;
}

// ---------------------------------------------------------------------------
// Decoupled look-back (single-pass prefix over ordered tiles).
//
// A tile's state word holds a 2-bit flag in bits 63..62 and a 62-bit payload
// that adds without carries between its fields.  Tile ids are handed out in
// order by an atomic ticket, so every predecessor of a running tile is itself
// running or finished and the wait always ends; it is still bounded by a
// wall-clock limit, after which the status word gets EF_ERR_DEVICE_TIMEOUT
// and the tile proceeds with what it has (no hang, outputs unspecified).
// ---------------------------------------------------------------------------

constexpr uint64_t kFlagAgg = 1ull << 62;
constexpr uint64_t kFlagIncl = 2ull << 62;
constexpr uint64_t kPayloadMask = (1ull << 62) - 1;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Called by all 32 lanes of ONE warp.  `states` indexes tiles globally;
// the chain of this tile starts at `first` (exclusive prefix 0 there).
// Publishes this tile's aggregate, looks back, publishes the inclusive prefix
// and returns the exclusive prefix (same value in every lane).
__device__ __forceinline__ uint64_t lookback_warp(uint64_t* states, int64_t tile,
                                                  int64_t first, uint64_t agg,
                                                  int32_t* status,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  const unsigned lane = lane_id();
  if (tile == first) {
    if (lane == 0) st_release(&states[tile], kFlagIncl | agg);
    return 0;
  }
  if (lane == 0) st_release(&states[tile], kFlagAgg | agg);
  uint64_t excl = 0;
  int64_t base = tile - 1;
  const uint64_t t0 = global_ns();
  bool gave_up = false;
  while (base >= first) {
    const int64_t t = base - (int64_t)lane;
    uint64_t s = (t >= first) ? ld_acquire(&states[t]) : kFlagIncl;
    uint32_t spins = 0;
    while (__any_sync(kFull, (s >> 62) == 0)) {
      if ((s >> 62) == 0) s = ld_acquire(&states[t]);
      if ((++spins & 63u) == 0) {
        int bad = 0;
        if (lane == 0)
          bad = (global_ns() - t0 > limit_ns) || (ld_volatile(status) != 0) ||
                spins > (1u << 26);
        bad = __shfl_sync(kFull, bad, 0);
        if (bad) {
          if (lane == 0) set_status(status, EF_ERR_DEVICE_TIMEOUT);
          gave_up = true;
          break;
        }
      }
      __nanosleep(32);
    }
    if (gave_up) break;
    const unsigned incl = __ballot_sync(kFull, (s >> 62) == 2);
    if (incl) {
      const int stop = __ffs(incl) - 1;
      uint64_t v = (lane <= (unsigned)stop) ? (s & kPayloadMask) : 0;
      excl += warp_sum_u64(v);
      break;
    }
    excl += warp_sum_u64(s & kPayloadMask);
    base -= 32;
  }
  if (lane == 0) st_release(&states[tile], kFlagIncl | ((excl + agg) & kPayloadMask));
  return excl;
}

// lookback_warp for a short pass whose tiles all finish at about the same
// time (a few hundred tiles, one or a few per CTA): the chains of
// aggregates are then long, and each round of the look-back is a round trip
// to L2.  Lane l reads predecessors base - l * P - j (j < P) in each round,
// so one round trip covers 32 P of them.  The states are read with relaxed
// loads and published with atomic exchanges, which are performed at L2 at
// once: a state word carries its flag and its payload together, and the
// readers use nothing else the tile wrote before the kernel ends.  (Acquire
// loads would be performed one after another; a release store first waits,
// through the block barrier before it, for the CTA's streaming stores to
// reach memory; a relaxed store measured microseconds late to other SMs --
// the 2^20-element call's look-backs ended 4.9 us after their last
// predecessor's aggregate with it, 1.9 us with the exchange.)
template <int P>
__device__ __forceinline__ uint64_t lookback_warp_short(uint64_t* states, int64_t tile,
                                                        int64_t first, uint64_t agg,
                                                        int32_t* status,
                                                        uint64_t limit_ns = kWaitLimitNs) {
  const unsigned lane = lane_id();
  if (tile == first) {
    if (lane == 0)
      atomicExch(reinterpret_cast<unsigned long long*>(&states[tile]), kFlagIncl | agg);
    return 0;
  }
  if (lane == 0)
    atomicExch(reinterpret_cast<unsigned long long*>(&states[tile]), kFlagAgg | agg);
  uint64_t excl = 0;
  int64_t base = tile - 1;
  const uint64_t t0 = global_ns();
  bool gave_up = false;
  while (base >= first) {
    const int64_t t = base - (int64_t)lane * P;
    uint64_t s[P];
#pragma unroll
    for (int j = 0; j < P; ++j) s[j] = (t - j >= first) ? ld_relaxed(&states[t - j]) : kFlagIncl;
    uint32_t spins = 0;
    for (;;) {
      bool pending = false;
#pragma unroll
      for (int j = 0; j < P; ++j) pending |= (s[j] >> 62) == 0;
      if (!__any_sync(kFull, pending)) break;
#pragma unroll
      for (int j = 0; j < P; ++j)
        if ((s[j] >> 62) == 0) s[j] = ld_relaxed(&states[t - j]);
      if ((++spins & 63u) == 0) {
        int bad = 0;
        if (lane == 0)
          bad = (global_ns() - t0 > limit_ns) || (ld_volatile(status) != 0) ||
                spins > (1u << 26);
        bad = __shfl_sync(kFull, bad, 0);
        if (bad) {
          if (lane == 0) set_status(status, EF_ERR_DEVICE_TIMEOUT);
          gave_up = true;
          break;
        }
      }
      __nanosleep(32);
    }
    if (gave_up) break;
    // the nearest inclusive predecessor: the lowest (lane, j) holding one
    int jinc = P;
#pragma unroll
    for (int j = P - 1; j >= 0; --j)
      if ((s[j] >> 62) == 2) jinc = j;
    const unsigned incl = __ballot_sync(kFull, jinc < P);
    const int stop = incl ? __ffs(incl) - 1 : 32;
    uint64_t v = 0;
#pragma unroll
    for (int j = 0; j < P; ++j)
      if ((int)lane < stop || ((int)lane == stop && j <= jinc)) v += s[j] & kPayloadMask;
    excl += warp_sum_u64(v);
    if (incl) break;
    base -= 32 * P;
  }
  if (lane == 0)
    atomicExch(reinterpret_cast<unsigned long long*>(&states[tile]),
               kFlagIncl | ((excl + agg) & kPayloadMask));
  return excl;
}

// ---------------------------------------------------------------------------
// Block radix select over keys in shared memory.
//
// Finds the k-th largest (1 <= k <= n) key T of keys[0..n), each key taken as
// its low 31 bits (so float bit patterns give |x| keys): after the call,
// gt = #keys > T and need = k - gt (>= 1 keys equal to T are taken, lowest
// positions first).  Digits: bits 30..20 (2048 bins), 19..10, 9..0.
// `hist` holds 2048 words of shared memory, `scratch` >= 41 words.
// All threads of the block must call it.
// ---------------------------------------------------------------------------

struct SelectResult {
  uint32_t T;
  uint32_t gt;
  uint32_t need;
};

// Given a histogram of `nbins` bins in shared memory and a rank `krem`
// (1-based, counted from the top bin), find the bin b holding that rank and
// the count of entries in bins above it.  All threads call it; results are
// returned to every thread.  Thread t owns `per` consecutive positions
// counted from the top bin; its lane reads them starting at a rotated
// offset, so that with 32 positions per thread a warp's 32 reads fall in 32
// distinct banks (in order they would all hit one).  Every warp scans the
// warp totals itself, and the owner of rank krem is resolved by its whole
// warp, one position per lane: three barriers in all.  `scratch` holds
// >= 38 words.
__device__ __forceinline__ void block_find_bin(const uint32_t* hist, int nbins, uint32_t krem,
                                               uint32_t* scratch, uint32_t* bin_out,
                                               uint32_t* above_out) {
  const int per = (nbins + blockDim.x - 1) / blockDim.x;
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int q0 = (int)threadIdx.x * per;
  const int r0 = (int)lane % per;
  uint32_t local = 0;
  for (int j = 0; j < per; ++j) {
    int r = r0 + j;
    if (r >= per) r -= per;
    if (q0 + r < nbins) local += hist[nbins - 1 - (q0 + r)];
  }
  const uint32_t inc = warp_incl_scan(local);
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  const uint32_t wt = (int)lane < nwarps ? scratch[lane] : 0u;
  const uint32_t wi = warp_incl_scan(wt);
  const uint32_t excl = __shfl_sync(kFull, wi - wt, (int)warp) + inc - local;
  const bool own = excl < krem && krem <= excl + local;  // one thread at most
  if (per <= 32) {
    const unsigned m = __ballot_sync(kFull, own);
    if (m != 0u) {  // warp-uniform
      const int o = __ffs(m) - 1;
      const int q = __shfl_sync(kFull, q0, o) + (int)lane;
      const uint32_t eo = __shfl_sync(kFull, excl, o);
      const bool in = (int)lane < per && q < nbins;
      const uint32_t c = in ? hist[nbins - 1 - q] : 0u;
      const uint32_t ci = warp_incl_scan(c);
      const unsigned hit = __ballot_sync(kFull, in && eo + ci >= krem);
      if ((int)lane == __ffs(hit) - 1) {
        scratch[36] = (uint32_t)(nbins - 1 - q);
        scratch[37] = eo + ci - c;
      }
    }
  } else if (own) {
    uint32_t cum = excl;
    for (int q = q0; q < q0 + per && q < nbins; ++q) {
      const uint32_t c = hist[nbins - 1 - q];
      if (cum + c >= krem) {
        scratch[36] = (uint32_t)(nbins - 1 - q);
        scratch[37] = cum;
        break;
      }
      cum += c;
    }
  }
  __syncthreads();
  *bin_out = scratch[36];
  *above_out = scratch[37];
  __syncthreads();
}

// The same over keys produced by `key_at(i)` (i < n < 2^31), e.g. read from
// global memory; eight keys per thread are loaded before any is counted, so
// a global source keeps eight loads in flight per thread.  With `sub` (room
// for `sub_cap` keys of shared memory) the second digit pass also copies the
// keys it counts -- those sharing the first digit with the k-th key -- into
// `sub`, and if they fit, the third pass reads only them.
template <typename KeyAt>
__device__ __forceinline__ SelectResult block_radix_select_at(int n, uint32_t k, uint32_t* hist,
                                                              uint32_t* scratch, KeyAt key_at,
                                                              uint32_t* sub = nullptr,
                                                              int sub_cap = 0) {
  uint32_t prefix = 0, krem = k, gt = 0;
  uint32_t* sub_count = scratch + 40;
  int m = -1;  // keys in sub for the last pass (-1: read all n keys)
  for (int p = 0; p < 3; ++p) {
    // digits: bits 30..20, 19..10, 9..0
    const int shift = 20 - 10 * p, width = p == 0 ? 11 : 10;
    const int nb = 1 << width;
    const int hi = shift + width;  // bits above this digit are fixed
    const bool collect = sub != nullptr && p == 1;
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
    uint32_t bin, above;
    block_find_bin(hist, nb, krem, scratch, &bin, &above);
    prefix |= bin << shift;
    gt += above;
    krem -= above;
  }
  return SelectResult{prefix, gt, krem};
}

__device__ __forceinline__ SelectResult block_radix_select(const uint32_t* keys, int n, uint32_t k,
                                                           uint32_t* hist, uint32_t* scratch,
                                                           uint32_t* sub = nullptr,
                                                           int sub_cap = 0) {
  return block_radix_select_at(n, k, hist, scratch, [keys](int i) { return keys[i]; }, sub,
                               sub_cap);
}

}  // namespace ef
