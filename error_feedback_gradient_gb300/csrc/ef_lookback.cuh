// Block-wide bounded decoupled look-back, shared by the kernels whose tiles
// are resolved by a whole CTA (top-k emit, the random-sparsification packet).
#pragma once

#include <climits>

#include "ef_common.cuh"

namespace ef {

// Shared scratch of lookback_block.
struct LookbackShared {
  int first_incl[32];  // per warp: lowest thread index seeing an inclusive state
  uint64_t part[32];   // per warp: partial sums
};

// Block-wide form of the bounded decoupled look-back (same flags, payloads,
// wait limits and error report as lookback_warp): in each round thread i
// reads the state of predecessor base - i, so one round trip covers
// blockDim.x predecessors instead of 32.  Called by every thread of the CTA;
// every thread gets the exclusive prefix.  blockDim.x is a multiple of 32.
__device__ __forceinline__ uint64_t lookback_block(uint64_t* states, int64_t tile, int64_t first, uint64_t agg,
                                   int32_t* status, LookbackShared& sh) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const unsigned lane = lane_id();
  const int wid = tid >> 5, nwarps = nthr >> 5;
  if (tile == first) {
    if (tid == 0) st_release(&states[tile], kFlagIncl | agg);
    return 0;
  }
  if (tid == 0) st_release(&states[tile], kFlagAgg | agg);
  uint64_t excl = 0;
  int64_t base = tile - 1;
  const uint64_t t0 = global_ns();
  while (base >= first) {
    const int64_t t = base - tid;
    uint64_t s = (t >= first) ? ld_acquire(&states[t]) : kFlagIncl;
    uint32_t spins = 0;
    bool gave_up = false;
    while (__syncthreads_or((s >> 62) == 0)) {
      if ((s >> 62) == 0) s = ld_acquire(&states[t]);
      if ((++spins & 63u) == 0) {  // spins is uniform across the CTA
        int bad = 0;
        if (tid == 0)
          bad = (global_ns() - t0 > kWaitLimitNs) || (ld_volatile(status) != 0) ||
                spins > (1u << 26);
        if (__syncthreads_or(bad)) {
          if (tid == 0) set_status(status, EF_ERR_DEVICE_TIMEOUT);
          gave_up = true;
          break;
        }
      }
      __nanosleep(32);
    }
    if (gave_up) break;
    // the nearest inclusive predecessor of this round: the lowest thread
    // index whose state is inclusive (predecessors before `first` count as
    // inclusive zeros)
    const unsigned incl = __ballot_sync(kFull, (s >> 62) == 2);
    if (lane == 0) sh.first_incl[wid] = incl ? wid * 32 + __ffs(incl) - 1 : INT_MAX;
    __syncthreads();
    int stop = INT_MAX;
    for (int w = 0; w < nwarps; ++w) stop = min(stop, sh.first_incl[w]);
    const uint64_t ws = warp_sum_u64(tid <= stop ? (s & kPayloadMask) : 0ull);
    if (lane == 0) sh.part[wid] = ws;
    __syncthreads();
    for (int w = 0; w < nwarps; ++w) excl += sh.part[w];
    __syncthreads();  // the scratch is reused by the next round
    if (stop != INT_MAX) break;
    base -= nthr;
  }
  if (tid == 0) st_release(&states[tile], kFlagIncl | ((excl + agg) & kPayloadMask));
  return excl;
}

}  // namespace ef
