// Device steps of the index-range packet exchange ("梯度稀疏化：只传输重要的
// 梯度元素", §详细算法流程 step 5 and §与Allreduce的融合): the packets are
// ascending, so the entries a rank sends to the owner of index range
// [b_q, b_{q+1}) form one slice, found by a search per bound; the receiver
// rebases the slices it gets to its own range before the receive side runs
// on that range alone.
#include <cuda_runtime.h>

#include "ef_common.cuh"

namespace ef {
namespace {

constexpr int kSplitThreads = 1024;
constexpr int kMaxParts = 1024;

struct Bounds {
  int64_t b[kMaxParts + 1];
};

// Block q: starts[q] = #{ j < k : indices[j] < bounds[q] }, i.e. the first
// position whose index is >= bounds[q] in an ascending packet.  Two rounds of
// loads: thread t reads the sample at s_t = floor(t * k / 1024); the c
// samples below the bound put the answer in (s_{c-1}, s_c], whose entries
// (at most ceil(k / 1024)) are then counted by the whole CTA.  Every access
// is in [0, k) whatever the packet holds; an unsorted packet gives some
// position in [0, k], and the receive side reports it as malformed.
__global__ void __launch_bounds__(kSplitThreads)
packet_split_kernel(const int32_t* __restrict__ indices, int64_t k, Bounds bd,
                    int64_t* __restrict__ starts) {
  pdl_wait();
  __shared__ uint32_t scratch[64];
  const int64_t bound = bd.b[blockIdx.x];
  const int t = threadIdx.x;
  if (k == 0) {
    if (t == 0) starts[blockIdx.x] = 0;
    return;
  }
  const int64_t m = kSplitThreads;
  const int64_t s_t = (int64_t)t * k / m;
  // the samples repeat positions when k < 1024; counting them is harmless
  // because only the count of samples below the bound is used
  const bool below = (int64_t)indices[s_t] < bound;
  uint32_t total;
  (void)block_excl_scan(below ? 1u : 0u, scratch, &total);
  const int64_t c = total;
  int64_t lo, hi;  // the answer is lo + #{ j in [lo, hi) : indices[j] < bound }
  if (c == 0) {
    lo = 0;
    hi = 0;
  } else {
    lo = (c - 1) * k / m + 1;
    hi = c < m ? c * k / m : k;
  }
  uint32_t cnt = 0;
  for (int64_t j = lo + t; j < hi; j += kSplitThreads) cnt += (int64_t)indices[j] < bound;
  uint32_t sum;
  (void)block_excl_scan(cnt, scratch, &sum);
  if (t == 0) starts[blockIdx.x] = lo + sum;
}

__global__ void __launch_bounds__(256)
index_rebase_kernel(int32_t* __restrict__ indices, int64_t count, int64_t base) {
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < count; j += stride)
    indices[j] = (int32_t)((int64_t)indices[j] - base);
}

}  // namespace
}  // namespace ef

extern "C" ef_status ef_packet_split(const int32_t* indices, int64_t k, int32_t nparts,
                                     const int64_t* h_bounds, int64_t* d_starts, void* stream) {
  using namespace ef;
  if (k < 0 || k > (int64_t(1) << 31)) return EF_ERR_SIZE;
  if (nparts < 1 || nparts > kMaxParts) return EF_ERR_ARG;
  if (!h_bounds || !d_starts || (k > 0 && !indices)) return EF_ERR_NULL;
  if ((indices && !aligned4(indices)) || (reinterpret_cast<uintptr_t>(d_starts) & 7u) != 0)
    return EF_ERR_ALIGN;
  Bounds bd;
  for (int q = 0; q <= nparts; ++q) {
    bd.b[q] = h_bounds[q];
    if (q > 0 && bd.b[q] < bd.b[q - 1]) return EF_ERR_SEGMENTS;
  }
  if (overlaps(indices, (size_t)k * 4, d_starts, (size_t)(nparts + 1) * 8)) return EF_ERR_ALIAS;
  DeviceInfo dev;
  ef_status st = current_device(&dev);
  if (st != EF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  launch_pdl(packet_split_kernel, nparts + 1, kSplitThreads, 0, s, indices, k, bd, d_starts);
  return check_launch();
}

extern "C" ef_status ef_index_rebase(int32_t* indices, int64_t count, int64_t base,
                                     void* stream) {
  using namespace ef;
  if (count < 0 || count > (int64_t(1) << 31)) return EF_ERR_SIZE;
  if (base < 0 || base > (int64_t(1) << 31)) return EF_ERR_ARG;
  if (count > 0 && !indices) return EF_ERR_NULL;
  if (indices && !aligned4(indices)) return EF_ERR_ALIGN;
  if (count == 0) return EF_OK;
  DeviceInfo dev;
  ef_status st = current_device(&dev);
  if (st != EF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t blocks = (count + 255) / 256;
  const int grid = (int)(blocks < (int64_t)dev.sms * 8 ? blocks : (int64_t)dev.sms * 8);
  launch_pdl(index_rebase_kernel, grid, 256, 0, s, indices, count, base);
  return check_launch();
}
