// 1-bit error feedback: sender (sign quantisation with an EMA error buffer)
// and receiver (sum of decoded signs, then SGD or the 1-bit momentum).
//
// Sender, "1bit Adam梯度压缩技术原理与分布式训练优化" §2.1:
//   v = g + eps;  bit = !(v < 0);  s = bit ? +1 : -1;  d = v - s;
//   eps' = beta1 * eps + (1 - beta1) * d
// Receiver: G = sum_w s_w ("梯度稀疏化" §详细算法流程 step 6 applied to sign
// packets), then w -= eta * G (step 7) or m = beta1 * m + (1 - beta1) * G
// (1-bit Adam §2.2).
//
// Both passes are HBM-bound streams (sender: 12 B + 1/8 B per element;
// receiver with SGD: 8 B + 4 B for G + W/8 B).  They use 16-byte loads and
// stores, a persistent grid of whole SM multiples, and keep four groups of
// loads in flight per warp.  Every float operation is an explicit
// round-to-nearest intrinsic, so no multiply-add is contracted.
#include <cuda_runtime.h>

#include <cmath>

#include "ef_common.cuh"

namespace ef {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;       // 128-element groups in flight per warp (sender)
constexpr int kSpan = 32;        // 128-element groups in a warp's span on large inputs
static_assert(kSpan % kUnroll == 0, "span layout");
constexpr int kApplyUnroll = 2;  // float4 chunks in flight per thread (receiver)

__device__ __forceinline__ float sign_step(float g, float e, float b1, float c, bool* bit) {
  const float v = __fadd_rn(g, e);
  const bool b = !(v < 0.0f);
  const float s = b ? 1.0f : -1.0f;
  const float d = __fsub_rn(v, s);
  *bit = b;
  return __fadd_rn(__fmul_rn(b1, e), __fmul_rn(c, d));
}

// Groups of 128 elements [0, ngroups): lane l of a warp owns elements
// 4l..4l+3 of a group, so a group's four bit words are built from 8-lane
// nibble sets.  g and eps must be 16-byte aligned.
template <int kSpanT>
__global__ void __launch_bounds__(kThreads)
sign_compress_vec(const float* __restrict__ g, float* __restrict__ eps,
                  uint32_t* __restrict__ bits, int64_t ngroups, float b1, float c,
                  bool bits16) {
  pdl_wait();
  const unsigned lane = lane_id();
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  // Each warp streams a contiguous span of kSpanT groups (a multiple of
  // kUnroll; 16 KB of g and of eps on large inputs), kUnroll groups at a
  // time; spans are dealt to warps round-robin.  The span length is a
  // compile-time constant so that the compiler can unroll it and issue the
  // next groups' loads early.
  for (int64_t s0 = warp * kSpanT; s0 < ngroups; s0 += nwarps * kSpanT)
#pragma unroll
  for (int64_t g0 = s0; g0 < s0 + kSpanT; g0 += kUnroll) {
    if (g0 >= ngroups) break;  // warp-uniform
    float4 gv[kUnroll], ev[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (g0 + u < ngroups) {
        const int64_t i = (g0 + u) * 128 + lane * 4;
        gv[u] = __ldcs(reinterpret_cast<const float4*>(g + i));
        ev[u] = __ldcs(reinterpret_cast<const float4*>(eps + i));
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t grp = g0 + u;
      if (grp >= ngroups) break;  // warp-uniform
      bool b0, b1_, b2, b3;
      float4 o;
      o.x = sign_step(gv[u].x, ev[u].x, b1, c, &b0);
      o.y = sign_step(gv[u].y, ev[u].y, b1, c, &b1_);
      o.z = sign_step(gv[u].z, ev[u].z, b1, c, &b2);
      o.w = sign_step(gv[u].w, ev[u].w, b1, c, &b3);
      __stcs(reinterpret_cast<float4*>(eps + grp * 128 + lane * 4), o);
      uint32_t v = ((uint32_t)b0 | ((uint32_t)b1_ << 1) | ((uint32_t)b2 << 2) |
                    ((uint32_t)b3 << 3))
                   << (4 * (lane & 7));
      v |= __shfl_xor_sync(kFull, v, 1);
      v |= __shfl_xor_sync(kFull, v, 2);
      v |= __shfl_xor_sync(kFull, v, 4);
      if (bits16) {
        const uint32_t w1 = __shfl_sync(kFull, v, 8);
        const uint32_t w2 = __shfl_sync(kFull, v, 16);
        const uint32_t w3 = __shfl_sync(kFull, v, 24);
        if (lane == 0)
          *reinterpret_cast<uint4*>(bits + grp * 4) = make_uint4(v, w1, w2, w3);
      } else if ((lane & 7) == 0) {
        bits[grp * 4 + (lane >> 3)] = v;
      }
    }
  }
}

// One 32-element word per warp step: lane l owns element 32w + l.  Used for
// the tail after the vector groups and for buffers that are not 16-byte
// aligned.  Padding bits beyond n are 0.
__global__ void __launch_bounds__(kThreads)
sign_compress_words(const float* __restrict__ g, float* __restrict__ eps,
                    uint32_t* __restrict__ bits, int64_t n, int64_t w_begin,
                    int64_t w_end, float b1, float c) {
  pdl_wait();
  const unsigned lane = lane_id();
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t w0 = w_begin + warp * kUnroll; w0 < w_end; w0 += nwarps * kUnroll) {
    float gv[kUnroll], ev[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = (w0 + u) * 32 + lane;
      const bool in = (w0 + u < w_end) && i < n;
      gv[u] = in ? __ldcs(g + i) : 0.0f;
      ev[u] = in ? __ldcs(eps + i) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (w0 + u >= w_end) break;  // warp-uniform
      const int64_t i = (w0 + u) * 32 + lane;
      const bool in = i < n;
      bool b = false;
      const float o = sign_step(gv[u], ev[u], b1, c, &b);
      if (in) __stcs(eps + i, o);
      const uint32_t word = __ballot_sync(kFull, in && b);
      if (lane == 0) bits[w0 + u] = word;
    }
  }
}

struct SignApplyArgs {
  const uint32_t* bits[EF_MAX_WORKERS];
  int32_t W;
  int32_t mode;
  float eta, b1, c;
};

__device__ __forceinline__ float apply_one(float x, float G, const SignApplyArgs& a) {
  if (a.mode == EF_APPLY_SGD) return __fsub_rn(x, __fmul_rn(a.eta, G));
  return __fadd_rn(__fmul_rn(a.b1, x), __fmul_rn(a.c, G));
}

// Float4 chunks [0, nchunks): G = 2 * (#set bits) - W (the exact sum of W
// terms +-1), then the update.  w and G must be 16-byte aligned.
__global__ void __launch_bounds__(kThreads, 8)
sign_apply_vec(SignApplyArgs a, float* __restrict__ G, float* __restrict__ x,
               int64_t nchunks) {
  pdl_wait();
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  for (int64_t q0 = tid; q0 < nchunks; q0 += nthr * kApplyUnroll) {
    float4 xv[kApplyUnroll];
#pragma unroll
    for (int u = 0; u < kApplyUnroll; ++u) {
      const int64_t q = q0 + (int64_t)u * nthr;
      if (q < nchunks) xv[u] = __ldcs(reinterpret_cast<const float4*>(x) + q);
    }
#pragma unroll
    for (int u = 0; u < kApplyUnroll; ++u) {
      const int64_t q = q0 + (int64_t)u * nthr;
      if (q >= nchunks) break;
      const int64_t i = q * 4;
      const int sh = (int)(i & 31);
      int c0 = 0, c1 = 0, c2 = 0, c3 = 0;
      for (int w = 0; w < a.W; ++w) {
        const uint32_t nib = (__ldg(a.bits[w] + (i >> 5)) >> sh) & 0xFu;
        c0 += nib & 1u;
        c1 += (nib >> 1) & 1u;
        c2 += (nib >> 2) & 1u;
        c3 += (nib >> 3) & 1u;
      }
      float4 gs = make_float4((float)(2 * c0 - a.W), (float)(2 * c1 - a.W),
                              (float)(2 * c2 - a.W), (float)(2 * c3 - a.W));
      if (G) __stcs(reinterpret_cast<float4*>(G) + q, gs);
      float4 o;
      o.x = apply_one(xv[u].x, gs.x, a);
      o.y = apply_one(xv[u].y, gs.y, a);
      o.z = apply_one(xv[u].z, gs.z, a);
      o.w = apply_one(xv[u].w, gs.w, a);
      __stcs(reinterpret_cast<float4*>(x) + q, o);
    }
  }
}

// Elements [begin, n) one per thread (tail, or unaligned buffers).
__global__ void __launch_bounds__(kThreads)
sign_apply_scalar(SignApplyArgs a, float* __restrict__ G, float* __restrict__ x,
                  int64_t begin, int64_t n) {
  pdl_wait();
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = begin + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += nthr) {
    int cnt = 0;
    for (int w = 0; w < a.W; ++w) cnt += (__ldg(a.bits[w] + (i >> 5)) >> (i & 31)) & 1u;
    const float gs = (float)(2 * cnt - a.W);
    if (G) G[i] = gs;
    x[i] = apply_one(x[i], gs, a);
  }
}

int grid_for(int64_t work_items, int per_block, int sms, int blocks_per_sm) {
  int64_t need = (work_items + per_block - 1) / per_block;
  int64_t cap = (int64_t)sms * blocks_per_sm;
  if (need < 1) need = 1;
  return (int)(need < cap ? need : cap);
}

}  // namespace
}  // namespace ef

extern "C" ef_status ef_sign_compress(const float* g, float* eps, int64_t n, float beta1,
                                      uint32_t* out_bits, void* stream) {
  using namespace ef;
  if (n < 0) return EF_ERR_SIZE;
  if (!std::isfinite(beta1)) return EF_ERR_ARG;
  if (n == 0) return EF_OK;
  if (!g || !eps || !out_bits) return EF_ERR_NULL;
  if (!aligned4(g) || !aligned4(eps) || !aligned4(out_bits)) return EF_ERR_ALIGN;
  const int64_t nwords = (n + 31) / 32;
  const size_t fb = (size_t)n * 4, wb = (size_t)nwords * 4;
  if (overlaps(g, fb, eps, fb) || overlaps(out_bits, wb, g, fb) || overlaps(out_bits, wb, eps, fb))
    return EF_ERR_ALIAS;
  DeviceInfo dev;
  ef_status st = current_device(&dev);
  if (st != EF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float b1 = beta1;
  const float c = 1.0f - b1;  // one float32 subtraction, round to nearest
  const int warps_per_block = kThreads / 32;
  prof_begin(EF_KERNEL_SIGN, s);
  int64_t w_begin = 0;
  if (aligned16(g) && aligned16(eps)) {
    const int64_t ngroups = n / 128;
    if (ngroups > 0) {
      // long spans only once every resident warp gets at least two of them
      const int64_t resident_warps = (int64_t)dev.sms * 8 * warps_per_block;
      if (ngroups >= 2 * resident_warps * kSpan) {
        const int grid = grid_for(ngroups, warps_per_block * kSpan, dev.sms, 8);
        launch_pdl(sign_compress_vec<kSpan>, grid, kThreads, 0, s, g, eps, out_bits, ngroups, b1, c,
                                                           aligned16(out_bits));
      } else {
        const int grid = grid_for(ngroups, warps_per_block * kUnroll, dev.sms, 8);
        launch_pdl(sign_compress_vec<kUnroll>, grid, kThreads, 0, s, g, eps, out_bits, ngroups, b1, c,
                                                             aligned16(out_bits));
      }
      if ((st = check_launch()) != EF_OK) return st;
    }
    w_begin = ngroups * 4;
  }
  if (w_begin < nwords) {
    const int grid = grid_for(nwords - w_begin, warps_per_block * kUnroll, dev.sms, 8);
    launch_pdl(sign_compress_words, grid, kThreads, 0, s, g, eps, out_bits, n, w_begin, nwords, b1, c);
    if ((st = check_launch()) != EF_OK) return st;
  }
  prof_end(EF_KERNEL_SIGN, s);
  return EF_OK;
}

extern "C" ef_status sign_aggregate_apply(int32_t W, const uint32_t* const* h_bits, int64_t n,
                                          int32_t mode, float eta, float beta1, float* G,
                                          float* w_or_m, void* stream) {
  using namespace ef;
  if (W < 1 || W > EF_MAX_WORKERS) return EF_ERR_WORKERS;
  if (n < 0) return EF_ERR_SIZE;
  if (mode != EF_APPLY_SGD && mode != EF_APPLY_MOMENTUM) return EF_ERR_ARG;
  if (mode == EF_APPLY_SGD && !std::isfinite(eta)) return EF_ERR_ARG;
  if (mode == EF_APPLY_MOMENTUM && !std::isfinite(beta1)) return EF_ERR_ARG;
  if (!h_bits) return EF_ERR_NULL;
  if (n == 0) return EF_OK;
  if (!w_or_m) return EF_ERR_NULL;
  if (!aligned4(w_or_m) || (G && !aligned4(G))) return EF_ERR_ALIGN;
  const size_t fb = (size_t)n * 4, wb = (size_t)((n + 31) / 32) * 4;
  if (G && overlaps(G, fb, w_or_m, fb)) return EF_ERR_ALIAS;
  SignApplyArgs a;
  for (int w = 0; w < W; ++w) {
    if (!h_bits[w]) return EF_ERR_NULL;
    if (!aligned4(h_bits[w])) return EF_ERR_ALIGN;
    if (overlaps(h_bits[w], wb, w_or_m, fb) || (G && overlaps(h_bits[w], wb, G, fb)))
      return EF_ERR_ALIAS;
    a.bits[w] = h_bits[w];
  }
  for (int w = W; w < EF_MAX_WORKERS; ++w) a.bits[w] = nullptr;
  a.W = W;
  a.mode = mode;
  a.eta = eta;
  a.b1 = beta1;
  a.c = 1.0f - beta1;
  DeviceInfo dev;
  ef_status st = current_device(&dev);
  if (st != EF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  prof_begin(EF_KERNEL_SIGN_APPLY, s);
  int64_t begin = 0;
  if (aligned16(w_or_m) && (!G || aligned16(G))) {
    const int64_t nchunks = n / 4;
    if (nchunks > 0) {
      const int grid = grid_for(nchunks, kThreads * kApplyUnroll, dev.sms, 8);
      launch_pdl(sign_apply_vec, grid, kThreads, 0, s, a, G, w_or_m, nchunks);
      if ((st = check_launch()) != EF_OK) return st;
    }
    begin = nchunks * 4;
  }
  if (begin < n) {
    const int grid = grid_for(n - begin, kThreads, dev.sms, 8);
    launch_pdl(sign_apply_scalar, grid, kThreads, 0, s, a, G, w_or_m, begin, n);
    if ((st = check_launch()) != EF_OK) return st;
  }
  prof_end(EF_KERNEL_SIGN_APPLY, s);
  return EF_OK;
}
