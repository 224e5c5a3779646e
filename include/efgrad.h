/*
 * efgrad.h -- C ABI of libefgrad: error-feedback gradient compression on
 * GB300 (sm_103a).
 *
 * Sources, cited by page title and section:
 *   [SPARSE] "梯度稀疏化：只传输重要的梯度元素" (Gradient sparsification:
 *            transmit only the important gradient elements).
 *   [ONEBIT] "1bit Adam梯度压缩技术原理与分布式训练优化" (1-bit Adam gradient
 *            compression: principle and distributed-training optimisation).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.  Pointers named h_* are host memory; every other buffer pointer is
 *   device memory of the current CUDA device.  The caller owns all buffers.
 *   The library allocates no device memory and keeps no caller pointer after
 *   a call returns.  The state it keeps between calls: per thread, the last
 *   CUDA error, a launch counter (ef_kernel_launches) and a profiling hook
 *   (ef_profile_events); per device, a cached description of the device (SM
 *   count, compute capability, shared-memory limit) and, for
 *   ef_topk_compress_noalloc only, the address of its own static scratch
 *   array.
 *   Scratch memory comes from a caller-provided workspace whose size the
 *   matching *_workspace_size query returns; it must be 256-byte aligned and
 *   may be reused by the next call on the same stream.
 * Streams.  `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *   default stream).  Calls enqueue work on it and return without
 *   synchronising; no device-to-host read-back happens inside a call.  The
 *   kernels are launched with programmatic stream serialization: one may be
 *   scheduled while the kernel before it in the stream drains, but none
 *   touches memory before every earlier kernel in the stream has completed,
 *   so the order of effects is the stream order.  A caller's own kernel
 *   launched with that attribute right after a call must likewise wait
 *   (cudaGridDependencySynchronize) before reading the call's outputs.
 * Numbers.  Every float is IEEE-754 binary32; every arithmetic step is a
 *   single round-to-nearest-even operation, never a fused multiply-add, in
 *   the order stated per function, so results are reproducible bit for bit.
 * Alignment.  Float / int32 / uint32 buffers must be 4-byte aligned.  The
 *   kernels use 16-byte vector accesses where the addresses allow it and
 *   scalar accesses otherwise; results do not depend on the path taken.
 * Errors.  Every call returns an ef_status.  Argument errors are detected on
 *   the host before anything is enqueued and leave every output untouched.
 *   Conditions that only the device can see (a bounded wait that ran out, a
 *   malformed packet) are written to a status word inside the workspace and
 *   read with ef_workspace_status().
 */
#ifndef EFGRAD_H
#define EFGRAD_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define EF_API __attribute__((visibility("default")))
#else
#define EF_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t ef_status;

#define EF_OK                  0
#define EF_ERR_NULL            1  /* a required pointer is NULL                        */
#define EF_ERR_SIZE            2  /* n < 0, or a size limit below is exceeded          */
#define EF_ERR_K               3  /* k < 0 or k > its segment's length                 */
#define EF_ERR_SEGMENTS        4  /* offsets do not rise monotonically from 0 to n     */
#define EF_ERR_ALIAS           5  /* an output overlaps a buffer it must not overlap   */
#define EF_ERR_WORKSPACE       6  /* workspace NULL, misaligned or too small           */
#define EF_ERR_WORKERS         7  /* W < 1 or W > EF_MAX_WORKERS                       */
#define EF_ERR_ARG             8  /* unknown enum value, or a non-finite scalar        */
#define EF_ERR_ALIGN           9  /* a pointer is not 4-byte aligned                   */
#define EF_ERR_ARCH           10  /* the current device is not compute capability 10.3 */
#define EF_ERR_CUDA           11  /* a CUDA call failed; see ef_last_cuda_error()      */
#define EF_ERR_DEVICE_TIMEOUT 12  /* device-side: a bounded inter-block wait ran out   */
#define EF_ERR_PACKET         13  /* device-side: packet indices not strictly ascending,
                                     out of range, or a bitmap whose population count
                                     differs from the stated k                         */
#define EF_ERR_INTERNAL       14  /* device-side: a consistency check failed (a library
                                     defect); the offending write was skipped           */
#define EF_ERR_CAPACITY       15  /* device-side: more elements were kept than the packet
                                     holds; the packet stops at its capacity and the
                                     rest stay in the residual                          */

#define EF_IDX_INT32   0  /* packet = fp32 values[k] + int32 global indices[k]        */
#define EF_IDX_BITMAP  1  /* packet = fp32 values[k] + uint32 bitmap[ceil(n/32)]      */

#define EF_APPLY_SGD       0  /* w <- w - eta * G                                    */
#define EF_APPLY_MOMENTUM  1  /* m <- beta1 * m + (1 - beta1) * G                      */

#define EF_MAX_WORKERS 64
#define EF_ABI_VERSION 1

/* Library ABI version (EF_ABI_VERSION of the build). */
EF_API int32_t ef_abi_version(void);

/* Static, NUL-terminated description of a status code. */
EF_API const char* ef_status_string(ef_status s);

/* cudaError_t of the last failed CUDA call made by this thread inside the
 * library (0 if none). */
EF_API int32_t ef_last_cuda_error(void);

/* Number of kernels this thread has launched through the library since the
 * library was loaded (memsets and event records are not counted). */
EF_API int64_t ef_kernel_launches(void);

/* ------------------------------------------------------------------------
 * Top-k error feedback, sender side.
 *
 * [SPARSE] §详细算法流程 steps 2-5, applied to each segment (tensor)
 * independently as §分层阈值与自适应稀疏率 and §分层自适应Top-k describe:
 *   g      = g_raw + e                     (step 2, e_0 = 0)
 *   S_s    = the k_s elements of segment s with the largest |g|; ties in |g|
 *            go to the lower index, and |g| is compared as the float's bit
 *            pattern with the sign cleared, so NaN ranks above +Inf and +0
 *            ties -0                        (step 3, §Top-k 稀疏化)
 *   e'     = g off S, +0.0 on S             (step 4: e = g - g~)
 *   packet = (g[i], i) for i in S           (step 5, §梯度稀疏化的基本原理 step 3)
 *
 * g_raw        [n] fp32, read only.
 * e            [n] fp32, in: e_{t-1}, out: e_t (updated in place).
 * n            elements in the flat buffer, 0 <= n; with EF_IDX_INT32 also
 *              n <= 2^31 so that every global index fits an int32.
 * nseg         number of segments, >= 1.
 * h_seg_offsets[nseg+1] host, 0 = off[0] <= off[1] <= ... <= off[nseg] = n;
 *              segment s is [off[s], off[s+1]), at most 2^31 elements.
 * h_seg_k[nseg] host, 0 <= k_s <= segment length.
 * idx_format   EF_IDX_INT32 or EF_IDX_BITMAP ([SPARSE] §索引编码压缩).
 * out_values   [sum k] fp32: segment 0's entries first; within a segment in
 *              ascending index order, so the packet ascends globally.
 * out_indices  [sum k] int32 global indices (INT32 format; NULL for BITMAP).
 * out_bitmap   [ceil(n/32)] uint32 (BITMAP format; NULL for INT32): bit i%32
 *              of word i/32 is set iff i is selected; padding bits are 0.
 * workspace    device scratch of at least ef_topk_workspace_size() bytes.
 * Outputs must not overlap g_raw, e, the workspace or each other; g_raw and
 * e must not overlap.  The result is unique (the order above is total), so it
 * does not depend on the launch configuration.
 * ---------------------------------------------------------------------- */
EF_API ef_status ef_topk_workspace_size(int64_t n, int32_t nseg,
                                 const int64_t* h_seg_offsets,
                                 const int64_t* h_seg_k, int32_t idx_format,
                                 size_t* bytes);

EF_API ef_status ef_topk_compress(const float* g_raw, float* e, int64_t n,
                           int32_t nseg, const int64_t* h_seg_offsets,
                           const int64_t* h_seg_k, int32_t idx_format,
                           float* out_values, int32_t* out_indices,
                           uint32_t* out_bitmap, void* workspace,
                           size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Top-k error feedback for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point; it is a library
 * convenience.  Some callers cannot call cudaMalloc when they compress: a
 * gradient hook that runs while a framework's caching allocator already
 * holds all free device memory (a raw cudaMalloc would fail or force the
 * pool to give memory back mid-step), or a host program in a latency-critical
 * section where an allocation, which may synchronise the device, is not
 * acceptable.  This call computes exactly what ef_topk_compress computes,
 * with the same arguments minus the workspace: its scratch is one
 * library-owned device array of EF_NOALLOC_SCRATCH_BYTES, which every GPU
 * that loads the library holds until the process exits.
 *
 * - Requests whose ef_topk_workspace_size() exceeds EF_NOALLOC_SCRATCH_BYTES
 *   are rejected with EF_ERR_WORKSPACE before anything is enqueued (use
 *   ef_topk_compress with your own workspace for those).
 * - The first call on each device looks up the array's device address with
 *   that device current; make that first call before any stream capture.
 * - All calls share the one array and it keeps the last call's contents (the
 *   call clears what must start at zero itself).  Calls whose GPU work can
 *   overlap -- on different streams, or from different threads without
 *   ordering -- race on it; issue them on one stream.
 * - Device-side conditions (EF_ERR_DEVICE_TIMEOUT, EF_ERR_INTERNAL) land in
 *   the status word at the start of the library's array; read them with
 *   ef_topk_noalloc_status() (which synchronises `stream`), before the next
 *   call on that device resets the word.
 * - The array's address is cached per device for the life of the process:
 *   after cudaDeviceReset() on a device, do not call this entry point (or
 *   its status query) on that device again in the same process.
 * It allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine.
 * ---------------------------------------------------------------------- */
#define EF_NOALLOC_SCRATCH_BYTES 33554432
EF_API ef_status ef_topk_compress_noalloc(const float* g_raw, float* e, int64_t n,
                                          int32_t nseg, const int64_t* h_seg_offsets,
                                          const int64_t* h_seg_k, int32_t idx_format,
                                          float* out_values, int32_t* out_indices,
                                          uint32_t* out_bitmap, void* stream);
/* Device-side status word of the last ef_topk_compress_noalloc call on the
 * current device: synchronises `stream`, then copies the word (EF_OK,
 * EF_ERR_DEVICE_TIMEOUT or EF_ERR_INTERNAL) to *device_status.  Allocates
 * nothing. */
EF_API ef_status ef_topk_noalloc_status(void* stream, int32_t* device_status);

/* ------------------------------------------------------------------------
 * Top-k error feedback with 8-bit packet values.
 *
 * [SPARSE] §与其他压缩技术的比较: after top-k, the selected values are
 * quantised to 8 bits.  The page gives no formula; the reading here is:
 *   per segment: s = RN(max|v| / 127) over its finite selected values
 *                (0 if it has none),
 *   q = round-half-even(clamp(RN(v / s), -127, 127)), 0 for NaN or s = 0,
 *   the receiver's value is RN(q * s), and the residual at a selected
 *   position becomes RN(v - RN(q * s)) (step 4, e = g - g~ with g~ what the
 *   packet carries); elsewhere it is g as in ef_topk_compress.
 *
 * Arguments as ef_topk_compress, except:
 * out_q       [sum k] int8 codes, in the same order as out_values would be.
 * out_scale   [nseg] fp32 per-segment scale (0 for a segment with k = 0).
 * workspace   >= ef_topk_q8_workspace_size() bytes, 256-byte aligned; it
 *             also holds the unquantised values and each entry's position.
 * out_q and out_scale must not overlap each other, the inputs, the index
 * output or the workspace.
 * ---------------------------------------------------------------------- */
EF_API ef_status ef_topk_q8_workspace_size(int64_t n, int32_t nseg,
                                           const int64_t* h_seg_offsets,
                                           const int64_t* h_seg_k, int32_t idx_format,
                                           size_t* bytes);
EF_API ef_status ef_topk_compress_q8(const float* g_raw, float* e, int64_t n, int32_t nseg,
                                     const int64_t* h_seg_offsets, const int64_t* h_seg_k,
                                     int32_t idx_format, int8_t* out_q, float* out_scale,
                                     int32_t* out_indices, uint32_t* out_bitmap,
                                     void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Receiver of 8-bit packet values: out_values[j] = RN(q[j] * scales[s])
 * for every entry j of segment s (the reading above).  The result feeds
 * sparse_aggregate_apply like any fp32 packet.
 *
 * q          [sum k] int8 codes (device).
 * scales     [nseg] fp32 per-segment scales (device, 4-byte aligned).
 * h_seg_k    [nseg] host array of per-segment entry counts (each 0..2^31).
 * out_values [sum k] fp32 (device, 4-byte aligned); must not overlap q or
 *            scales.
 * ---------------------------------------------------------------------- */
EF_API ef_status ef_q8_dequantize(const int8_t* q, const float* scales, int32_t nseg,
                                  const int64_t* h_seg_k, float* out_values, void* stream);

/* ------------------------------------------------------------------------
 * Index codecs for top-k packets.
 *
 * [SPARSE] §索引编码压缩 (block-sparse index: a dropped block costs one flag
 * bit, a kept block sends its inner indices; run-length and delta codes of
 * variable length) and §快速上手指南 step 4 (indices first as 16-bit
 * integers).  The page gives no formats; these are the library's readings.
 * Each codec maps an ascending int32 index list of K entries from [0, n)
 * (n <= 2^31) to one little-endian byte stream and back:
 *   EF_CODEC_LOCAL16    uint32 block_start[nblk + 1] (entries before each
 *                       65536-element block, nblk = ceil(n / 65536)), then
 *                       each entry's uint16 offset in its block.
 *                       Size 4 * (nblk + 1) + 2 * K.
 *   EF_CODEC_RUNVARINT  per entry, the number of unselected elements since
 *                       the previous entry (i_j - i_{j-1} - 1, i_{-1} = -1)
 *                       as unsigned LEB128 (7-bit groups, low first, the
 *                       high bit set on all but the last byte).  At most
 *                       5 * K bytes.
 *   EF_CODEC_BLOCK256   uint32 flags[nfw] (bit b % 32 of word b / 32 set when
 *                       256-element block b holds an entry; nfw =
 *                       ceil(ceil(n / 256) / 32)), then uint8 (count - 1)
 *                       of every flagged block in order, then each entry's
 *                       uint8 offset in its block.  Size 4 * nfw + (flagged
 *                       blocks) + K, at most 4 * nfw + 2 * K.
 *
 * ef_index_codec_sizes   upper bound of a stream's bytes and the workspace
 *                        bytes (for encode and decode) for K, n.
 * ef_index_encode        indices [K] int32 (device, 4-byte aligned) ->
 *                        out [out_capacity >= max bytes] (device, 4-byte
 *                        aligned); the stream's length is written to
 *                        *d_out_bytes (device uint64, 8-byte aligned), so
 *                        no host synchronisation is needed.
 * ef_index_decode        in [in_bytes] (device, 4-byte aligned; in_bytes is
 *                        the encoded length) -> indices [K] (device).
 *                        A length the format cannot have returns
 *                        EF_ERR_PACKET at once.
 * workspace: >= workspace_bytes, 256-byte aligned, not overlapping the
 * buffers.  Unsorted or out-of-range indices, and streams that do not parse
 * into K valid indices, set EF_ERR_PACKET in the workspace status word
 * (read it with ef_workspace_status); nothing is ever read or written out
 * of bounds.
 * ---------------------------------------------------------------------- */
#define EF_CODEC_LOCAL16 1
#define EF_CODEC_RUNVARINT 2
#define EF_CODEC_BLOCK256 3
EF_API ef_status ef_index_codec_sizes(int32_t codec, int64_t K, int64_t n,
                                      size_t* max_stream_bytes, size_t* workspace_bytes);
EF_API ef_status ef_index_encode(int32_t codec, const int32_t* indices, int64_t K, int64_t n,
                                 uint8_t* out, size_t out_capacity, uint64_t* d_out_bytes,
                                 void* workspace, size_t workspace_bytes, void* stream);
EF_API ef_status ef_index_decode(int32_t codec, const uint8_t* in, size_t in_bytes, int64_t K,
                                 int64_t n, int32_t* indices, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Random magnitude-proportional sparsification with error feedback.
 *
 * [SPARSE] §随机稀疏化: each element is kept with probability proportional to
 * |g|, normalised so that the expected count is k (in place of the top-k
 * selection of §详细算法流程 step 3; steps 2, 4 and 5 as ef_topk_compress).
 * The page gives no formula; the reading here, per segment:
 *   g = RN(g_raw + e), written over e;
 *   S = the exact sum of |g| over the finite elements, rounded once to fp64;
 *   c = RN32(k / S), 0 when S = 0;
 *   p_i = fmin(1, RN32(c * |g_i|)), 1 for Inf / NaN;
 *   u_i = (w_i >> 8) * 2^-24, w_i = word (i mod 4) of Philox4x32-10 at
 *         counter (i/4 low 32 bits, i/4 high, step low, step high) and key
 *         (seed low, seed high), i the global element index;
 *   kept iff u_i < p_i (segments with k = 0 keep nothing).  Where c|g_i| > 1
 *   the element is kept surely, so the expected count falls short of k by
 *   the clipped excess.
 * Kept elements are sent unscaled, in ascending global index order across
 * segments: out_values[j] = g_i, out_indices[j] = i, for the first
 * `capacity` kept elements; e = +0 where sent and g elsewhere (a kept
 * element past the capacity is not sent and keeps g; the device status
 * word then reads EF_ERR_CAPACITY).
 *
 * n            <= 2^31 (int32 indices); segments as ef_topk_compress.
 * seed, step   the generator's key and the counter's upper half.
 * out_values   [capacity] fp32, out_indices [capacity] int32 (device).
 * d_counts     [nseg + 1] int64 (device, 8-byte aligned): entries sent per
 *              segment, then their total (the packet length).
 * workspace    >= ef_randk_workspace_size() bytes, 256-byte aligned: about
 *              n/8 bytes of keep bits plus 16 bytes per 8192 elements.
 * No buffer may overlap another.
 * ---------------------------------------------------------------------- */
EF_API ef_status ef_randk_workspace_size(int64_t n, int32_t nseg, const int64_t* h_seg_offsets,
                                         const int64_t* h_seg_k, size_t* bytes);
EF_API ef_status ef_randk_compress(const float* g_raw, float* e, int64_t n, int32_t nseg,
                                   const int64_t* h_seg_offsets, const int64_t* h_seg_k,
                                   uint64_t seed, uint64_t step, float* out_values,
                                   int32_t* out_indices, int64_t capacity, int64_t* d_counts,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * 1-bit sign error feedback, sender side.
 *
 * [ONEBIT] §2.1 量化与误差补偿机制:
 *   v      = RN(g + eps)
 *   bit    = !(v < 0)            (sign(0) = +1, also for -0 and NaN)
 *   s      = bit ? +1 : -1       (the quantised gradient ghat)
 *   Delta  = RN(v - s)
 *   c      = RN(1 - beta1)
 *   eps'   = RN(RN(beta1 * eps) + RN(c * Delta))
 *
 * g        [n] fp32 gradient, read only.
 * eps      [n] fp32 error buffer, in: eps_{t-1}, out: eps_t (in place).
 * beta1    EMA coefficient (the pages use 0.9); must be finite.
 * out_bits [ceil(n/32)] uint32: bit i%32 of word i/32 is element i's bit;
 *          padding bits 0.  Must not overlap g or eps; g and eps must not
 *          overlap.
 * Device status: none can arise.  The kernels have no inter-block waits and
 * every address they touch follows from n alone (no index is read from
 * memory), so this call and sign_aggregate_apply take no workspace and have
 * no device-side status word; argument errors are returned directly.
 * ---------------------------------------------------------------------- */
EF_API ef_status ef_sign_compress(const float* g, float* eps, int64_t n, float beta1,
                           uint32_t* out_bits, void* stream);

/* ------------------------------------------------------------------------
 * Receive side for top-k packets.
 *
 * [SPARSE] §详细算法流程 steps 6-7 (and the receiver of §梯度稀疏化的基本原理):
 *   G[i] = (((+0 + p_0[i]) + p_1[i]) + ... + p_{W-1}[i])   worker order,
 *          where p_w[i] is worker w's packet value at i or absent (no term)
 *   w[i] = RN(w[i] - RN(eta * G[i]))   at every i some packet contains;
 *          elsewhere w is not accessed (and would be unchanged: G = 0).
 *
 * W           number of workers' packets, 1 <= W <= EF_MAX_WORKERS.
 * idx_format  EF_IDX_INT32 or EF_IDX_BITMAP, the same for all packets.
 * h_values[W] host array of device pointers to fp32 values[k_w].
 * h_indices[W] host array of device pointers to int32 indices[k_w], strictly
 *             ascending within a packet, each in [0, n) (INT32; else NULL).
 * h_bitmaps[W] host array of device pointers to uint32 bitmaps[ceil(n/32)]
 *             (BITMAP; else NULL); values follow the set bits in order.
 * h_k[W]      host, entries per packet, 0 <= k_w <= n.
 * n           length of the dense gradient / parameter vector.
 * eta         learning rate, finite.
 * G           [n] fp32 dense aggregated gradient, written in full; may be
 *             NULL to skip the dense write (then only touched w change).
 * w           [n] fp32 parameters, updated in place.
 * workspace   device scratch of at least ef_aggregate_workspace_size().
 * Malformed packets (unsorted, out-of-range index, bitmap population count
 * different from k_w) are never read out of bounds; they set EF_ERR_PACKET
 * in the workspace status and the outputs are then unspecified.
 * ---------------------------------------------------------------------- */
EF_API ef_status ef_aggregate_workspace_size(int32_t W, int32_t idx_format, int64_t n,
                                      size_t* bytes);

EF_API ef_status sparse_aggregate_apply(int32_t W, int32_t idx_format,
                                 const float* const* h_values,
                                 const int32_t* const* h_indices,
                                 const uint32_t* const* h_bitmaps,
                                 const int64_t* h_k, int64_t n, float eta,
                                 float* G, float* w, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Packet exchange between data-parallel ranks, index-range form.
 *
 * [SPARSE] §详细算法流程 step 5 and §与Allreduce的融合: the workers' sparse
 * packets are exchanged with collectives and summed by the receivers.  In
 * the index-range form rank q owns the indices [b_q, b_{q+1}): every rank
 * sends each owner the slice of its ascending packet that falls in the
 * owner's range, and each owner runs sparse_aggregate_apply on its range
 * alone with the slices rebased to it.  These two calls are the device
 * steps of that exchange (the collectives themselves are the caller's).
 *
 * ef_packet_split  d_starts[q] = number of entries j < k with
 *                  indices[j] < h_bounds[q], for q = 0 .. nparts: in an
 *                  ascending packet, the slice for range q is
 *                  [d_starts[q], d_starts[q+1]).
 *   indices   [k] int32 (device, 4-byte aligned), 0 <= k <= 2^31.
 *   nparts    1 .. 1024 ranges; h_bounds [nparts + 1] host int64,
 *             non-decreasing (EF_ERR_SEGMENTS otherwise).
 *   d_starts  [nparts + 1] int64 (device, 8-byte aligned), must not overlap
 *             indices.
 *   Reads only indices[0 .. k); an unsorted packet gives positions in
 *   [0, k] that the receive side then reports as malformed.
 * ef_index_rebase  indices[j] = indices[j] - base for j < count, in place
 *                  (0 <= count <= 2^31, 0 <= base <= 2^31).
 * ---------------------------------------------------------------------- */
EF_API ef_status ef_packet_split(const int32_t* indices, int64_t k, int32_t nparts,
                                 const int64_t* h_bounds, int64_t* d_starts, void* stream);
EF_API ef_status ef_index_rebase(int32_t* indices, int64_t count, int64_t base,
                                 void* stream);

/* ------------------------------------------------------------------------
 * Receive side for 1-bit packets.
 *
 * G[i] = sum over workers of (bit_w[i] ? +1 : -1), added in worker order onto
 *        +0 (exact small integers), the sum of [SPARSE] §详细算法流程 step 6
 *        applied to [ONEBIT] sign packets; then
 *   EF_APPLY_SGD:       w[i] = RN(w[i] - RN(eta * G[i]))   ([SPARSE] step 7)
 *   EF_APPLY_MOMENTUM:  m[i] = RN(RN(beta1 * m[i]) + RN(RN(1 - beta1) * G[i]))
 *                       ([ONEBIT] §2.2 动量修正策略; with W = 1, G = ghat)
 *
 * h_bits[W]   host array of device pointers to uint32 bits[ceil(n/32)].
 * mode        EF_APPLY_SGD or EF_APPLY_MOMENTUM; eta / beta1 finite (the one
 *             the mode does not use is ignored).
 * G           [n] fp32, written in full; may be NULL.
 * w_or_m      [n] fp32 parameters (SGD) or momentum (MOMENTUM), in place.
 * ---------------------------------------------------------------------- */
EF_API ef_status sign_aggregate_apply(int32_t W, const uint32_t* const* h_bits,
                               int64_t n, int32_t mode, float eta, float beta1,
                               float* G, float* w_or_m, void* stream);

/* ------------------------------------------------------------------------
 * Device-side status of the last call that used `workspace`: synchronises
 * `stream`, then copies the status word (EF_OK, EF_ERR_DEVICE_TIMEOUT or
 * EF_ERR_PACKET) to *device_status.  Each call that takes a workspace resets
 * the word when it starts.
 * ---------------------------------------------------------------------- */
EF_API ef_status ef_workspace_status(const void* workspace, void* stream,
                              int32_t* device_status);

/* ------------------------------------------------------------------------
 * Self-test of the bounded inter-block wait.  Launches one warp that runs
 * the library's look-back wait on a predecessor whose state nothing ever
 * publishes, with a wall-clock limit of limit_ns (1 ms .. 10 s).  The wait
 * must give up, record EF_ERR_DEVICE_TIMEOUT in the workspace status word and
 * return, leaving the context usable; read the result with
 * ef_workspace_status().  workspace: >= 512 bytes, 256-byte aligned.
 * ---------------------------------------------------------------------- */
EF_API ef_status ef_selftest_wait_timeout(void* workspace, size_t workspace_bytes,
                                          int64_t limit_ns, void* stream);

/* ------------------------------------------------------------------------
 * Profiling hook (per calling thread).  While set, every launch of kernel
 * `kernel_id` made by this thread is bracketed by cudaEventRecord(start) and
 * cudaEventRecord(stop) on the call's stream, so the caller can time that
 * one kernel with its own events.  Pass NULL events to clear.
 * ---------------------------------------------------------------------- */
#define EF_KERNEL_TOPK_FUSED   1  /* compensate + residual write + candidates */
#define EF_KERNEL_SIGN         2  /* 1-bit compress                           */
#define EF_KERNEL_SPARSE_APPLY 3  /* dense tile merge + SGD                   */
#define EF_KERNEL_SIGN_APPLY   4  /* 1-bit aggregate + SGD / momentum         */
EF_API ef_status ef_profile_events(int32_t kernel_id, void* start_event,
                            void* stop_event);

#ifdef __cplusplus
}
#endif

#endif /* EFGRAD_H */
