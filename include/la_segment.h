/*
 * la_segment.h -- C ABI of the segmented-sequence Lightning Attention prefill (GB300, sm_103a).
 *
 * The same operation as la_prefill_fwd (include/la_prefill.h, whose contract every argument
 * below shares), for batches with few (sequence, value head) chains: a long prefill on a
 * tensor-parallel shard of a few heads, say, where one chain per SM would leave most of the
 * GPU idle while each chain walks its chunks in order.  Each sequence is cut into segments
 * of S tokens.  Since a chain's state is affine in its initial state (a segment of L tokens
 * maps H to lambda^L H + Sloc, Sloc being the segment run from a zero state), the segments
 * run in parallel in three passes:
 *   1. Sloc of every segment but the last of each sequence (tensor cores, reads K and V);
 *   2. a scan over each sequence's segments: H_0 = h0, H_{i+1} = lambda^{L_i} H_i + Sloc_i;
 *   3. the chunkwise prefill of every segment from its initial state H_i (la_prefill_fwd's
 *      kernel), whose last segment leaves the sequence's final state.
 * The segmented affine scan is the one page "linear_attention: add a Hopper (sm90) KDA
 * prefill path - #1017" (How) uses for a decayed recurrence of the same shape.  The
 * outputs equal la_prefill_fwd's up to FP32 rounding order (the initial states are exact
 * sums computed in another order); they are not bitwise equal.
 *
 * Cost: pass 1 reads K and V of every segment but the last once more, so it pays off only
 * when the batch has far fewer chains than SMs.  With segment_len == 0 the library decides:
 * it runs la_prefill_fwd unchanged (no workspace used) unless N * HV is at most half the SM
 * count, and otherwise picks S so that the segments fill the SMs about once.  When that gives
 * two segments per fixed-length sequence, the automatic plan instead cuts the first half of
 * each sequence into two segments of the resolved length and keeps the second half as one
 * longer last segment: pass 1 (which the last segment does not need) then runs twice as many
 * units of half the length.
 *
 * Every pointer is a DEVICE pointer owned by the caller.  The call allocates nothing, never
 * synchronises with the host and enqueues its kernels (6 at most) on `stream`.
 */
#ifndef LA_SEGMENT_H
#define LA_SEGMENT_H

#include <stddef.h>
#include <stdint.h>

#include "la_prefill.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * la_prefill_segmented_workspace -- device workspace bytes la_prefill_fwd_segmented needs.
 *
 * Same B, T, N, HV and mode (packed = 1 when cu_seqlens will be given) as the call, and the
 * same segment_len (0 = automatic, resolved with the CURRENT device's SM count; else a
 * positive multiple of 64).  Writes the byte count to *bytes (0 when the call would run
 * la_prefill_fwd unchanged) and the resolved segment length to *resolved_segment_len
 * (nullable; 0 when no segmentation is done).  Errors: LA_ERR_INVALID_ARGUMENT for bad sizes
 * or a segment_len that is not a positive multiple of 64, LA_ERR_CUDA when the device
 * query fails.
 *
 * The workspace holds one FP32 [128 x 128] state per (segment, value head) -- 64 KiB each --
 * plus five int32 tables; the segment count is at most N + floor(B*T / S) (packed) or
 * B * ceil(T / S) (fixed length).  The size does not depend on D: a D = V = 64 call keeps its
 * [64 x 64] states in the first quarter of the same state region.
 */
la_status la_prefill_segmented_workspace(int B, int T, int N, int HV, int packed, int segment_len, size_t* bytes,
                                         int* resolved_segment_len);

/*
 * la_prefill_fwd_segmented -- la_prefill_fwd over segments of segment_len tokens.
 *
 * Arguments as la_prefill_fwd (no schedule; D == V == 128 or 64), plus:
 *   segment_len      0 = automatic, else a positive multiple of 64 (the same value given to
 *                    la_prefill_segmented_workspace)
 *   workspace        device buffer of at least the queried size, 256-byte aligned; may be
 *                    null when the queried size is 0.  Its contents on entry do not matter,
 *                    and it may be reused as soon as the stream has run the call; two calls
 *                    that share one workspace must not overlap on the GPU.
 *   workspace_bytes  its size
 *
 * Device-side errors go to *dev_error as for la_prefill_fwd; bounds whose segments would not
 * fit the workspace (overlapping cu_seqlens ranges) also set LA_DEV_ERR_BAD_SEQLENS and
 * skip the sequences concerned.  The buffers follow la_prefill_fwd's rule on overlap, and the
 * workspace may share no memory with any of them.  Returns LA_OK after enqueueing;
 * LA_ERR_INVALID_ARGUMENT / LA_ERR_UNSUPPORTED with nothing enqueued; LA_ERR_CUDA if a launch failed (earlier passes
 * may then have been enqueued).
 */
la_status la_prefill_fwd_segmented(const void* q, const void* k, const void* v, const float* slopes, float scale,
                                   const float* h0, const int32_t* state_indices, const int32_t* cu_seqlens,
                                   void* o, float* h_final, int B, int T, int N, int H, int HV, int D, int V,
                                   int pool_size, int segment_len, void* workspace, size_t workspace_bytes,
                                   int* dev_error, void* stream);

/*
 * la_prefill_fwd_segmented_static -- la_prefill_fwd_segmented without a caller workspace.
 *
 * No counterpart in the pages: an addition of this library for callers that cannot allocate
 * device memory -- a plugin inside an inference server or framework that owns every byte of
 * device memory and offers its extensions no allocation call, or a latency-critical path that
 * must not call cudaMalloc (which may synchronise the device).  The scratch the segmented
 * prefill needs comes from a 16 MiB buffer built into the library: a file-scope device array
 * that every GPU holds, once the library's code is loaded on it, until the process exits.  The
 * call itself allocates no device memory.
 *
 * Arguments as la_prefill_fwd_segmented, without workspace / workspace_bytes.
 *   - Calls whose plan needs more than 16 MiB (la_prefill_segmented_workspace) return
 *     LA_ERR_UNSUPPORTED and launch nothing; every automatic segment length (segment_len = 0) on
 *     a GB300 (152 SMs) needs at most about 14.3 MiB.
 *   - The first call on a device that segments looks the buffer's address up (one
 *     cudaGetSymbolAddress, with that device current, which may load the library's code on it);
 *     make that first call before any stream capture.
 *   - Every call on a device shares the one buffer and leaves its contents behind; nothing in it
 *     has to start at zero (each call rewrites every table entry and state before reading it).
 *     Two calls that overlap on the GPU (different streams, or threads without ordering) race on
 *     the buffer and corrupt each other's results: order them on one stream.
 */
la_status la_prefill_fwd_segmented_static(const void* q, const void* k, const void* v, const float* slopes,
                                          float scale, const float* h0, const int32_t* state_indices,
                                          const int32_t* cu_seqlens, void* o, float* h_final, int B, int T, int N,
                                          int H, int HV, int D, int V, int pool_size, int segment_len,
                                          int* dev_error, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LA_SEGMENT_H */
