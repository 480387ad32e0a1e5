/*
 * la_d256.h -- C ABI of the GB300 (sm_103a) Lightning Attention prefill at head dimension
 * D = V = 256.
 *
 * The operation is la_prefill_fwd's (include/la_prefill.h; page "[Lightning Attention] Add
 * Hopper SM90 CuTe DSL prefill", Description, whose Reviewer notes leave head sizes other than
 * 128 out of that kernel's scope) with D = V = 256.  A 256 x 256 FP32 state fills the whole
 * tensor memory of an SM, so this library evaluates it as four 128 x 128 blocks, which the
 * recurrence keeps independent of one another:
 *
 *   S[v][k] = lambda S[v][k] + v_t[v] k_t[k] updates every element on its own, so the blocks
 *   S_ab = S[a half of v][b half of k] (a, b in {0, 1}) evolve separately, each from its own
 *   block of h0; and since q_t . k_j = q_t[lo] . k_j[lo] + q_t[hi] . k_j[hi],
 *       o_t[a half] = sum over b of  lightning(q[b half], k[b half], v[a half], S_ab)_t
 *   where lightning() is the D = 128 chunkwise computation of la_prefill_fwd.
 *
 * So one call runs the D = 128 chunkwise kernel over 4 HV virtual heads (q, k read in place as
 * [tokens, 2H, 128], v as [tokens, 2HV, 128]), each writing its part of o in FP32; a sum adds the
 * two key halves of every output and rounds once to BF16.  Around it, small kernels copy the
 * selected h0 blocks into the workspace and the final blocks back to h_final.  Outputs equal the
 * D = 256 recurrence up to FP32 rounding order.
 *
 * Layouts as la_prefill_fwd with D = V = 256: q, k bf16 [B*T, H, 256]; v, o bf16 [B*T, HV, 256];
 * slopes fp32 [HV]; h0, h_final fp32 [P, HV, 256, 256] (nullable; h_final may be h0).
 * Fixed-length batches (cu_seqlens null) with T <= 32 run the tokenwise recurrence instead, on
 * whole 256 x 256 states (the D = 256 instance of the speculative-decoding ops' kernel, see
 * la_decode.h): BF16 outputs directly, no workspace.
 */
#ifndef LA_D256_H
#define LA_D256_H

#include <stddef.h>
#include <stdint.h>

#include "la_prefill.h"
#include "la_segment.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * la_prefill_d256_workspace -- device workspace bytes la_prefill_fwd_d256 needs for a batch of
 * B*T tokens, N sequences and HV value heads: the FP32 parts of o (B*T x 4 HV x 128 floats), one
 * [4 HV, 128, 128] FP32 block set per sequence (only when h0 or h_final is given: has_state), the
 * per-virtual-head slopes and the per-sequence slot table.  Errors: LA_ERR_INVALID_ARGUMENT for
 * negative sizes, LA_ERR_UNSUPPORTED when a size overflows.
 */
la_status la_prefill_d256_workspace(int B, int T, int N, int HV, int has_state, size_t* bytes);

/*
 * la_prefill_fwd_d256 -- la_prefill_fwd at D = V = 256.
 *
 * Arguments as la_prefill_fwd (no schedule; D and V must be 256), plus
 *   workspace        device buffer of at least la_prefill_d256_workspace(B, T, N, HV,
 *                    h0 || h_final) bytes, 256-byte aligned; its contents on entry do not
 *                    matter; it may share no memory with any other argument.  Not used (and
 *                    may be null) for a fixed-length batch with T <= 32
 *   workspace_bytes  its size
 * Device-side errors go to *dev_error as for la_prefill_fwd (a bad state index skips its
 * sequence, bad bounds skip theirs).  Returns LA_OK after enqueueing (or with nothing to do);
 * LA_ERR_INVALID_ARGUMENT / LA_ERR_UNSUPPORTED with nothing enqueued; LA_ERR_CUDA if a launch
 * failed (earlier kernels of the call may then have been enqueued).
 */
la_status la_prefill_fwd_d256(const void* q, const void* k, const void* v, const float* slopes, float scale,
                              const float* h0, const int32_t* state_indices, const int32_t* cu_seqlens, void* o,
                              float* h_final, int B, int T, int N, int H, int HV, int D, int V, int pool_size,
                              void* workspace, size_t workspace_bytes, int* dev_error, void* stream);

/*
 * la_prefill_d256_segmented_workspace -- device workspace bytes la_prefill_fwd_d256_segmented
 * needs: la_prefill_d256_workspace's, plus la_prefill_segmented_workspace's for the 4 HV block
 * heads (B, T, N, packed and segment_len as there; 0 = automatic, resolved with the CURRENT
 * device's SM count over the 4 N HV block chains).  Writes the resolved segment length to
 * *resolved_segment_len (nullable; 0 when no segmentation is done).  Errors as the two queries.
 */
la_status la_prefill_d256_segmented_workspace(int B, int T, int N, int HV, int packed, int segment_len, int has_state,
                                              size_t* bytes, int* resolved_segment_len);

/*
 * la_prefill_fwd_d256_segmented -- la_prefill_fwd_d256 with every sequence cut into segments of
 * segment_len tokens that run in parallel from their exact initial states (include/la_segment.h),
 * for batches with few (sequence, value head) chains.  The segmented prefill runs on the block
 * heads (4 HV per sequence), so its local states, scan and chunkwise pass are those of D = 128;
 * the sum of the key halves and the final blocks follow as in la_prefill_fwd_d256.  Every
 * sequence, however short, takes this path (no tokenwise path).
 *
 * Arguments as la_prefill_fwd_d256, plus segment_len (as given to the workspace query); the
 * workspace is at least la_prefill_d256_segmented_workspace(...) bytes.  Outputs equal
 * la_prefill_fwd_d256's up to FP32 rounding order.  Returns as la_prefill_fwd_d256.
 */
la_status la_prefill_fwd_d256_segmented(const void* q, const void* k, const void* v, const float* slopes, float scale,
                                        const float* h0, const int32_t* state_indices, const int32_t* cu_seqlens,
                                        void* o, float* h_final, int B, int T, int N, int H, int HV, int D, int V,
                                        int pool_size, int segment_len, void* workspace, size_t workspace_bytes,
                                        int* dev_error, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LA_D256_H */
