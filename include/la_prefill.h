/*
 * la_prefill.h -- C ABI of the GB300 (sm_103a) Lightning Attention chunkwise prefill.
 *
 * The operation (page "[Lightning Attention] Add Hopper SM90 CuTe DSL prefill",
 * Description and Reviewer notes; closed form on page "[LA] Lightning Attention MTP
 * decode + KVBuffer parallel verify / commit", Description):
 *
 *   for every sequence n and value head hv, with q/k head hq = hv / (HV / H) and
 *   lambda = exp(-slopes[hv]):
 *       S = h0[slot(n)][hv]  (or 0)                 S is FP32 [V][K]
 *       for t = 0 .. len(n) - 1:
 *           S   = lambda * S + v_t^T k_t            (S[v][k] += v_t[v] * k_t[k])
 *           o_t = scale * S q_t                     (o_t[v] = scale * sum_k S[v][k] q_t[k])
 *       h_final[slot(n)][hv] = S
 *
 * evaluated on the GPU in 64-token chunks: an intra-chunk term (Q K^T masked by the
 * causal decay lambda^(s-j)) V, an inter-chunk term lambda^(s+1) Q S^T, and one state
 * advance S <- lambda^L S + sum_j lambda^(L-1-j) v_j^T k_j per chunk of L tokens.
 *
 * Short sequences are evaluated token by token instead (one read and write of the state
 * and a few FP32 updates cost less than a chunkwise pipeline for one partial chunk), with
 * results within the same bounds: every sequence of a fixed-length batch with T <= 32, and
 * the sequences of at most 32 tokens of a packed batch whose average length is at most 64
 * (both kernels are then enqueued and each skips the other's sequences).
 *
 * Every pointer argument is a DEVICE pointer owned by the caller; the library keeps no
 * reference after the call returns and allocates no device memory.  The call is
 * asynchronous on `stream` and never synchronises with the host, so it may be
 * captured in a CUDA graph.
 */
#ifndef LA_PREFILL_H
#define LA_PREFILL_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LA_OK = 0,
  LA_ERR_INVALID_ARGUMENT = 1, /* null required pointer, bad size, misaligned pointer */
  LA_ERR_UNSUPPORTED = 2,      /* a shape this kernel does not implement (D != V, D not 64 or 128, ...) */
  LA_ERR_CUDA = 3              /* a CUDA runtime / driver call failed (launch, no sm_103a device) */
} la_status;

typedef enum {
  LA_SCHED_AUTO = 0,           /* library picks: currently persistent */
  LA_SCHED_PERSISTENT = 1,     /* one CTA per SM, each walks a static list of (sequence, head) units */
  LA_SCHED_NON_PERSISTENT = 2  /* one CTA per (sequence, head) unit */
} la_schedule;

/* Bits the kernel may OR into *dev_error (device memory, caller zeroes it). */
#define LA_DEV_ERR_BAD_SEQLENS 1u  /* cu_seqlens not non-decreasing / outside [0, B*T]: unit skipped */
#define LA_DEV_ERR_BAD_INDEX 2u    /* state_indices[n] >= pool_size: unit skipped */
#define LA_DEV_ERR_TIMEOUT 4u      /* an internal pipeline wait exceeded its limit: CTA stopped early */

/*
 * la_prefill_fwd -- forward (prefill) of decayed linear attention, chunkwise.
 *
 * Layouts (row-major, innermost dimension contiguous):
 *   q, k      bf16  [B*T, H, D]     token-major, heads interleaved
 *   v         bf16  [B*T, HV, V]
 *   o         bf16  [B*T, HV, V]    output; rows of padded sequences are not written
 *   slopes    fp32  [HV]            per value head; lambda = exp(-slope), slope >= 0 expected
 *   h0        fp32  [P, HV, V, D]   nullable (zero initial state); [V][K] orientation
 *   h_final   fp32  [P, HV, V, D]   nullable (final state not returned); may equal h0
 *                                   (in-place pool update); only selected slots written
 *   state_indices int32 [N]         nullable: sequence n uses slot n (P must be N);
 *                                   else slot state_indices[n], and a negative index
 *                                   marks a padded sequence: nothing is read or written
 *                                   for it.  Non-negative indices must be unique.
 *   cu_seqlens int32 [N+1]          nullable: fixed-length mode, N == B sequences of T
 *                                   tokens each; else packed mode: B must be 1, T is the
 *                                   total token count, sequence n spans
 *                                   [cu_seqlens[n], cu_seqlens[n+1]).
 *   P = pool_size                   number of state slots in h0 / h_final
 *   dev_error                       nullable device int; see LA_DEV_ERR_* (device-side
 *                                   checks never synchronise with the host)
 *
 * Supported: D == V == 128 or D == V == 64 (state [P, HV, D, D]), HV % H == 0, any
 * N >= 0 and any sequence lengths (including 0 and lengths that are not multiples of 64).
 * q, k, v, o, h0, h_final must be 16-byte aligned.  The outputs (o, h_final, dev_error) may
 * share no memory with an input or with each other (the kernels read ahead of their stores),
 * except that h_final may be h0 itself; the host checks the address ranges (the state ranges
 * span P slots with state_indices, N without) and returns LA_ERR_INVALID_ARGUMENT.
 *
 * Returns LA_OK after enqueueing the kernels (or with nothing to do when N == 0 or
 * B*T == 0 and no state is requested).  LA_ERR_INVALID_ARGUMENT and LA_ERR_UNSUPPORTED
 * mean nothing was launched; LA_ERR_CUDA from a failed launch may follow an enqueued
 * tokenwise kernel of the same call.
 */
la_status la_prefill_fwd(const void* q, const void* k, const void* v, const float* slopes, float scale,
                         const float* h0, const int32_t* state_indices, const int32_t* cu_seqlens, void* o,
                         float* h_final, int B, int T, int N, int H, int HV, int D, int V, int pool_size,
                         la_schedule schedule, int* dev_error, void* stream);

/* Human-readable name of a status code (static string). */
const char* la_status_string(la_status status);

/* Text of the last error recorded by this thread's calls (static per-thread buffer). */
const char* la_last_error(void);

/* Size in bytes of dynamic shared memory the kernel requests per CTA. */
int la_prefill_smem_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* LA_PREFILL_H */
