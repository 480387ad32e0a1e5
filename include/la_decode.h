/*
 * la_decode.h -- C ABI of the GB300 (sm_103a) Lightning Attention speculative-decoding ops:
 * multi-token (MTP) decode, parallel verify with an optional KV buffer, and commit.
 *
 * The operations (page "[LA] Lightning Attention MTP decode + KVBuffer parallel verify /
 * commit", Description; the recurrence is the one of la_prefill.h):
 *
 *   for every request b with slot = state_indices[b] (or b) >= 0 and value head hv,
 *   q/k head hq = hv / (HV / H), lambda = exp(-slopes[hv]), S = state[slot][hv] (FP32 [V][K]):
 *
 *   la_decode_mtp  over the T draft tokens t = 0 .. T-1 of the request:
 *                      S = lambda S + v_t^T k_t ;  o_t = scale S q_t
 *                  and S is written back to state[slot][hv] (the pool is updated in place).
 *   la_verify      the same outputs o_t, t = 0 .. T-1, by the closed form ("Closed form used
 *                  by verify")
 *                      o_t = lambda^(t+1) scale (S q_t) + sum_{i<=t} lambda^(t-i) scale (q_t . k_i) v_i
 *                  with the pool left untouched; optionally k_t, v_t are copied into a
 *                  pooled KV buffer at the request's slot for a later commit.  For T <= 8 the
 *                  products S q_t run on the tensor cores with S and q_t as TF32 operands (the
 *                  pages' verify kernel also multiplies the state by q in TF32), so the outputs
 *                  equal la_decode_mtp's within that rounding; for T > 8, and for D = 64 and
 *                  256, verify runs decode's tokenwise recurrence and its outputs are bitwise
 *                  decode's.
 *   la_commit      with L = accepted_len[b] (0 <= L <= T) taken from that KV buffer:
 *                      S = lambda^L S + sum_{i<L} lambda^(L-1-i) v_i^T k_i   (L = 0: no-op)
 *                  written back to state[slot][hv].  With L == T the committed state is
 *                  bitwise the state la_decode_mtp leaves (same arithmetic in the same order).
 *
 * Requests with a negative state index are padded: nothing is read or written for them
 * (their o rows and every pool slot are left untouched).  Every pointer is a caller-owned
 * DEVICE pointer; nothing is allocated and no call synchronises with the host.
 *
 * Layouts (row-major, innermost contiguous):
 *   q, k      bf16 [B*T, H, D]        token-major, T tokens per request
 *   v, o      bf16 [B*T, HV, V]
 *   slopes    fp32 [HV]
 *   state     fp32 [P, HV, V, D]      the state pool, [V][K] orientation
 *   state_indices int32 [B]           nullable: request b uses slot b (P >= B); else the slot,
 *                                     negative = padded; non-negative indices must be unique
 *   kbuf      bf16 [P, T, H, D]       KV buffer (nullable in la_verify: no copy), slot-major
 *   vbuf      bf16 [P, T, HV, V]
 *   accepted_len int32 [B]            tokens to commit per request, clamped to [0, T]
 *   dev_error device int, nullable    LA_DEV_ERR_BAD_INDEX when a slot >= P (request skipped)
 * Supported: D == V == 128, 64 or 256, HV % H == 0, T >= 1 (any B >= 0); 16-byte aligned
 * pointers.
 * What a call writes (o, kbuf, vbuf; the pool in decode and commit; dev_error) may share no
 * memory with what it reads or with another of its outputs: LA_ERR_INVALID_ARGUMENT (address
 * ranges checked on the host; pool and KV buffer span P slots with state_indices, B without).
 * Returns LA_OK after enqueueing (or with nothing to do when B == 0); any other status means
 * nothing was launched.
 */
#ifndef LA_DECODE_H
#define LA_DECODE_H

#include <stdint.h>

#include "la_prefill.h"

#ifdef __cplusplus
extern "C" {
#endif

la_status la_decode_mtp(const void* q, const void* k, const void* v, const float* slopes, float scale,
                        float* state, const int32_t* state_indices, void* o, int B, int T, int H, int HV, int D,
                        int V, int pool_size, int* dev_error, void* stream);

la_status la_verify(const void* q, const void* k, const void* v, const float* slopes, float scale,
                    const float* state, const int32_t* state_indices, void* o, void* kbuf, void* vbuf, int B, int T,
                    int H, int HV, int D, int V, int pool_size, int* dev_error, void* stream);

la_status la_commit(float* state, const int32_t* state_indices, const void* kbuf, const void* vbuf,
                    const int32_t* accepted_len, const float* slopes, int B, int T, int H, int HV, int D, int V,
                    int pool_size, int* dev_error, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LA_DECODE_H */
