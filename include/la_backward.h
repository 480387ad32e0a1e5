/*
 * la_backward.h -- C ABI of the backward pass of the Lightning Attention prefill.
 *
 * The pages describe the forward pass only ("[Lightning Attention] Add Hopper SM90 CuTe DSL
 * prefill", Reviewer notes, name the backward outside that kernel's scope); the backward here
 * is the chain rule applied to the forward recurrence of that page's Description,
 *     S_t = lambda S_{t-1} + v_t k_t^T   (S_{-1} = h0, S stored [V][K]),   o_t = scale S_t q_t,
 * for a scalar loss L with dout_t = dL/do_t and dh_final = dL/dS_{L-1}:
 *     dq_t = scale S_t^T dout_t
 *     G_t  = dL/dS_t = scale dout_t q_t^T + lambda G_{t+1},   G_{L-1} = scale dout q^T + dh_final
 *     dk_t = G_t^T v_t,   dv_t = G_t k_t,   dh0 = lambda G_0   (dh0 = dh_final when L = 0)
 * Each of dq, dv and dk is itself the forward recurrence on rearranged inputs, so the call runs
 * the chunkwise kernel three times:
 *     dq = forward(q' = dout, k' = v, v' = k, h0' = h0^T)                          in token order
 *     dv = forward(q' = k, k' = q, v' = dout, h0' = dh_final / (lambda scale))     in reverse order
 *     dk = forward(q' = v, k' = dout, v' = q, h0' = (dh_final / (lambda scale))^T) in reverse order
 * where reverse order runs the recurrence over each sequence from its last token to its first,
 * on the tokens in place (the kernel's reverse instance: chunks from last to first, the causal
 * mask and the decay exponents of a chunk mirrored), and dh0 = lambda scale times the final
 * state of the dv run.  With G = HV / H value heads per q/k head (GVA), dv runs per value head
 * as written; dq and dk are sums over a q/k head's value heads, so their runs go per value head
 * (q' and k' of HV heads, v' of the H q/k heads) into FP32 parts that are summed per group.  (The forward pass decays its initial
 * state by lambda^(t+1) at token t, the gradient of the final state enters G undecayed at the
 * last token: hence the 1 / lambda.)  For a head with slope > 64 (lambda < e^-64) the reversed
 * runs start from zero and dh_final's term, which is below FP32 resolution at every token but
 * the last, is added at the last token by a small fix-up kernel.
 */
#ifndef LA_BACKWARD_H
#define LA_BACKWARD_H

#include <stddef.h>
#include <stdint.h>

#include "la_prefill.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Bytes of device workspace la_prefill_bwd needs for these sizes (has_h0 / has_dh_final: 0 or
 * 1): a transposed copy of h0 and the scaled (and transposed) dh_final, P x HV states of D x D
 * FP32 each, and, when value heads share q/k heads (HV > H), one B*T x HV x D FP32 buffer for the
 * value heads' parts of dq and dk; 0 when none of these is needed.  Host only.
 */
la_status la_prefill_bwd_workspace(int B, int T, int H, int HV, int D, int pool_size, int has_h0,
                                   int has_dh_final, size_t* bytes);

/*
 * la_prefill_bwd -- gradients of the prefill with respect to q, k, v and h0.
 *
 * Inputs: the forward call's q, k, v, slopes, scale, h0 (nullable), state_indices (nullable),
 * cu_seqlens (nullable) with the forward's layouts and meaning (la_prefill.h), plus
 *   dout      bf16  [B*T, HV, D]    dL/do
 *   dh_final  fp32  [P, HV, D, D]   nullable (dL/dh_final = 0); needs scale != 0
 * Outputs (caller-owned device memory; rows of padded sequences and unselected slots are not
 * written):
 *   dq, dk    bf16 [B*T, H, D]
 *   dv        bf16 [B*T, HV, D]
 *   dh0       fp32  [P, HV, D, D]   nullable (not computed)
 * workspace: device memory of at least la_prefill_bwd_workspace(...) bytes, 256-byte aligned,
 * owned by the caller, not read before it is written (nullable when that size is 0); calls
 * sharing one workspace must not overlap on the GPU.
 *
 * Supported: HV a multiple of H (GVA: the G = HV / H value heads of a q/k head each contribute
 * to its dq and dk, which are summed in FP32 over the group before the one rounding to BF16),
 * D == V == 128 or 64, any N >= 0 and any sequence lengths; 16-byte aligned tensors.  Other shapes return LA_ERR_UNSUPPORTED and
 * launch nothing; invalid arguments LA_ERR_INVALID_ARGUMENT, among them outputs (dq, dk, dv,
 * dh0, the workspace, dev_error) that share memory with an input or with each other (address
 * ranges checked on the host).  Device-side errors (bad
 * cu_seqlens, bad state indices) set bits in *dev_error as for la_prefill_fwd.  The call
 * enqueues its kernels on `stream` and never synchronises with the host.
 */
la_status la_prefill_bwd(const void* q, const void* k, const void* v, const float* slopes, float scale,
                         const float* h0, const void* dout, const float* dh_final, const int32_t* state_indices,
                         const int32_t* cu_seqlens, void* dq, void* dk, void* dv, float* dh0, int B, int T, int N,
                         int H, int HV, int D, int V, int pool_size, void* workspace, size_t workspace_bytes,
                         int* dev_error, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LA_BACKWARD_H */
