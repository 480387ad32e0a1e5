// la_prefill_internal.h -- entry points shared between the library's translation units, not part
// of the C ABI.
#pragma once

#include <cstdint>

#include "../../include/la_prefill.h"

namespace la_internal {

// The chunkwise kernel on every sequence, however short (no tokenwise split), with its units
// dealt out round robin: the recurrence of la_prefill_fwd per (sequence, head h < HV),
//     S_t = lambda_h S_(t-1) + v_t^T k_t,   o_t = scale S_t q_t,
// with q, k of head h / (HV / H) (H heads) and v of head h / (HV / v_heads) (v_heads heads, a
// divisor of HV: v_heads = HV is la_prefill_fwd's layout, v_heads = H shares one v head among a
// group of HV / H), the state and the output of head h.  With `reverse` the recurrence runs over
// each sequence from its last token to its first, on the tokens in place (S starts from h0 after
// the last token, h_final is the state before the first).  The output is BF16 into `o`, or FP32
// into `o_f32` when that is not null (same [tokens, HV, D] layout).  Arguments, layouts and checks
// otherwise as la_prefill_fwd (D == V).  Used by the backward pass.
la_status chunkwise(const void* q, const void* k, const void* v, const float* slopes, float scale, const float* h0,
                    const int32_t* state_indices, const int32_t* cu_seqlens, void* o, float* o_f32, float* h_final,
                    int B, int T, int N, int H, int HV, int v_heads, int D, int pool_size, bool reverse,
                    int* dev_error, void* stream);

}  // namespace la_internal
