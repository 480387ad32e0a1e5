// la_prefill_internal.h -- entry points shared between the library's translation units, not part
// of the C ABI.
#pragma once

#include <cstdint>

#include "../../include/la_prefill.h"

namespace la_internal {

// The recurrence of la_prefill_fwd run over each sequence from its last token to its first:
//     S_t = lambda S_(t+1) + v_t^T k_t   (S_L = h0),   o_t = scale S_t q_t,   h_final = S_0,
// on the tokens in place (o written in token order).  Same arguments, layouts and checks as
// la_prefill_fwd; the chunkwise kernel's reverse instance takes every sequence, whatever its
// length, with units dealt out round robin.  Used by the backward pass.
la_status prefill_reverse(const void* q, const void* k, const void* v, const float* slopes, float scale,
                          const float* h0, const int32_t* state_indices, const int32_t* cu_seqlens, void* o,
                          float* h_final, int B, int T, int N, int H, int HV, int D, int V, int pool_size,
                          int* dev_error, void* stream);

}  // namespace la_internal
