// la_prefill_internal.h -- entry points shared between the library's translation units, not part
// of the C ABI.
#pragma once

#include <cuda_bf16.h>

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
// into `o_f32` when that is not null (same [tokens, HV, D] layout).  With v_fold > 0 (FP32 output
// only, v_heads = HV / 2) head h reads v's head (h / (2 v_fold)) v_fold + h % v_fold instead: the
// digit of weight v_fold of h is dropped (the D = 256 decomposition, where it selects a half of
// the key dimension).  short_max >= 0 (packed batches) leaves the sequences of at most that many
// tokens to another kernel.  Arguments, layouts and checks otherwise as la_prefill_fwd (D == V).
// Used by the backward pass and by the D = 256 prefill.
la_status chunkwise(const void* q, const void* k, const void* v, const float* slopes, float scale, const float* h0,
                    const int32_t* state_indices, const int32_t* cu_seqlens, void* o, float* o_f32, float* h_final,
                    int B, int T, int N, int H, int HV, int v_heads, int D, int pool_size, bool reverse,
                    int* dev_error, void* stream, int v_fold = 0, int short_max = -1);

// The segmented prefill (include/la_segment.h) with FP32 output parts and the value-head fold
// vfold (v with HV / 2 heads), on arguments the caller has checked: the D = 256 prefill's view
// of its problem.  The workspace is la_prefill_segmented_workspace(B, T, N, HV, ...) bytes; a
// plan without segments runs chunkwise() directly and needs none.
la_status segmented_f32(const void* q, const void* k, const void* v, const float* slopes, float scale, const float* h0,
                        const int32_t* state_indices, const int32_t* cu_seqlens, float* o_f32, float* h_final, int B,
                        int T, int N, int H, int HV, int D, int pool_size, int segment_len, void* workspace,
                        size_t workspace_bytes, int* dev_error, void* stream, int vfold);


// The sequence of token row r (fixed length T, or the packed bounds cu_seqlens), or -1 when the
// row belongs to no sequence that the chunkwise runs computed (bad bounds, a padded or invalid
// state index).
__device__ __forceinline__ int row_sequence(const int32_t* cu, const int32_t* state_indices, int N, int T, int tokens,
                                            int pool, int r) {
  int n;
  if (!cu) {
    n = r / T;
  } else {
    int lo = 0, hi = N - 1;  // the last n with cu[n] <= r
    if (N <= 0 || __ldg(cu) > r) return -1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(cu + mid) <= r) lo = mid;
      else hi = mid - 1;
    }
    n = lo;
    const int b = __ldg(cu + n), e = __ldg(cu + n + 1);
    if (b < 0 || e < b || e > tokens || r >= e) return -1;
  }
  if (state_indices) {
    const int slot = __ldg(state_indices + n);
    if (slot < 0 || slot >= pool) return -1;
  }
  return n;
}

// Two FP32 values rounded to BF16 (nearest even), the first in the low half.
__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

}  // namespace la_internal
