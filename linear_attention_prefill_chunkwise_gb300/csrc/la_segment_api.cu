// la_segment_api.cu -- host side of the C ABI declared in include/la_segment.h: the choice
// of the segment length, the workspace layout and the launches of the segmented prefill
// (plan, local states, combine, chunkwise prefill over the segments, final-state copy).
//
// Nothing here allocates device memory, reads device memory or synchronises with the host.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "../../include/la_segment.h"
#include "la_host_common.h"
#include "la_prefill_internal.h"
#include "la_segment_kernels.cuh"

namespace {

using la_host::fail;

la_host::DeviceState g_dev[la_host::kMaxDevices];

int state_smem_bytes() { return static_cast<int>(sizeof(las::StateSmem)) + 1024; }

// The workspace is sized for D = V = 128 states whatever D is (the size query takes no D); a
// D = 64 call keeps its [nseg, HV, 64, 64] states in the first quarter of that region.
constexpr int kWsDim = 128;

constexpr size_t kWsAlign = 256;
size_t align_up(size_t x) { return (x + kWsAlign - 1) & ~(kWsAlign - 1); }

// Segment length and workspace layout of one call.
struct SegPlan {
  int S = 0;             // 0: no segmentation (la_prefill_fwd runs unchanged)
  int S_last = 0;        // > 0: each sequence's last segment is its last S_last tokens (plan kernel)
  int64_t nseg_max = 0;  // upper bound of the segment count
  size_t off_states = 0, off_seg_cu = 0, off_seg_slot = 0, off_seg_flags = 0, off_seq_seg0 = 0, off_seq_slot = 0;
  size_t bytes = 0;
};

la_status make_plan(int B, int T, int N, int HV, bool packed, int segment_len, int sms, SegPlan* out) {
  *out = SegPlan{};
  if (B < 0 || T < 0 || N < 0 || HV <= 0) return fail(LA_ERR_INVALID_ARGUMENT, "B, T, N >= 0 and HV > 0 required");
  if (segment_len < 0 || segment_len % las::kChunk != 0)
    return fail(LA_ERR_INVALID_ARGUMENT, "segment_len must be 0 (automatic) or a positive multiple of 64 (got %d)",
                segment_len);
  if (packed && B != 1) return fail(LA_ERR_INVALID_ARGUMENT, "packed mode needs B == 1 (got %d)", B);
  if (!packed && N != B) return fail(LA_ERR_INVALID_ARGUMENT, "fixed-length mode needs N == B (got N=%d, B=%d)", N, B);
  const int64_t tokens = static_cast<int64_t>(B) * T;
  const int64_t units = static_cast<int64_t>(N) * HV;
  if (N == 0 || tokens == 0) return LA_OK;
  int64_t S = segment_len, S_last = 0;
  if (S == 0) {
    // Segment only when the chains fill at most half of the SMs, and then aim at about one
    // segment per SM: the extra pass over K and V costs more than a nearly full GPU gains.
    if (units * 2 > sms) return LA_OK;
    if (!packed) {
      const int64_t m = sms / units;  // segments per sequence
      S = (T + m - 1) / m;
      // Two segments per sequence leave the local-state pass (one unit per sequence and head)
      // on at most half of the SMs: cut the first segment in two instead, so that twice as many
      // shorter local states run in parallel, and keep the last segment, which needs none, at
      // full length (the prefill's longest unit, and so its time, is unchanged).
      if (m == 2 && T >= 4 * las::kChunk) {
        S_last = (S + las::kChunk - 1) / las::kChunk * las::kChunk;
        S = ((T - S_last + 1) / 2 + las::kChunk - 1) / las::kChunk * las::kChunk;
      }
    } else {
      S = (tokens * HV + sms - 1) / sms;
    }
    S = (S + las::kChunk - 1) / las::kChunk * las::kChunk;
    if (S < las::kChunk) S = las::kChunk;
  }
  // no sequence is longer than one segment: nothing to gain
  if ((!packed && S >= T) || (packed && S >= tokens)) return LA_OK;
  const int64_t nseg = packed ? N + tokens / S
                              : static_cast<int64_t>(B) *
                                    (S_last > 0 ? ((T > S_last ? T - S_last : 0) + S - 1) / S + 1 : (T + S - 1) / S);
  if (nseg >= INT32_MAX || nseg * HV > INT32_MAX)
    return fail(LA_ERR_UNSUPPORTED, "too many segments (%lld x %d heads); use a longer segment_len", (long long)nseg,
                HV);
  SegPlan p;
  p.S = static_cast<int>(S);
  p.S_last = static_cast<int>(S_last);
  p.nseg_max = nseg;
  size_t off = 0;
  p.off_states = off;
  off = align_up(off + static_cast<size_t>(nseg) * HV * kWsDim * kWsDim * sizeof(float));
  p.off_seg_cu = off;
  off = align_up(off + static_cast<size_t>(nseg + 1) * sizeof(int32_t));
  p.off_seg_slot = off;
  off = align_up(off + static_cast<size_t>(nseg) * sizeof(int32_t));
  p.off_seg_flags = off;
  off = align_up(off + static_cast<size_t>(nseg) * sizeof(int32_t));
  p.off_seq_seg0 = off;
  off = align_up(off + static_cast<size_t>(N + 1) * sizeof(int32_t));
  p.off_seq_slot = off;
  off = align_up(off + static_cast<size_t>(N) * sizeof(int32_t));
  p.bytes = off;
  *out = p;
  return LA_OK;
}

la_status segment_device(la_host::DeviceState** ds) {
  return la_host::current_device(g_dev, ds, [] {
    cudaError_t e = cudaFuncSetAttribute(las::la_segment_state_kernel<128>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, state_smem_bytes());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(las::la_segment_state_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               state_smem_bytes());
    return e;
  });
}

// The status of a launch: the launch call's own result, else any earlier error it left pending.
la_status launched(const char* what, cudaError_t launch_result = cudaSuccess) {
  const cudaError_t ce = launch_result != cudaSuccess ? launch_result : cudaGetLastError();
  if (ce != cudaSuccess) return fail(LA_ERR_CUDA, "%s launch failed: %s", what, cudaGetErrorString(ce));
  return LA_OK;
}

// Steps 1-5 of a segmented call on validated arguments and a workspace of at least pl.bytes.
// With o_f32 (the D = 256 decomposition) the output is FP32 parts, and v is read through the
// value-head fold vfold (v then has HV / 2 heads).
la_status seg_launch(const SegPlan& pl, la_host::DeviceState* ds, const void* q, const void* k, const void* v,
                     const float* slopes, float scale, const float* h0, const int32_t* state_indices,
                     const int32_t* cu_seqlens, void* o, float* o_f32, float* h_final, int B, int T, int N, int H,
                     int HV, int D, int V, int pool_size, void* workspace, int* dev_error, void* stream, int vfold) {
  la_status st;
  const int64_t tokens = static_cast<int64_t>(B) * T;
  const int nseg = static_cast<int>(pl.nseg_max);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* states = reinterpret_cast<float*>(ws + pl.off_states);
  int32_t* seg_cu = reinterpret_cast<int32_t*>(ws + pl.off_seg_cu);
  int32_t* seg_slot = reinterpret_cast<int32_t*>(ws + pl.off_seg_slot);
  int32_t* seg_flags = reinterpret_cast<int32_t*>(ws + pl.off_seg_flags);
  int32_t* seq_seg0 = reinterpret_cast<int32_t*>(ws + pl.off_seq_seg0);
  int32_t* seq_slot = reinterpret_cast<int32_t*>(ws + pl.off_seq_slot);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  CUtensorMap tm_k, tm_v;
  memset(&tm_k, 0, sizeof(tm_k));
  memset(&tm_v, 0, sizeof(tm_v));
  if ((st = la_host::encode_bf16_rows_map(&tm_k, k, tokens, H, "k", D)) != LA_OK) return st;
  if ((st = la_host::encode_bf16_rows_map(&tm_v, v, tokens, vfold ? HV / 2 : HV, "v", D)) != LA_OK) return st;

  // 1. segment table
  las::PlanParams pp;
  pp.cu_seqlens = cu_seqlens;
  pp.state_indices = state_indices;
  pp.dev_error = dev_error;
  pp.seg_cu = seg_cu;
  pp.seg_slot = seg_slot;
  pp.seg_flags = seg_flags;
  pp.seq_seg0 = seq_seg0;
  pp.seq_slot = seq_slot;
  pp.N = N;
  pp.T = cu_seqlens ? 0 : T;
  pp.tokens = static_cast<int>(tokens);
  pp.S = pl.S;
  pp.S_last = pl.S_last;
  pp.nseg_max = nseg;
  pp.pool_size = la_host::effective_pool_size(h0, h_final, state_indices, pool_size, N);
  if ((st = launched("segment plan", la_host::launch_pdl(las::la_segment_plan_kernel, 1, las::kPlanThreads, 0, s,
                                                         pp))) != LA_OK)
    return st;

  // 2. local states of the segments that are not the last of their sequence
  las::StateParams sp;
  sp.slopes = slopes;
  sp.seg_cu = seg_cu;
  sp.seg_flags = seg_flags;
  sp.states = states;
  sp.dev_error = dev_error;
  sp.HV = HV;
  sp.G = HV / H;
  sp.num_units = nseg * HV;
  sp.vfold = vfold;
  const int grid_a = sp.num_units < ds->sms ? sp.num_units : ds->sms;
  if ((st = launched("segment state",
                     la_host::launch_pdl(D == 128 ? las::la_segment_state_kernel<128> : las::la_segment_state_kernel<64>,
                                         grid_a, las::kStThreads, state_smem_bytes(), s, tm_k, tm_v, sp))) != LA_OK)
    return st;

  // 3. initial state of every segment
  las::CombineParams cp;
  cp.slopes = slopes;
  cp.h0 = h0;
  cp.h_final = h_final;
  cp.seg_cu = seg_cu;
  cp.seq_seg0 = seq_seg0;
  cp.seq_slot = seq_slot;
  cp.states = states;
  cp.HV = HV;
  const dim3 grid_c(static_cast<unsigned>(N) * HV, D == 128 ? las::comb_split<128>() : las::comb_split<64>());
  if ((st = launched("segment combine",
                     la_host::launch_pdl(D == 128 ? las::la_segment_combine_kernel<128> : las::la_segment_combine_kernel<64>,
                                         grid_c, las::kCombThreads, 0, s, cp))) != LA_OK)
    return st;

  // 4. the chunkwise prefill of every segment: a packed batch whose state pool is the
  //    workspace (segment g reads its initial state from slot g and leaves its final one there)
  if (o_f32)
    st = la_internal::chunkwise(q, k, v, slopes, scale, states, seg_slot, seg_cu, nullptr, o_f32,
                                h_final ? states : nullptr, 1, static_cast<int>(tokens), nseg, H, HV, HV / 2, D, nseg,
                                false, dev_error, stream, vfold);
  else
    st = la_prefill_fwd(q, k, v, slopes, scale, states, seg_slot, seg_cu, o, h_final ? states : nullptr, 1,
                        static_cast<int>(tokens), nseg, H, HV, D, V, nseg, LA_SCHED_AUTO, dev_error, stream);
  if (st != LA_OK) return st;

  // 5. final states
  if (h_final) {
    if ((st = launched("segment final",
                       la_host::launch_pdl(D == 128 ? las::la_segment_final_kernel<128> : las::la_segment_final_kernel<64>,
                                           grid_c, las::kCombThreads, 0, s, cp))) != LA_OK)
      return st;
  }
  return LA_OK;
}

}  // namespace

extern "C" {

la_status la_prefill_segmented_workspace(int B, int T, int N, int HV, int packed, int segment_len, size_t* bytes,
                                         int* resolved_segment_len) {
  la_host::g_last_error[0] = '\0';
  if (!bytes) return fail(LA_ERR_INVALID_ARGUMENT, "bytes is null");
  int sms = 0;
  if (segment_len == 0) {
    la_host::DeviceState* ds = nullptr;
    const la_status st = segment_device(&ds);
    if (st != LA_OK) return st;
    sms = ds->sms;
  }
  SegPlan pl;
  const la_status st = make_plan(B, T, N, HV, packed != 0, segment_len, sms, &pl);
  if (st != LA_OK) return st;
  *bytes = pl.bytes;
  if (resolved_segment_len) *resolved_segment_len = pl.S;
  return LA_OK;
}

la_status la_prefill_fwd_segmented(const void* q, const void* k, const void* v, const float* slopes, float scale,
                                   const float* h0, const int32_t* state_indices, const int32_t* cu_seqlens,
                                   void* o, float* h_final, int B, int T, int N, int H, int HV, int D, int V,
                                   int pool_size, int segment_len, void* workspace, size_t workspace_bytes,
                                   int* dev_error, void* stream) {
  la_host::g_last_error[0] = '\0';
  bool nothing = false;
  la_status st = la_host::check_prefill_args(q, k, v, slopes, h0, state_indices, cu_seqlens, o, h_final, B, T, N, H,
                                             HV, D, V, pool_size, dev_error, &nothing);
  if (st != LA_OK || nothing) return st;
  // An explicit segment length fixes the plan without the device: the workspace is checked
  // before any device state is touched.
  la_host::DeviceState* ds = nullptr;
  int sms = 0;
  if (segment_len == 0) {
    if ((st = segment_device(&ds)) != LA_OK) return st;
    sms = ds->sms;
  }
  SegPlan pl;
  if ((st = make_plan(B, T, N, HV, cu_seqlens != nullptr, segment_len, sms, &pl)) != LA_OK) return st;
  if (pl.S == 0)
    return la_prefill_fwd(q, k, v, slopes, scale, h0, state_indices, cu_seqlens, o, h_final, B, T, N, H, HV, D, V,
                          pool_size, LA_SCHED_AUTO, dev_error, stream);
  if (!workspace || workspace_bytes < pl.bytes)
    return fail(LA_ERR_INVALID_ARGUMENT, "workspace too small: %zu bytes given, %zu needed", workspace_bytes,
                pl.bytes);
  if (reinterpret_cast<uintptr_t>(workspace) % kWsAlign)
    return fail(LA_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
  st = la_host::check_prefill_disjoint(q, k, v, slopes, h0, state_indices, cu_seqlens, o, h_final, dev_error, B, T, N,
                                       H, HV, D, V, pool_size, workspace, pl.bytes);
  if (st != LA_OK) return st;
  if (!ds && (st = segment_device(&ds)) != LA_OK) return st;

  return seg_launch(pl, ds, q, k, v, slopes, scale, h0, state_indices, cu_seqlens, o, nullptr, h_final, B, T, N, H,
                    HV, D, V, pool_size, workspace, dev_error, stream, 0);
}

}  // extern "C"

namespace la_internal {

la_status segmented_f32(const void* q, const void* k, const void* v, const float* slopes, float scale, const float* h0,
                        const int32_t* state_indices, const int32_t* cu_seqlens, float* o_f32, float* h_final, int B,
                        int T, int N, int H, int HV, int D, int pool_size, int segment_len, void* workspace,
                        size_t workspace_bytes, int* dev_error, void* stream, int vfold) {
  la_host::DeviceState* ds = nullptr;
  la_status st = segment_device(&ds);
  if (st != LA_OK) return st;
  SegPlan pl;
  if ((st = make_plan(B, T, N, HV, cu_seqlens != nullptr, segment_len, ds->sms, &pl)) != LA_OK) return st;
  if (pl.S == 0)
    return chunkwise(q, k, v, slopes, scale, h0, state_indices, cu_seqlens, nullptr, o_f32, h_final, B, T, N, H, HV,
                     HV / 2, D, pool_size, false, dev_error, stream, vfold);
  if (!workspace || workspace_bytes < pl.bytes)
    return fail(LA_ERR_INVALID_ARGUMENT, "segment workspace too small: %zu bytes given, %zu needed", workspace_bytes,
                pl.bytes);
  if (reinterpret_cast<uintptr_t>(workspace) % kWsAlign)
    return fail(LA_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
  return seg_launch(pl, ds, q, k, v, slopes, scale, h0, state_indices, cu_seqlens, nullptr, o_f32, h_final, B, T, N, H,
                    HV, D, D, pool_size, workspace, dev_error, stream, vfold);
}

}  // namespace la_internal
