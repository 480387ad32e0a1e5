// la_prefill_api.cu -- host side of the C ABI declared in include/la_prefill.h:
// argument validation, TMA tensor-map construction and the kernel launches.
//
// Sequences of at most kShortMax tokens go to the tokenwise kernel (one state read and
// write and a few token updates), the others to the chunkwise kernel.  A fixed-length batch
// goes to one of the two; a packed batch, whose lengths only the device knows, launches both
// (each skips the other's units) when its average length is at most kSplitAvg tokens, and
// otherwise leaves every sequence to the chunkwise kernel rather than pay a second launch
// for the few short ones it may hold.
// Nothing here allocates device memory, reads device memory or synchronises with the
// host: a call only encodes three tensor maps on the host stack and enqueues one or two
// kernels on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "../../include/la_prefill.h"
#include "la_decode_kernels.cuh"
#include "la_host_common.h"
#include "la_prefill_internal.h"
#include "la_prefill_kernel.cuh"

namespace {

using la_host::fail;
using la_host::g_last_error;

// Per-device facts looked up once: SM count, and the kernel's shared-memory attribute set.
la_host::DeviceState g_dev[la_host::kMaxDevices];

int smem_bytes() { return static_cast<int>(sizeof(lap::SharedStorage)) + 1024; }

// Longest sequence the tokenwise kernel takes: up to four of its 8-token staging tiles.
constexpr int kShortMax = 32;
// Packed batches with at most this many tokens per sequence on average are split.
constexpr int kSplitAvg = 64;

cudaError_t setup_kernels() {
  const cudaFuncAttribute attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(lap::la_prefill_fwd_kernel<false, 128>, attr, smem_bytes());
  if (e == cudaSuccess) e = cudaFuncSetAttribute(lap::la_prefill_fwd_kernel<true, 128>, attr, smem_bytes());
  if (e == cudaSuccess) e = cudaFuncSetAttribute(lap::la_prefill_fwd_kernel<false, 64>, attr, smem_bytes());
  if (e == cudaSuccess) e = cudaFuncSetAttribute(lap::la_prefill_fwd_kernel<true, 64>, attr, smem_bytes());
  if (e == cudaSuccess) e = cudaFuncSetAttribute(lap::la_prefill_fwd_kernel<false, 128, true>, attr, smem_bytes());
  if (e == cudaSuccess) e = cudaFuncSetAttribute(lap::la_prefill_fwd_kernel<false, 64, true>, attr, smem_bytes());
  if (e == cudaSuccess) e = cudaFuncSetAttribute(lap::la_prefill_fwd_kernel<false, 128, false, true>, attr, smem_bytes());
  if (e == cudaSuccess) e = cudaFuncSetAttribute(lap::la_prefill_fwd_kernel<false, 128, true, true>, attr, smem_bytes());
  if (e == cudaSuccess) e = cudaFuncSetAttribute(lap::la_prefill_fwd_kernel<false, 64, false, true>, attr, smem_bytes());
  if (e == cudaSuccess) e = cudaFuncSetAttribute(lap::la_prefill_fwd_kernel<false, 64, true, true>, attr, smem_bytes());
  return e;
}

}  // namespace

extern "C" {

const char* la_status_string(la_status status) {
  switch (status) {
    case LA_OK: return "LA_OK";
    case LA_ERR_INVALID_ARGUMENT: return "LA_ERR_INVALID_ARGUMENT";
    case LA_ERR_UNSUPPORTED: return "LA_ERR_UNSUPPORTED";
    case LA_ERR_CUDA: return "LA_ERR_CUDA";
  }
  return "unknown la_status";
}

const char* la_last_error(void) { return g_last_error; }

int la_prefill_smem_bytes(void) { return smem_bytes(); }

la_status la_prefill_fwd(const void* q, const void* k, const void* v, const float* slopes, float scale,
                         const float* h0, const int32_t* state_indices, const int32_t* cu_seqlens, void* o,
                         float* h_final, int B, int T, int N, int H, int HV, int D, int V, int pool_size,
                         la_schedule schedule, int* dev_error, void* stream) {
  g_last_error[0] = '\0';
  if (schedule != LA_SCHED_AUTO && schedule != LA_SCHED_PERSISTENT && schedule != LA_SCHED_NON_PERSISTENT)
    return fail(LA_ERR_INVALID_ARGUMENT, "unknown schedule %d", (int)schedule);
  bool nothing = false;
  la_status st0 = la_host::check_prefill_args(q, k, v, slopes, h0, state_indices, cu_seqlens, o, h_final, B, T, N,
                                              H, HV, D, V, pool_size, dev_error, &nothing);
  if (st0 != LA_OK || nothing) return st0;
  st0 = la_host::check_prefill_disjoint(q, k, v, slopes, h0, state_indices, cu_seqlens, o, h_final, dev_error, B, T,
                                        N, H, HV, D, V, pool_size);
  if (st0 != LA_OK) return st0;
  const int64_t tokens = static_cast<int64_t>(B) * T;
  const int64_t units = static_cast<int64_t>(N) * HV;

  // ---- device
  la_host::DeviceState* dsp = nullptr;
  la_status dst = la_host::current_device(g_dev, &dsp, setup_kernels);
  if (dst != LA_OK) return dst;
  la_host::DeviceState& ds = *dsp;
  cudaError_t ce;

  // ---- tensor maps (unused when there are no tokens)
  CUtensorMap tm_q, tm_k, tm_v, tm_o;
  memset(&tm_q, 0, sizeof(tm_q));
  memset(&tm_k, 0, sizeof(tm_k));
  memset(&tm_v, 0, sizeof(tm_v));
  memset(&tm_o, 0, sizeof(tm_o));
  if (tokens > 0) {
    la_status st;
    if ((st = la_host::encode_bf16_rows_map(&tm_q, q, tokens, H, "q", D)) != LA_OK) return st;
    if ((st = la_host::encode_bf16_rows_map(&tm_k, k, tokens, H, "k", D)) != LA_OK) return st;
    if ((st = la_host::encode_bf16_rows_map(&tm_v, v, tokens, HV, "v", D)) != LA_OK) return st;
    if ((st = la_host::encode_bf16_out_map(&tm_o, o, tokens, HV, D)) != LA_OK) return st;
  }

  const bool packed = cu_seqlens != nullptr;
  const bool split = packed && tokens <= static_cast<int64_t>(kSplitAvg) * N;
  const bool run_tokenwise = split || (!packed && T <= kShortMax);
  const bool run_chunkwise = packed || T > kShortMax;
  const int pool = la_host::effective_pool_size(h0, h_final, state_indices, pool_size, N);
  if (run_tokenwise) {
    lad::Params tp{};
    tp.q = static_cast<const __nv_bfloat16*>(q);
    tp.k = static_cast<const __nv_bfloat16*>(k);
    tp.v = static_cast<const __nv_bfloat16*>(v);
    tp.slopes = slopes;
    tp.state_indices = state_indices;
    tp.o = static_cast<__nv_bfloat16*>(o);
    tp.h0 = h0;
    tp.h_final = h_final;
    tp.cu_seqlens = cu_seqlens;
    tp.dev_error = dev_error;
    tp.scale = scale;
    tp.B = N;
    tp.T = packed ? 0 : T;
    tp.H = H;
    tp.HV = HV;
    tp.G = HV / H;
    tp.pool_size = pool;
    tp.num_tokens = static_cast<int>(tokens);
    tp.short_max = kShortMax;
    const int64_t parts = units * (D == 128 ? lad::split_of<128>() : lad::split_of<64>());
    if (parts > INT32_MAX) return fail(LA_ERR_UNSUPPORTED, "N*HV too large (%lld)", (long long)units);
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    ce = D == 128 ? la_host::launch_pdl(lad::la_tokenwise_kernel<lad::kPrefill, 128>,
                                        lad::tokenwise_grid<128>(static_cast<int>(parts), ds.sms), lad::kThreads,
                                        lad::tokenwise_smem_bytes<128>(), cs, tp)
                  : la_host::launch_pdl(lad::la_tokenwise_kernel<lad::kPrefill, 64>,
                                        lad::tokenwise_grid<64>(static_cast<int>(parts), ds.sms), lad::kThreads,
                                        lad::tokenwise_smem_bytes<64>(), cs, tp);
    if (ce == cudaSuccess) ce = cudaGetLastError();
    if (ce != cudaSuccess) return fail(LA_ERR_CUDA, "tokenwise kernel launch failed: %s", cudaGetErrorString(ce));
  }
  if (!run_chunkwise) return LA_OK;

  lap::KernelParams p;
  p.slopes = slopes;
  p.h0 = h0;
  p.state_indices = state_indices;
  p.cu_seqlens = cu_seqlens;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.o_f32 = nullptr;
  p.h_final = h_final;
  p.dev_error = dev_error;
  p.scale = scale;
  p.num_tokens = static_cast<int>(tokens);
  p.T = cu_seqlens ? 0 : T;
  p.N = N;
  p.H = H;
  p.HV = HV;
  p.G = HV / H;
  p.vdiv = 1;
  p.vfold = 0;
  p.pool_size = pool;
  p.num_units = static_cast<int>(units);
  p.short_max = split ? kShortMax : -1;

  int grid = static_cast<int>(units);
  if (schedule != LA_SCHED_NON_PERSISTENT && grid > ds.sms) grid = ds.sms;
  // A packed batch of few sequences gets the longest-first schedule (the lengths vary, and a
  // CTA runs a handful of units); other batches deal units out round robin.
  const bool listed = packed && N <= lap::kSchedSeqMax && (units + grid - 1) / grid <= lap::kSchedMax;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  void (*kernel)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, lap::KernelParams) =
      D == 128 ? (listed ? lap::la_prefill_fwd_kernel<true, 128> : lap::la_prefill_fwd_kernel<false, 128>)
               : (listed ? lap::la_prefill_fwd_kernel<true, 64> : lap::la_prefill_fwd_kernel<false, 64>);
  ce = la_host::launch_pdl(kernel, grid, lap::kThreads, smem_bytes(), cs, tm_q, tm_k, tm_v, tm_o, p);
  if (ce == cudaSuccess) ce = cudaGetLastError();
  if (ce != cudaSuccess) return fail(LA_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(ce));
  return LA_OK;
}

}  // extern "C"

namespace la_internal {

la_status chunkwise(const void* q, const void* k, const void* v, const float* slopes, float scale, const float* h0,
                    const int32_t* state_indices, const int32_t* cu_seqlens, void* o, float* o_f32, float* h_final,
                    int B, int T, int N, int H, int HV, int v_heads, int D, int pool_size, bool reverse,
                    int* dev_error, void* stream, int v_fold, int short_max) {
  if (v_heads <= 0 || HV % v_heads != 0)
    return fail(LA_ERR_UNSUPPORTED, "HV (%d) must be a multiple of v's heads (%d)", HV, v_heads);
  if (v_fold < 0 || (v_fold > 0 && (!o_f32 || v_heads * 2 != HV || HV % (2 * v_fold) != 0)))
    return fail(LA_ERR_UNSUPPORTED, "bad value-head fold %d (HV %d, v heads %d)", v_fold, HV, v_heads);
  // the checks of la_prefill_fwd; o (or o_f32) has the layout of the output, h_final of the states
  bool nothing = false;
  la_status st = la_host::check_prefill_args(q, k, v, slopes, h0, state_indices, cu_seqlens,
                                             o_f32 ? static_cast<const void*>(o_f32) : o, h_final, B, T, N, H, HV, D,
                                             D, pool_size, dev_error, &nothing);
  if (st != LA_OK || nothing) return st;
  const int64_t tokens = static_cast<int64_t>(B) * T;
  const int64_t units = static_cast<int64_t>(N) * HV;
  la_host::DeviceState* dsp = nullptr;
  if ((st = la_host::current_device(g_dev, &dsp, setup_kernels)) != LA_OK) return st;
  CUtensorMap tm_q, tm_k, tm_v, tm_o;
  memset(&tm_q, 0, sizeof(tm_q));
  memset(&tm_k, 0, sizeof(tm_k));
  memset(&tm_v, 0, sizeof(tm_v));
  memset(&tm_o, 0, sizeof(tm_o));
  if (tokens > 0) {
    if ((st = la_host::encode_bf16_rows_map(&tm_q, q, tokens, H, "q", D)) != LA_OK) return st;
    if ((st = la_host::encode_bf16_rows_map(&tm_k, k, tokens, H, "k", D)) != LA_OK) return st;
    if ((st = la_host::encode_bf16_rows_map(&tm_v, v, tokens, v_heads, "v", D)) != LA_OK) return st;
    if (!o_f32 && (st = la_host::encode_bf16_out_map(&tm_o, o, tokens, HV, D)) != LA_OK) return st;
  }
  lap::KernelParams p;
  p.slopes = slopes;
  p.h0 = h0;
  p.state_indices = state_indices;
  p.cu_seqlens = cu_seqlens;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.o_f32 = o_f32;
  p.h_final = h_final;
  p.dev_error = dev_error;
  p.scale = scale;
  p.num_tokens = static_cast<int>(tokens);
  p.T = cu_seqlens ? 0 : T;
  p.N = N;
  p.H = H;
  p.HV = HV;
  p.G = HV / H;
  p.vdiv = HV / v_heads;
  p.vfold = v_fold;
  p.pool_size = la_host::effective_pool_size(h0, h_final, state_indices, pool_size, N);
  p.num_units = static_cast<int>(units);
  p.short_max = cu_seqlens ? short_max : -1;  // -1: every sequence, however short, runs here
  const int grid = static_cast<int>(units < dsp->sms ? units : dsp->sms);
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const int variant = (D == 128 ? 0 : 4) + (reverse ? 2 : 0) + (o_f32 ? 1 : 0);
  static void (*const kernels[8])(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, lap::KernelParams) = {
      lap::la_prefill_fwd_kernel<false, 128, false, false>, lap::la_prefill_fwd_kernel<false, 128, false, true>,
      lap::la_prefill_fwd_kernel<false, 128, true, false>,  lap::la_prefill_fwd_kernel<false, 128, true, true>,
      lap::la_prefill_fwd_kernel<false, 64, false, false>,  lap::la_prefill_fwd_kernel<false, 64, false, true>,
      lap::la_prefill_fwd_kernel<false, 64, true, false>,   lap::la_prefill_fwd_kernel<false, 64, true, true>};
  cudaError_t ce = la_host::launch_pdl(kernels[variant], grid, lap::kThreads, smem_bytes(), cs, tm_q, tm_k, tm_v,
                                       tm_o, p);
  if (ce == cudaSuccess) ce = cudaGetLastError();
  if (ce != cudaSuccess) return fail(LA_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(ce));
  return LA_OK;
}

}  // namespace la_internal
