// la_prefill_api.cu -- host side of the C ABI declared in include/la_prefill.h:
// argument validation, TMA tensor-map construction and the kernel launch.
//
// Nothing here allocates device memory, reads device memory or synchronises with
// the host: a call only encodes three tensor maps on the host stack and enqueues
// one kernel on the caller's stream.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/la_prefill.h"
#include "la_host_common.h"
#include "la_prefill_kernel.cuh"

namespace {

using la_host::aligned16;
using la_host::fail;
using la_host::g_last_error;

unsigned long long* g_trace = nullptr;  // device buffer for timeline tracing builds

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Per-device facts looked up once: SM count, and the kernel's shared-memory attribute set.
la_host::DeviceState g_dev[la_host::kMaxDevices];

int smem_bytes() { return static_cast<int>(sizeof(lap::SharedStorage)) + 1024; }

// Map over a [rows, heads * 128] BF16 matrix: 64 x 64 boxes, 128-byte swizzle.
la_status encode_map(CUtensorMap* map, const void* base, int64_t rows, int64_t heads, const char* name) {
  auto enc = tensor_map_encoder();
  if (!enc) return fail(LA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the CUDA driver");
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(heads * lap::kDim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(heads * lap::kDim * 2)};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r =
      enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(LA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name, (int)r);
  return LA_OK;
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

int la_prefill_trace_events(void) {
#ifdef LA_TRACE
  return lap::kTrEvents * lap::kTraceChunks;
#else
  return 0;
#endif
}

void la_prefill_set_trace_buffer(void* device_buffer) { g_trace = static_cast<unsigned long long*>(device_buffer); }

la_status la_prefill_fwd(const void* q, const void* k, const void* v, const float* slopes, float scale,
                         const float* h0, const int32_t* state_indices, const int32_t* cu_seqlens, void* o,
                         float* h_final, int B, int T, int N, int H, int HV, int D, int V, int pool_size,
                         la_schedule schedule, int* dev_error, void* stream) {
  g_last_error[0] = '\0';
  // ---- shapes
  if (D != lap::kDim || V != lap::kDim)
    return fail(LA_ERR_UNSUPPORTED, "only D == V == 128 is implemented (got D=%d, V=%d)", D, V);
  if (H <= 0 || HV <= 0) return fail(LA_ERR_INVALID_ARGUMENT, "H and HV must be positive (got %d, %d)", H, HV);
  if (HV % H != 0) return fail(LA_ERR_UNSUPPORTED, "HV (%d) must be a multiple of H (%d)", HV, H);
  if (B < 0 || T < 0 || N < 0) return fail(LA_ERR_INVALID_ARGUMENT, "B, T, N must be >= 0");
  if (schedule != LA_SCHED_AUTO && schedule != LA_SCHED_PERSISTENT && schedule != LA_SCHED_NON_PERSISTENT)
    return fail(LA_ERR_INVALID_ARGUMENT, "unknown schedule %d", (int)schedule);
  if (cu_seqlens) {
    if (B != 1) return fail(LA_ERR_INVALID_ARGUMENT, "packed mode (cu_seqlens given) needs B == 1 (got %d)", B);
  } else if (N != B) {
    return fail(LA_ERR_INVALID_ARGUMENT, "fixed-length mode needs N == B (got N=%d, B=%d)", N, B);
  }
  const int64_t tokens = static_cast<int64_t>(B) * T;
  if (tokens + lap::kChunk > INT32_MAX) return fail(LA_ERR_UNSUPPORTED, "B*T too large (%lld)", (long long)tokens);
  const int64_t units = static_cast<int64_t>(N) * HV;
  if (units > INT32_MAX) return fail(LA_ERR_UNSUPPORTED, "N*HV too large (%lld)", (long long)units);
  if (static_cast<int64_t>(HV) * lap::kDim * 2 > (int64_t(1) << 39))
    return fail(LA_ERR_UNSUPPORTED, "HV too large for a tensor map stride");
  if (N == 0) return LA_OK;
  // ---- pointers
  if (!slopes) return fail(LA_ERR_INVALID_ARGUMENT, "slopes is null");
  if (tokens > 0 && (!q || !k || !v || !o)) return fail(LA_ERR_INVALID_ARGUMENT, "q, k, v and o must be non-null");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(h0) || !aligned16(h_final))
    return fail(LA_ERR_INVALID_ARGUMENT, "q, k, v, o, h0 and h_final must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(slopes) & 3u) || (reinterpret_cast<uintptr_t>(dev_error) & 3u) ||
      (reinterpret_cast<uintptr_t>(state_indices) & 3u) || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
    return fail(LA_ERR_INVALID_ARGUMENT, "slopes, dev_error, state_indices, cu_seqlens must be 4-byte aligned");
  if (h0 || h_final) {
    if (state_indices) {
      if (pool_size <= 0) return fail(LA_ERR_INVALID_ARGUMENT, "pool_size must be positive with state_indices");
    } else if (pool_size < N) {
      return fail(LA_ERR_INVALID_ARGUMENT, "pool_size (%d) must be >= N (%d) without state_indices", pool_size, N);
    }
  }
  if (tokens == 0 && !h_final) return LA_OK;  // no output rows and no state to write

  // ---- device
  la_host::DeviceState* dsp = nullptr;
  la_status dst = la_host::current_device(g_dev, &dsp, [] {
    return cudaFuncSetAttribute(lap::la_prefill_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_bytes());
  });
  if (dst != LA_OK) return dst;
  la_host::DeviceState& ds = *dsp;
  cudaError_t ce;

  // ---- tensor maps (unused when there are no tokens)
  CUtensorMap tm_q, tm_k, tm_v;
  memset(&tm_q, 0, sizeof(tm_q));
  memset(&tm_k, 0, sizeof(tm_k));
  memset(&tm_v, 0, sizeof(tm_v));
  if (tokens > 0) {
    la_status st;
    if ((st = encode_map(&tm_q, q, tokens, H, "q")) != LA_OK) return st;
    if ((st = encode_map(&tm_k, k, tokens, H, "k")) != LA_OK) return st;
    if ((st = encode_map(&tm_v, v, tokens, HV, "v")) != LA_OK) return st;
  }

  lap::KernelParams p;
  p.slopes = slopes;
  p.h0 = h0;
  p.state_indices = state_indices;
  p.cu_seqlens = cu_seqlens;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.h_final = h_final;
  p.dev_error = dev_error;
  p.trace = g_trace;
  p.scale = scale;
  p.num_tokens = static_cast<int>(tokens);
  p.T = cu_seqlens ? 0 : T;
  p.N = N;
  p.H = H;
  p.HV = HV;
  p.G = HV / H;
  p.pool_size = (h0 || h_final) ? pool_size : (state_indices ? INT32_MAX : N);
  p.num_units = static_cast<int>(units);

  int grid = static_cast<int>(units);
  if (schedule != LA_SCHED_NON_PERSISTENT && grid > ds.sms) grid = ds.sms;
  lap::la_prefill_fwd_kernel<<<grid, lap::kThreads, smem_bytes(), static_cast<cudaStream_t>(stream)>>>(
      tm_q, tm_k, tm_v, p);
  ce = cudaGetLastError();
  if (ce != cudaSuccess) return fail(LA_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(ce));
  return LA_OK;
}

}  // extern "C"
