// la_host_common.h -- host-side helpers shared by the C-ABI translation units: the
// per-thread last-error text, argument checks, the one-time per-device lookup and the
// TMA tensor maps over the token-major BF16 inputs.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <utility>

#include "../../include/la_prefill.h"

namespace la_host {

// Text of the last error of this thread's calls (la_last_error).
inline thread_local char g_last_error[512] = "";

inline la_status fail(la_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

inline bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }
inline bool aligned4(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; }

// A launch with programmatic stream serialization: the grid may be placed on the GPU while the
// previous kernel in the stream is still finishing, which hides the launch gap between
// back-to-back calls.  Every kernel launched this way starts with griddepcontrol.wait, so none
// of its memory accesses happens before that previous kernel has completed.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 threads, int smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = threads;
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// A caller's buffer as a byte range (a null pointer or an empty range holds no byte).
struct Span {
  const void* p;
  uint64_t bytes;
  const char* name;
};

// Outputs may share no byte with an input or with another output: the kernels read their
// inputs ahead of their stores and write their states after their last read, so an overlap
// is a race, not an in-place update.  A buffer that a call updates in place (the state pool)
// is listed once, as an output.  Only addresses are compared; nothing is read.
inline la_status check_disjoint(const Span* outs, int n_out, const Span* ins, int n_in) {
  auto meet = [](const Span& a, const Span& b) {
    if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
    const uint64_t x = reinterpret_cast<uintptr_t>(a.p), y = reinterpret_cast<uintptr_t>(b.p);
    return x < y + b.bytes && y < x + a.bytes;
  };
  for (int i = 0; i < n_out; ++i) {
    for (int j = 0; j < n_in; ++j)
      if (meet(outs[i], ins[j]))
        return fail(LA_ERR_INVALID_ARGUMENT, "%s overlaps %s (an output may share no memory with an input)",
                    outs[i].name, ins[j].name);
    for (int j = 0; j < i; ++j)
      if (meet(outs[i], outs[j]))
        return fail(LA_ERR_INVALID_ARGUMENT, "%s overlaps %s (outputs may share no memory)", outs[i].name,
                    outs[j].name);
  }
  return LA_OK;
}

// The buffers of a prefill call (la_prefill_fwd and the segmented entry points): q, k, v,
// slopes, h0, state_indices and cu_seqlens are read; o, h_final and dev_error are written;
// h_final may be h0 itself (an in-place pool), which then counts as an output only.
inline la_status check_prefill_disjoint(const void* q, const void* k, const void* v, const float* slopes,
                                        const float* h0, const int32_t* state_indices, const int32_t* cu_seqlens,
                                        const void* o, const float* h_final, const int* dev_error, int B, int T,
                                        int N, int H, int HV, int D, int V, int pool_size,
                                        const void* workspace = nullptr, uint64_t workspace_bytes = 0) {
  const uint64_t tokens = static_cast<uint64_t>(B) * static_cast<uint64_t>(T);
  const uint64_t bq = tokens * H * D * 2, bv = tokens * HV * V * 2;
  const uint64_t slots = state_indices ? static_cast<uint64_t>(pool_size) : static_cast<uint64_t>(N);
  const uint64_t bst = slots * HV * static_cast<uint64_t>(V) * D * 4;
  const Span ins[] = {{q, bq, "q"},
                      {k, bq, "k"},
                      {v, bv, "v"},
                      {slopes, static_cast<uint64_t>(HV) * 4, "slopes"},
                      {h0 == h_final ? nullptr : h0, bst, "h0"},
                      {state_indices, static_cast<uint64_t>(N) * 4, "state_indices"},
                      {cu_seqlens, cu_seqlens ? static_cast<uint64_t>(N + 1) * 4 : 0, "cu_seqlens"}};
  const Span outs[] = {{o, bv, "o"}, {h_final, bst, "h_final"}, {dev_error, 4, "dev_error"},
                       {workspace, workspace_bytes, "workspace"}};
  return check_disjoint(outs, 4, ins, 7);
}

// SM count and compute capability of the current device, looked up once per device, plus
// an optional one-time setup step (a kernel attribute) run with it.
constexpr int kMaxDevices = 64;
struct DeviceState {
  std::once_flag once;
  cudaError_t status = cudaSuccess;
  int sms = 0;
  int cc_major = 0, cc_minor = 0;
};

// Fills *ds for the current device (running setup() once per device on first use) and
// checks that it is an sm_103 part.
template <typename Setup>
la_status current_device(DeviceState (&table)[kMaxDevices], DeviceState** out, Setup setup) {
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return fail(LA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(ce));
  if (dev < 0 || dev >= kMaxDevices) return fail(LA_ERR_CUDA, "device ordinal %d out of range", dev);
  DeviceState& ds = table[dev];
  std::call_once(ds.once, [&ds, dev, &setup] {
    cudaError_t e = cudaDeviceGetAttribute(&ds.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&ds.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&ds.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = setup();
    ds.status = e;
  });
  if (ds.status != cudaSuccess)
    return fail(LA_ERR_CUDA, "device %d setup failed: %s", dev, cudaGetErrorString(ds.status));
  if (ds.cc_major != 10 || ds.cc_minor != 3)
    return fail(LA_ERR_CUDA, "device %d is sm_%d%d; this library is built for sm_103a only", dev, ds.cc_major,
                ds.cc_minor);
  *out = &ds;
  return LA_OK;
}

// cuTensorMapEncodeTiled, fetched once through the runtime's driver entry-point query (so the
// library has no link-time dependency on the driver library).
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// Map over a token-major [rows, heads * dim] BF16 matrix (dim = 64 or 128): 64 x 64 boxes (64
// tokens x 64 dims, 128-byte rows), 128-byte swizzle, the layout the kernels' MMA descriptors
// expect.
inline la_status encode_bf16_rows_map(CUtensorMap* map, const void* base, int64_t rows, int64_t heads,
                                      const char* name, int64_t dim = 128) {
  auto enc = tensor_map_encoder();
  if (!enc) return fail(LA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the CUDA driver");
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(heads * dim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(heads * dim * 2)};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r =
      enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(LA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name, (int)r);
  return LA_OK;
}

// Map over the token-major [rows, heads * dim] BF16 output for the epilogue's stores: 32 x 32
// boxes (32 tokens x 32 values, 64-byte rows), 64-byte swizzle.
inline la_status encode_bf16_out_map(CUtensorMap* map, void* base, int64_t rows, int64_t heads, int64_t dim) {
  auto enc = tensor_map_encoder();
  if (!enc) return fail(LA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the CUDA driver");
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(heads * dim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(heads * dim * 2)};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, elem_strides,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(LA_ERR_CUDA, "cuTensorMapEncodeTiled(o) failed with CUresult %d", (int)r);
  return LA_OK;
}

// Argument checks of a prefill call (la_prefill_fwd's contract): shapes, modes, pointers,
// alignment and the state pool.  Sets *nothing_to_do when the call has no work.
inline la_status check_prefill_args(const void* q, const void* k, const void* v, const float* slopes,
                                    const float* h0, const int32_t* state_indices, const int32_t* cu_seqlens,
                                    const void* o, const float* h_final, int B, int T, int N, int H, int HV, int D,
                                    int V, int pool_size, const int* dev_error, bool* nothing_to_do) {
  *nothing_to_do = false;
  if (D != V || (D != 128 && D != 64))
    return fail(LA_ERR_UNSUPPORTED, "only D == V == 128 and D == V == 64 are implemented (got D=%d, V=%d)", D, V);
  if (H <= 0 || HV <= 0) return fail(LA_ERR_INVALID_ARGUMENT, "H and HV must be positive (got %d, %d)", H, HV);
  if (HV % H != 0) return fail(LA_ERR_UNSUPPORTED, "HV (%d) must be a multiple of H (%d)", HV, H);
  if (B < 0 || T < 0 || N < 0) return fail(LA_ERR_INVALID_ARGUMENT, "B, T, N must be >= 0");
  if (cu_seqlens) {
    if (B != 1) return fail(LA_ERR_INVALID_ARGUMENT, "packed mode (cu_seqlens given) needs B == 1 (got %d)", B);
  } else if (N != B) {
    return fail(LA_ERR_INVALID_ARGUMENT, "fixed-length mode needs N == B (got N=%d, B=%d)", N, B);
  }
  const int64_t tokens = static_cast<int64_t>(B) * T;
  if (tokens + 64 > INT32_MAX) return fail(LA_ERR_UNSUPPORTED, "B*T too large (%lld)", (long long)tokens);
  const int64_t units = static_cast<int64_t>(N) * HV;
  if (units > INT32_MAX) return fail(LA_ERR_UNSUPPORTED, "N*HV too large (%lld)", (long long)units);
  if (static_cast<int64_t>(HV) * D * 2 > (int64_t(1) << 39))
    return fail(LA_ERR_UNSUPPORTED, "HV too large for a tensor map stride");
  if (N == 0) {
    *nothing_to_do = true;
    return LA_OK;
  }
  if (!slopes) return fail(LA_ERR_INVALID_ARGUMENT, "slopes is null");
  if (tokens > 0 && (!q || !k || !v || !o)) return fail(LA_ERR_INVALID_ARGUMENT, "q, k, v and o must be non-null");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(h0) || !aligned16(h_final))
    return fail(LA_ERR_INVALID_ARGUMENT, "q, k, v, o, h0 and h_final must be 16-byte aligned");
  if (!aligned4(slopes) || !aligned4(dev_error) || !aligned4(state_indices) || !aligned4(cu_seqlens))
    return fail(LA_ERR_INVALID_ARGUMENT, "slopes, dev_error, state_indices, cu_seqlens must be 4-byte aligned");
  if (h0 || h_final) {
    if (state_indices) {
      if (pool_size <= 0) return fail(LA_ERR_INVALID_ARGUMENT, "pool_size must be positive with state_indices");
    } else if (pool_size < N) {
      return fail(LA_ERR_INVALID_ARGUMENT, "pool_size (%d) must be >= N (%d) without state_indices", pool_size, N);
    }
  }
  if (tokens == 0 && !h_final) *nothing_to_do = true;  // no output rows and no state to write
  return LA_OK;
}

// The pool size the kernels check state indices against: the caller's when a state buffer
// is given, otherwise no bound (indices then only select which sequences run).
inline int effective_pool_size(const float* h0, const float* h_final, const int32_t* state_indices, int pool_size,
                               int N) {
  return (h0 || h_final) ? pool_size : (state_indices ? INT32_MAX : N);
}

}  // namespace la_host
