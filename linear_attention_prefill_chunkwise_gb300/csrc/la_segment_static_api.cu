// la_segment_static_api.cu -- la_prefill_fwd_segmented_static (include/la_segment.h): the
// segmented prefill with its scratch memory in a buffer built into the library, for callers
// that cannot allocate device memory themselves.
//
// The buffer is a file-scope __device__ array, so the CUDA runtime sets it aside when it loads
// this file's module on a device (with lazy module loading, at the first call here; with eager
// loading, when the context is created) and keeps it until the process exits.  Host code cannot
// use the array's name as a device address; the address is looked up once per device with
// cudaGetSymbolAddress and handed to la_prefill_fwd_segmented as its workspace.  No call here
// allocates device memory.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/la_segment.h"
#include "la_host_common.h"

namespace {

using la_host::fail;

// 16 MiB: 256 FP32 [128 x 128] (segment, value head) states, less the plan's small tables.
// Every automatic segment length on a 152-SM GPU needs at most 228 states.
constexpr size_t kScratchBytes = size_t(16) << 20;

static __device__ __align__(256) uint8_t g_segment_scratch[kScratchBytes];

la_host::DeviceState g_dev[la_host::kMaxDevices];
void* g_scratch_ptr[la_host::kMaxDevices];

// Address of this device's copy of the buffer, looked up on the first call per device.
la_status scratch_for_current_device(void** out) {
  int dev = 0;
  la_host::DeviceState* ds = nullptr;
  const la_status st = la_host::current_device(g_dev, &ds, [] {
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess) return e;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_segment_scratch);
    if (e == cudaSuccess) g_scratch_ptr[d] = p;
    return e;
  });
  if (st != LA_OK) return st;
  const cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return fail(LA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(ce));
  if (!g_scratch_ptr[dev]) return fail(LA_ERR_CUDA, "built-in scratch buffer unavailable on device %d", dev);
  *out = g_scratch_ptr[dev];
  return LA_OK;
}

}  // namespace

extern "C" {

la_status la_prefill_fwd_segmented_static(const void* q, const void* k, const void* v, const float* slopes,
                                          float scale, const float* h0, const int32_t* state_indices,
                                          const int32_t* cu_seqlens, void* o, float* h_final, int B, int T, int N,
                                          int H, int HV, int D, int V, int pool_size, int segment_len,
                                          int* dev_error, void* stream) {
  la_host::g_last_error[0] = '\0';
  // The arguments first, so that an invalid call is reported as such whatever its size.
  bool nothing = false;
  la_status st = la_host::check_prefill_args(q, k, v, slopes, h0, state_indices, cu_seqlens, o, h_final, B, T, N, H,
                                             HV, D, V, pool_size, dev_error, &nothing);
  if (st != LA_OK || nothing) return st;
  size_t need = 0;
  st = la_prefill_segmented_workspace(B, T, N, HV, cu_seqlens != nullptr, segment_len, &need, nullptr);
  if (st != LA_OK) return st;
  if (need > kScratchBytes)
    return fail(LA_ERR_UNSUPPORTED,
                "this call needs %zu bytes of scratch and the built-in buffer holds %zu; pass a longer "
                "segment_len, or call la_prefill_fwd_segmented with a workspace of your own",
                need, kScratchBytes);
  void* scratch = nullptr;
  if (need > 0 && (st = scratch_for_current_device(&scratch)) != LA_OK) return st;
  return la_prefill_fwd_segmented(q, k, v, slopes, scale, h0, state_indices, cu_seqlens, o, h_final, B, T, N, H, HV,
                                  D, V, pool_size, segment_len, scratch, need > 0 ? kScratchBytes : 0, dev_error,
                                  stream);
}

}  // extern "C"
