// la_host_common.h -- host-side helpers shared by the C-ABI translation units: the
// per-thread last-error text, argument checks and the one-time per-device lookup.
#pragma once

#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

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

}  // namespace la_host
