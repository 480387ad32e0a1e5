// la_decode_api.cu -- host side of the C ABI declared in include/la_decode.h: argument
// validation and one launch per call: the tokenwise kernel (D / 64 CTAs per (request, value
// head)) for decode, commit and long verifies, the tensor-core closed-form kernel for verifies
// of at most lav::kMaxTok tokens at D = 128.  Nothing here allocates device memory, reads device
// memory or synchronises with the host.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/la_decode.h"
#include "la_decode_kernels.cuh"
#include "la_host_common.h"
#include "la_verify_kernel.cuh"

namespace {

using la_host::aligned16;
using la_host::aligned4;
using la_host::fail;

la_host::DeviceState g_dev[la_host::kMaxDevices];

// Map over a pool of FP32 states viewed as [rows, 128] (rows = slots x heads x 128 value rows):
// 32 x 128 boxes (32 columns = 128 bytes, 128 rows), 128-byte swizzle, the K-major operand
// layout of a TF32 tensor-core product.
la_status encode_f32_state_map(CUtensorMap* map, const void* base, int64_t rows) {
  auto enc = la_host::tensor_map_encoder();
  if (!enc) return fail(LA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the CUDA driver");
  const cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {128 * 4};
  const cuuint32_t box[2] = {32, 128};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
                         elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(LA_ERR_CUDA, "cuTensorMapEncodeTiled(state) failed with CUresult %d", (int)r);
  return LA_OK;
}

// Map over a token-major [rows, heads * 128] BF16 matrix with boxes of `box_rows` tokens x 128
// values (one head's row), unswizzled: a request's draft tokens of one head in one copy.
la_status encode_bf16_token_map(CUtensorMap* map, const void* base, int64_t rows, int64_t heads,
                                       int box_rows, const char* name) {
  auto enc = la_host::tensor_map_encoder();
  if (!enc) return fail(LA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the CUDA driver");
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(heads * 128), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(heads * 128 * 2)};
  const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                         elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(LA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name, (int)r);
  return LA_OK;
}


// Shape checks shared by the three entry points.
la_status check_shapes(int B, int T, int H, int HV, int D, int V, int pool_size, const int32_t* state_indices) {
  if (D != V || (D != 128 && D != 64 && D != 256))
    return fail(LA_ERR_UNSUPPORTED, "only D == V == 128, 64 or 256 is implemented (got D=%d, V=%d)", D, V);
  if (H <= 0 || HV <= 0) return fail(LA_ERR_INVALID_ARGUMENT, "H and HV must be positive (got %d, %d)", H, HV);
  if (HV % H != 0) return fail(LA_ERR_UNSUPPORTED, "HV (%d) must be a multiple of H (%d)", HV, H);
  if (B < 0) return fail(LA_ERR_INVALID_ARGUMENT, "B must be >= 0 (got %d)", B);
  if (T < 1) return fail(LA_ERR_INVALID_ARGUMENT, "T must be >= 1 (got %d)", T);
  if (static_cast<int64_t>(B) * HV * lad::split_of<256>() > INT32_MAX || static_cast<int64_t>(B) * T > INT32_MAX)
    return fail(LA_ERR_UNSUPPORTED, "B*HV or B*T too large");
  if (state_indices ? pool_size <= 0 : pool_size < B)
    return fail(LA_ERR_INVALID_ARGUMENT, "pool_size (%d) must be positive, and >= B (%d) without state_indices",
                pool_size, B);
  if (!aligned4(state_indices)) return fail(LA_ERR_INVALID_ARGUMENT, "state_indices must be 4-byte aligned");
  return LA_OK;
}

// One-time setup per device: the shared memory of the closed-form verify kernel and of the
// tokenwise kernel's D = 256 instances exceeds the default.
cudaError_t setup_kernels() {
  const cudaFuncAttribute attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(lav::la_verify_tc_kernel, attr, lav::verify_smem_bytes());
  if (e == cudaSuccess) e = cudaFuncSetAttribute(lad::la_tokenwise_kernel<lad::kDecode, 256>, attr,
                                                 lad::tokenwise_smem_bytes<256>());
  if (e == cudaSuccess) e = cudaFuncSetAttribute(lad::la_tokenwise_kernel<lad::kVerify, 256>, attr,
                                                 lad::tokenwise_smem_bytes<256>());
  if (e == cudaSuccess) e = cudaFuncSetAttribute(lad::la_tokenwise_kernel<lad::kCommit, 256>, attr,
                                                 lad::tokenwise_smem_bytes<256>());
  return e;
}

template <int kMode>
la_status launch(const lad::Params& p, int D, void* stream) {
  la_host::DeviceState* ds = nullptr;
  la_status st = la_host::current_device(g_dev, &ds, setup_kernels);
  if (st != LA_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t ce;
  if (D == 128)
    ce = la_host::launch_pdl(lad::la_tokenwise_kernel<kMode, 128>,
                             lad::tokenwise_grid<128>(p.B * p.HV * lad::split_of<128>(), ds->sms), lad::kThreads,
                             lad::tokenwise_smem_bytes<128>(), cs, p);
  else if (D == 64)
    ce = la_host::launch_pdl(lad::la_tokenwise_kernel<kMode, 64>,
                             lad::tokenwise_grid<64>(p.B * p.HV * lad::split_of<64>(), ds->sms), lad::kThreads,
                             lad::tokenwise_smem_bytes<64>(), cs, p);
  else
    ce = la_host::launch_pdl(lad::la_tokenwise_kernel<kMode, 256>,
                             lad::tokenwise_grid<256>(p.B * p.HV * lad::split_of<256>(), ds->sms), lad::threads_of<256>(),
                             lad::tokenwise_smem_bytes<256>(), cs, p);
  if (ce == cudaSuccess) ce = cudaGetLastError();
  if (ce != cudaSuccess) return fail(LA_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(ce));
  return LA_OK;
}

lad::Params base_params(const float* slopes, float scale, float* state, const int32_t* state_indices, int* dev_error,
                        int B, int T, int H, int HV, int pool_size) {
  lad::Params p{};
  p.slopes = slopes;
  p.state = state;
  p.state_indices = state_indices;
  p.dev_error = dev_error;
  p.scale = scale;
  p.B = B;
  p.T = T;
  p.H = H;
  p.HV = HV;
  p.G = HV / H;
  p.pool_size = pool_size;
  return p;
}

// Byte sizes of a speculative-decoding call's buffers (the state pool and the KV buffer hold
// pool_size slots with state_indices, else one per request).
struct Sizes {
  uint64_t q, v, state, kbuf, vbuf, slopes, per_request;
};
Sizes sizes(int B, int T, int H, int HV, int D, int V, int pool_size, const int32_t* state_indices) {
  const uint64_t rows = static_cast<uint64_t>(B) * T;
  const uint64_t slots = state_indices ? static_cast<uint64_t>(pool_size) : static_cast<uint64_t>(B);
  Sizes z;
  z.q = rows * H * D * 2;
  z.v = rows * HV * V * 2;
  z.state = slots * HV * static_cast<uint64_t>(V) * D * 4;
  z.kbuf = slots * T * H * D * 2;
  z.vbuf = slots * T * HV * V * 2;
  z.slopes = static_cast<uint64_t>(HV) * 4;
  z.per_request = static_cast<uint64_t>(B) * 4;
  return z;
}

}  // namespace

extern "C" {

la_status la_decode_mtp(const void* q, const void* k, const void* v, const float* slopes, float scale,
                        float* state, const int32_t* state_indices, void* o, int B, int T, int H, int HV, int D,
                        int V, int pool_size, int* dev_error, void* stream) {
  la_host::g_last_error[0] = '\0';
  la_status st = check_shapes(B, T, H, HV, D, V, pool_size, state_indices);
  if (st != LA_OK) return st;
  if (B == 0) return LA_OK;
  if (!q || !k || !v || !o || !state || !slopes)
    return fail(LA_ERR_INVALID_ARGUMENT, "q, k, v, o, state and slopes must be non-null");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(state) || !aligned4(slopes) ||
      !aligned4(dev_error))
    return fail(LA_ERR_INVALID_ARGUMENT, "q, k, v, o, state must be 16-byte and slopes, dev_error 4-byte aligned");
  {
    const Sizes z = sizes(B, T, H, HV, D, V, pool_size, state_indices);
    const la_host::Span ins[] = {{q, z.q, "q"}, {k, z.q, "k"}, {v, z.v, "v"}, {slopes, z.slopes, "slopes"},
                                 {state_indices, z.per_request, "state_indices"}};
    const la_host::Span outs[] = {{o, z.v, "o"}, {state, z.state, "state"}, {dev_error, 4, "dev_error"}};
    if ((st = la_host::check_disjoint(outs, 3, ins, 5)) != LA_OK) return st;
  }
  lad::Params p = base_params(slopes, scale, state, state_indices, dev_error, B, T, H, HV, pool_size);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.o = static_cast<__nv_bfloat16*>(o);
  return launch<lad::kDecode>(p, D, stream);
}

la_status la_verify(const void* q, const void* k, const void* v, const float* slopes, float scale,
                    const float* state, const int32_t* state_indices, void* o, void* kbuf, void* vbuf, int B, int T,
                    int H, int HV, int D, int V, int pool_size, int* dev_error, void* stream) {
  la_host::g_last_error[0] = '\0';
  la_status st = check_shapes(B, T, H, HV, D, V, pool_size, state_indices);
  if (st != LA_OK) return st;
  if (B == 0) return LA_OK;
  if (!q || !k || !v || !o || !state || !slopes)
    return fail(LA_ERR_INVALID_ARGUMENT, "q, k, v, o, state and slopes must be non-null");
  if ((kbuf == nullptr) != (vbuf == nullptr))
    return fail(LA_ERR_INVALID_ARGUMENT, "kbuf and vbuf must be both given or both null");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(state) || !aligned16(kbuf) ||
      !aligned16(vbuf) || !aligned4(slopes) || !aligned4(dev_error))
    return fail(LA_ERR_INVALID_ARGUMENT,
                "q, k, v, o, state, kbuf, vbuf must be 16-byte and slopes, dev_error 4-byte aligned");
  {
    const Sizes z = sizes(B, T, H, HV, D, V, pool_size, state_indices);
    const la_host::Span ins[] = {{q, z.q, "q"},           {k, z.q, "k"}, {v, z.v, "v"}, {slopes, z.slopes, "slopes"},
                                 {state, z.state, "state"}, {state_indices, z.per_request, "state_indices"}};
    const la_host::Span outs[] = {{o, z.v, "o"}, {kbuf, z.kbuf, "kbuf"}, {vbuf, z.vbuf, "vbuf"},
                                  {dev_error, 4, "dev_error"}};
    if ((st = la_host::check_disjoint(outs, 4, ins, 6)) != LA_OK) return st;
  }
  lad::Params p = base_params(slopes, scale, const_cast<float*>(state), state_indices, dev_error, B, T, H, HV,
                              pool_size);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.kbuf = static_cast<__nv_bfloat16*>(kbuf);
  p.vbuf = static_cast<__nv_bfloat16*>(vbuf);
  if (D != 128 || T > lav::kMaxTok || static_cast<int64_t>(pool_size) * HV * 128 > INT32_MAX)
    return launch<lad::kVerify>(p, D, stream);

  // the closed form on the tensor cores (D = 128)
  la_host::DeviceState* ds = nullptr;
  st = la_host::current_device(g_dev, &ds, setup_kernels);
  if (st != LA_OK) return st;
  CUtensorMap tm_s, tm_q, tm_k, tm_v;
  const int64_t rows = static_cast<int64_t>(B) * T;
  if ((st = encode_f32_state_map(&tm_s, state, static_cast<int64_t>(pool_size) * HV * 128)) != LA_OK ||
      (st = encode_bf16_token_map(&tm_q, q, rows, H, lav::kMaxTok, "q")) != LA_OK ||
      (st = encode_bf16_token_map(&tm_k, k, rows, H, lav::kMaxTok, "k")) != LA_OK ||
      (st = encode_bf16_token_map(&tm_v, v, rows, HV, lav::kMaxTok, "v")) != LA_OK)
    return st;
  lav::Params vp{};
  vp.slopes = slopes;
  vp.state_indices = state_indices;
  vp.o = p.o;
  vp.kbuf = p.kbuf;
  vp.vbuf = p.vbuf;
  vp.dev_error = dev_error;
  vp.scale = scale;
  vp.B = B;
  vp.T = T;
  vp.H = H;
  vp.HV = HV;
  vp.G = HV / H;
  vp.pool_size = pool_size;
  const int units = B * HV;
  const int grid = units < ds->sms ? units : ds->sms;
  cudaError_t ce = la_host::launch_pdl(lav::la_verify_tc_kernel, grid, lav::kThreads, lav::verify_smem_bytes(),
                                       static_cast<cudaStream_t>(stream), tm_s, tm_q, tm_k, tm_v, vp);
  if (ce == cudaSuccess) ce = cudaGetLastError();
  if (ce != cudaSuccess) return fail(LA_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(ce));
  return LA_OK;
}

la_status la_commit(float* state, const int32_t* state_indices, const void* kbuf, const void* vbuf,
                    const int32_t* accepted_len, const float* slopes, int B, int T, int H, int HV, int D, int V,
                    int pool_size, int* dev_error, void* stream) {
  la_host::g_last_error[0] = '\0';
  la_status st = check_shapes(B, T, H, HV, D, V, pool_size, state_indices);
  if (st != LA_OK) return st;
  if (B == 0) return LA_OK;
  if (!state || !kbuf || !vbuf || !accepted_len || !slopes)
    return fail(LA_ERR_INVALID_ARGUMENT, "state, kbuf, vbuf, accepted_len and slopes must be non-null");
  if (!aligned16(state) || !aligned16(kbuf) || !aligned16(vbuf) || !aligned4(accepted_len) || !aligned4(slopes) ||
      !aligned4(dev_error))
    return fail(LA_ERR_INVALID_ARGUMENT,
                "state, kbuf, vbuf must be 16-byte and accepted_len, slopes, dev_error 4-byte aligned");
  {
    const Sizes z = sizes(B, T, H, HV, D, V, pool_size, state_indices);
    const la_host::Span ins[] = {{kbuf, z.kbuf, "kbuf"},
                                 {vbuf, z.vbuf, "vbuf"},
                                 {accepted_len, z.per_request, "accepted_len"},
                                 {slopes, z.slopes, "slopes"},
                                 {state_indices, z.per_request, "state_indices"}};
    const la_host::Span outs[] = {{state, z.state, "state"}, {dev_error, 4, "dev_error"}};
    if ((st = la_host::check_disjoint(outs, 2, ins, 5)) != LA_OK) return st;
  }
  lad::Params p = base_params(slopes, 0.f, state, state_indices, dev_error, B, T, H, HV, pool_size);
  p.kbuf = const_cast<__nv_bfloat16*>(static_cast<const __nv_bfloat16*>(kbuf));
  p.vbuf = const_cast<__nv_bfloat16*>(static_cast<const __nv_bfloat16*>(vbuf));
  p.accepted_len = accepted_len;
  return launch<lad::kCommit>(p, D, stream);
}

}  // extern "C"
