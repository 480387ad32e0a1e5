// la_backward_api.cu -- host side of include/la_backward.h and its helper kernels.
//
// The backward pass runs the chunkwise kernel three times on rearranged inputs (the derivation
// is in include/la_backward.h): once forward (la_prefill_fwd) and twice in its reverse instance,
// which walks every sequence from its last token to its first in place.  What is left to do here
// is transposing and scaling [D x D] states, the final scaling of dh0 and the large-slope
// fix-up; nothing here reads device memory on the host or synchronises.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "../../include/la_backward.h"
#include "la_host_common.h"
#include "la_prefill_internal.h"

namespace labw {

constexpr int kCopyThreads = 256;
// Largest slope whose 1 / lambda = e^slope scales dh_final into the reverse runs' initial state
// (e^64 = 6.2e27, far from FP32 overflow); heads with larger slopes start those runs from zero
// and get dh_final's only non-negligible term, at their sequence's last token, from
// la_bwd_big_slope_kernel (the others carry lambda^n <= e^-64).
constexpr float kBigSlope = 64.f;

// dst[s][b][a] = f * src[s][a][b] (transpose = 1) or dst[s][a][b] = f * src[s][a][b] (transpose
// = 0) for square [D x D] FP32 matrices, one block per (matrix, 32 x 32 tile); matrix s belongs to
// head s % HV.  f = 1 without slopes; with slopes f = e^slope / scale = 1 / (lambda scale) of
// the matrix's head (0 beyond kBigSlope).
__global__ void __launch_bounds__(kCopyThreads) la_transpose_states_kernel(const float* src, float* dst, int D,
                                                                         const float* slopes, int HV, float scale,
                                                                         int transpose) {
  __shared__ float tile[32][33];
  const size_t base = static_cast<size_t>(blockIdx.x) * D * D;
  float factor = 1.f;
  if (slopes) {
    const float sl = __ldg(slopes + blockIdx.x % HV);
    factor = sl <= kBigSlope ? expf(sl) / scale : 0.f;
  }
  const int tiles = D / 32;
  const int a0 = (blockIdx.y / tiles) * 32, b0 = (blockIdx.y % tiles) * 32;
  for (int i = threadIdx.y; i < 32; i += 8) tile[i][threadIdx.x] = __ldg(src + base + static_cast<size_t>(a0 + i) * D + b0 + threadIdx.x);
  __syncthreads();
  if (transpose) {
    for (int i = threadIdx.y; i < 32; i += 8)
      dst[base + static_cast<size_t>(b0 + i) * D + a0 + threadIdx.x] = factor * tile[threadIdx.x][i];
  } else {
    for (int i = threadIdx.y; i < 32; i += 8)
      dst[base + static_cast<size_t>(a0 + i) * D + b0 + threadIdx.x] = factor * tile[i][threadIdx.x];
  }
}

struct Dh0Params {
  float* dh0;
  const float* slopes;
  const int32_t* state_indices;
  const int32_t* cu_seqlens;
  float scale;
  int N, T, HV, D, tokens, pool;
};

// dh0[slot][hv] *= lambda scale: the dv run leaves G_0 / (lambda scale) there (its initial state
// dh_final / (lambda scale) carries the final state's gradient into G_{L-1} undecayed).
// Sequences the forward kernels skipped are skipped too.
__global__ void __launch_bounds__(kCopyThreads) la_finish_dh0_kernel(const Dh0Params p) {
  const int n = blockIdx.x / p.HV, hv = blockIdx.x - n * p.HV;
  int len = p.T;
  if (p.cu_seqlens) {
    const int b = __ldg(p.cu_seqlens + n), e = __ldg(p.cu_seqlens + n + 1);
    if (b < 0 || e < b || e > p.tokens) return;
    len = e - b;
  }
  const int slot = p.state_indices ? __ldg(p.state_indices + n) : n;
  if (slot < 0 || slot >= p.pool) return;
  (void)len;
  const float f = p.scale * expf(-__ldg(p.slopes + hv));
  float4* st = reinterpret_cast<float4*>(p.dh0 + (static_cast<size_t>(slot) * p.HV + hv) * p.D * p.D);
  for (int i = threadIdx.x; i < p.D * p.D / 4; i += kCopyThreads) {
    float4 x = st[i];
    x.x *= f;
    x.y *= f;
    x.z *= f;
    x.w *= f;
    st[i] = x;
  }
}

struct BigSlopeParams {
  const __nv_bfloat16 *q, *k, *v, *dout;
  const float* dh_final;
  const float* slopes;
  const int32_t* state_indices;
  const int32_t* cu_seqlens;
  __nv_bfloat16 *dq, *dk, *dv;
  float* dh0;
  float scale;
  int N, T, HV, D, tokens, pool;
};

// Heads with slope > kBigSlope, when dh_final is given: the reverse runs started from zero, so
// the last token's dv and dk lack dh_final's term.  With lambda <= e^-64 every other term of G at
// that token is below FP32 resolution, so dv = G k and dk = G^T v with G = scale dout q^T +
// dh_final are recomputed there in FP32 and rounded once; an empty sequence gets dh0 = dh_final.
// One block of D threads per (sequence, head); thread i owns value row i of G and key column i.
__global__ void __launch_bounds__(128) la_bwd_big_slope_kernel(const BigSlopeParams p) {
  __shared__ float sq[128], sk[128], sv[128], sd[128], red[2][4];
  const int n = blockIdx.x / p.HV, hv = blockIdx.x - n * p.HV, i = threadIdx.x, D = p.D;
  if (__ldg(p.slopes + hv) <= kBigSlope) return;
  int b = n * p.T, e = b + p.T;
  if (p.cu_seqlens) {
    b = __ldg(p.cu_seqlens + n);
    e = __ldg(p.cu_seqlens + n + 1);
    if (b < 0 || e < b || e > p.tokens) return;
  }
  const int slot = p.state_indices ? __ldg(p.state_indices + n) : n;
  if (slot < 0 || slot >= p.pool) return;
  const float* G = p.dh_final + (static_cast<size_t>(slot) * p.HV + hv) * D * D;
  if (e == b) {
    if (p.dh0) {
      float* dst = p.dh0 + (static_cast<size_t>(slot) * p.HV + hv) * D * D;
      for (int x = i; x < D * D; x += D) dst[x] = __ldg(G + x);
    }
    return;
  }
  const size_t row = (static_cast<size_t>(e - 1) * p.HV + hv) * D;
  sq[i] = __bfloat162float(p.q[row + i]);
  sk[i] = __bfloat162float(p.k[row + i]);
  sv[i] = __bfloat162float(p.v[row + i]);
  sd[i] = __bfloat162float(p.dout[row + i]);
  __syncthreads();
  // q . k and dout . v over the block (D / 32 warps)
  float a = sq[i] * sk[i], c = sd[i] * sv[i];
  for (int m = 16; m; m >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, m);
    c += __shfl_xor_sync(0xffffffffu, c, m);
  }
  if ((i & 31) == 0) {
    red[0][i >> 5] = a;
    red[1][i >> 5] = c;
  }
  __syncthreads();
  float qk = 0.f, dv_dot = 0.f;
  for (int w = 0; w < D / 32; ++w) {
    qk += red[0][w];
    dv_dot += red[1][w];
  }
  float gk = 0.f, gtv = 0.f;  // (dh_final k)_i and (dh_final^T v)_i
  for (int j = 0; j < D; ++j) {
    gk = fmaf(__ldg(G + static_cast<size_t>(i) * D + j), sk[j], gk);
    gtv = fmaf(__ldg(G + static_cast<size_t>(j) * D + i), sv[j], gtv);
  }
  p.dv[row + i] = __float2bfloat16_rn(p.scale * qk * sd[i] + gk);
  p.dk[row + i] = __float2bfloat16_rn(p.scale * dv_dot * sq[i] + gtv);
}

// Workspace layout, every section 256-byte aligned.
struct Layout {
  size_t h0t, dhf, dhft;
  size_t bytes;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline Layout layout(int H, int D, int pool, bool has_h0, bool has_dhf) {
  Layout l{};
  const size_t states = align256(static_cast<size_t>(pool) * H * D * D * 4);
  size_t off = 0;
  l.h0t = off;
  if (has_h0) off += states;
  l.dhf = off;
  if (has_dhf) off += states;
  l.dhft = off;
  if (has_dhf) off += states;
  l.bytes = off;
  return l;
}

}  // namespace labw

namespace {

using la_host::fail;

la_status launched(const char* what) {
  const cudaError_t ce = cudaGetLastError();
  if (ce != cudaSuccess) return fail(LA_ERR_CUDA, "%s kernel launch failed: %s", what, cudaGetErrorString(ce));
  return LA_OK;
}

la_status check_shape(int H, int HV, int D, int V) {
  if (H != HV) return fail(LA_ERR_UNSUPPORTED, "the backward pass needs H == HV (got H=%d, HV=%d)", H, HV);
  if (D != V || (D != 128 && D != 64))
    return fail(LA_ERR_UNSUPPORTED, "the backward pass needs D == V == 128 or 64 (got D=%d, V=%d)", D, V);
  return LA_OK;
}

}  // namespace

extern "C" {

la_status la_prefill_bwd_workspace(int B, int T, int H, int D, int pool_size, int has_h0, int has_dh_final,
                                   size_t* bytes) {
  la_host::g_last_error[0] = '\0';
  if (!bytes) return fail(LA_ERR_INVALID_ARGUMENT, "bytes is null");
  if (B < 0 || T < 0 || H <= 0 || D <= 0 || pool_size < 0) return fail(LA_ERR_INVALID_ARGUMENT, "bad sizes");
  *bytes = labw::layout(H, D, pool_size, has_h0 != 0, has_dh_final != 0).bytes;
  return LA_OK;
}

la_status la_prefill_bwd(const void* q, const void* k, const void* v, const float* slopes, float scale,
                         const float* h0, const void* dout, const float* dh_final, const int32_t* state_indices,
                         const int32_t* cu_seqlens, void* dq, void* dk, void* dv, float* dh0, int B, int T, int N,
                         int H, int HV, int D, int V, int pool_size, void* workspace, size_t workspace_bytes,
                         int* dev_error, void* stream) {
  la_host::g_last_error[0] = '\0';
  la_status st = check_shape(H, HV, D, V);
  if (st != LA_OK) return st;
  // The forward's checks cover q, k, v, slopes, the state pool and the modes; the gradients
  // share the layouts of q (dq, dk) and v (dv, dout), dh_final and dh0 that of h0.
  bool nothing = false;
  st = la_host::check_prefill_args(q, k, v, slopes, h0, state_indices, cu_seqlens, dq, dh0, B, T, N, H, HV, D, V,
                                   pool_size, dev_error, &nothing);
  if (st != LA_OK) return st;
  const int64_t tokens = static_cast<int64_t>(B) * T;
  if (N > 0 && tokens > 0 && (!dout || !dk || !dv))
    return fail(LA_ERR_INVALID_ARGUMENT, "dout, dq, dk and dv must be non-null");
  if (!la_host::aligned16(dout) || !la_host::aligned16(dk) || !la_host::aligned16(dv) ||
      !la_host::aligned16(dh_final))
    return fail(LA_ERR_INVALID_ARGUMENT, "dout, dk, dv and dh_final must be 16-byte aligned");
  if (dh_final && scale == 0.f) return fail(LA_ERR_INVALID_ARGUMENT, "dh_final needs scale != 0");
  if (dh_final && !dh0 && !h0 && !state_indices && pool_size < N)
    return fail(LA_ERR_INVALID_ARGUMENT, "pool_size (%d) must be >= N (%d) without state_indices", pool_size, N);
  if (N == 0) return LA_OK;
  if (tokens == 0 && !dh0) return LA_OK;
  const int pool = (h0 || dh0 || dh_final) ? pool_size : (state_indices ? 0 : N);
  const labw::Layout lay = labw::layout(H, D, pool, h0 != nullptr, dh_final != nullptr);
  if (lay.bytes > 0 && (!workspace || workspace_bytes < lay.bytes))
    return fail(LA_ERR_INVALID_ARGUMENT, "workspace too small: %zu bytes given, %zu needed", workspace_bytes,
                lay.bytes);
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return fail(LA_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return fail(LA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(ce));

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* h0t = h0 ? reinterpret_cast<float*>(ws + lay.h0t) : nullptr;
  float* dhf = dh_final ? reinterpret_cast<float*>(ws + lay.dhf) : nullptr;
  float* dhft = dh_final ? reinterpret_cast<float*>(ws + lay.dhft) : nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const dim3 tgrid(static_cast<unsigned>(pool) * HV, (D / 32) * (D / 32)), tblock(32, 8);

  // 1. dq: the forward recurrence with (q, k, v) -> (dout, v, k) from h0^T
  if (h0 && pool > 0) {
    labw::la_transpose_states_kernel<<<tgrid, tblock, 0, s>>>(h0, h0t, D, nullptr, HV, 1.f, 1);
    if ((st = launched("state transpose")) != LA_OK) return st;
  }
  if (tokens > 0) {
    st = la_prefill_fwd(dout, v, k, slopes, scale, h0t, state_indices, cu_seqlens, dq, nullptr, B, T, N, H, HV, D, V,
                        pool_size, LA_SCHED_AUTO, dev_error, stream);
    if (st != LA_OK) return st;
  }

  // 2. dh_final / (lambda scale), as it is and transposed: the reverse runs' initial states
  if (dh_final && pool > 0) {
    labw::la_transpose_states_kernel<<<tgrid, tblock, 0, s>>>(dh_final, dhf, D, slopes, HV, scale, 0);
    if ((st = launched("state scaling")) != LA_OK) return st;
    labw::la_transpose_states_kernel<<<tgrid, tblock, 0, s>>>(dh_final, dhft, D, slopes, HV, scale, 1);
    if ((st = launched("state transpose")) != LA_OK) return st;
  }

  // 3. dv (and dh0): the recurrence run backwards with (q, k, v) -> (k, q, dout)
  st = la_internal::prefill_reverse(k, q, dout, slopes, scale, dhf, state_indices, cu_seqlens, dv, dh0, B, T, N, H,
                                    HV, D, V, pool_size, dev_error, stream);
  if (st != LA_OK) return st;
  // 4. dk: the recurrence run backwards with (q, k, v) -> (v, dout, q)
  if (tokens > 0) {
    st = la_internal::prefill_reverse(v, dout, q, slopes, scale, dhft, state_indices, cu_seqlens, dk, nullptr, B, T,
                                      N, H, HV, D, V, pool_size, dev_error, stream);
    if (st != LA_OK) return st;
  }
  // 5. dh0 = scale lambda G_0 / scale
  if (dh0) {
    labw::Dh0Params dp{};
    dp.dh0 = dh0;
    dp.slopes = slopes;
    dp.state_indices = state_indices;
    dp.cu_seqlens = cu_seqlens;
    dp.scale = scale;
    dp.N = N;
    dp.T = cu_seqlens ? 0 : T;
    dp.HV = HV;
    dp.D = D;
    dp.tokens = static_cast<int>(tokens);
    dp.pool = pool_size;
    labw::la_finish_dh0_kernel<<<static_cast<unsigned>(N) * HV, labw::kCopyThreads, 0, s>>>(dp);
    if ((st = launched("dh0")) != LA_OK) return st;
  }
  // 6. heads with slopes beyond kBigSlope: dh_final's last-token term
  if (dh_final) {
    labw::BigSlopeParams bp{};
    bp.q = static_cast<const __nv_bfloat16*>(q);
    bp.k = static_cast<const __nv_bfloat16*>(k);
    bp.v = static_cast<const __nv_bfloat16*>(v);
    bp.dout = static_cast<const __nv_bfloat16*>(dout);
    bp.dh_final = dh_final;
    bp.slopes = slopes;
    bp.state_indices = state_indices;
    bp.cu_seqlens = cu_seqlens;
    bp.dk = static_cast<__nv_bfloat16*>(dk);
    bp.dv = static_cast<__nv_bfloat16*>(dv);
    bp.dh0 = dh0;
    bp.scale = scale;
    bp.N = N;
    bp.T = cu_seqlens ? 0 : T;
    bp.HV = HV;
    bp.D = D;
    bp.tokens = static_cast<int>(tokens);
    bp.pool = pool_size;
    labw::la_bwd_big_slope_kernel<<<static_cast<unsigned>(N) * HV, D, 0, s>>>(bp);
    if ((st = launched("large-slope final state")) != LA_OK) return st;
  }
  return LA_OK;
}

}  // extern "C"
