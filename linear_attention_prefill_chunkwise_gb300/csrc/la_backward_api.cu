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
  if (p.cu_seqlens) {
    const int b = __ldg(p.cu_seqlens + n), e = __ldg(p.cu_seqlens + n + 1);
    if (b < 0 || e < b || e > p.tokens) return;
  }
  const int slot = p.state_indices ? __ldg(p.state_indices + n) : n;
  if (slot < 0 || slot >= p.pool) return;
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
  float* dk_f32;  // GVA: value head hv's FP32 part of dk ([tokens, HV, D]), summed per group later
  float* dh0;
  float scale;
  int N, T, H, HV, D, tokens, pool;
};

// Heads with slope > kBigSlope, when dh_final is given: the reverse runs started from zero, so
// the last token's dv and dk lack dh_final's term.  With lambda <= e^-64 every other term of G at
// that token is below FP32 resolution, so dv = G k and dk = G^T v with G = scale dout q^T +
// dh_final are recomputed there in FP32 and rounded once (with value heads sharing a q/k head,
// dk's part of this value head is written in FP32, to be summed over the group); an empty
// sequence gets dh0 = dh_final.  One block of D threads per (sequence, value head); thread i
// owns value row i of G and key column i.
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
  const size_t qk_row = (static_cast<size_t>(e - 1) * p.H + hv / (p.HV / p.H)) * D;
  sq[i] = __bfloat162float(p.q[qk_row + i]);
  sk[i] = __bfloat162float(p.k[qk_row + i]);
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
  if (p.dk_f32)
    p.dk_f32[row + i] = p.scale * dv_dot * sq[i] + gtv;
  else
    p.dk[qk_row + i] = __float2bfloat16_rn(p.scale * dv_dot * sq[i] + gtv);
}

struct ReduceParams {
  const float* part;    // [tokens, HV, D] FP32: each value head's part
  __nv_bfloat16* dst;   // [tokens, H, D]: the sum over each q/k head's group of HV / H value heads
  const int32_t* cu_seqlens;
  const int32_t* state_indices;
  int N, T, tokens, pool, H, HV, D;
};

// dst[r][h][d] = bf16(sum over g of part[r][h G + g][d]) for the rows of computed sequences (the
// others are left as they are), 8 values per thread.
__global__ void __launch_bounds__(kCopyThreads) la_group_sum_kernel(const ReduceParams p) {
  const int G = p.HV / p.H, per_row = p.H * p.D / 8;
  for (int r = blockIdx.x; r < p.tokens; r += gridDim.x) {
    if (la_internal::row_sequence(p.cu_seqlens, p.state_indices, p.N, p.T, p.tokens, p.pool, r) < 0) continue;
    for (int i = threadIdx.x; i < per_row; i += kCopyThreads) {
      const int h = i / (p.D / 8), d = 8 * (i - h * (p.D / 8));
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int g = 0; g < G; ++g) {
        const float4* src =
            reinterpret_cast<const float4*>(p.part + (static_cast<size_t>(r) * p.HV + h * G + g) * p.D + d);
        const float4 a = __ldg(src), b = __ldg(src + 1);
        acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
        acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
      }
      uint4 out;
      out.x = la_internal::bf16x2(acc[0], acc[1]);
      out.y = la_internal::bf16x2(acc[2], acc[3]);
      out.z = la_internal::bf16x2(acc[4], acc[5]);
      out.w = la_internal::bf16x2(acc[6], acc[7]);
      *reinterpret_cast<uint4*>(p.dst + (static_cast<size_t>(r) * p.H + h) * p.D + d) = out;
    }
  }
}

// Workspace layout, every section 256-byte aligned.
struct Layout {
  size_t h0t, dhf, dhft, part;
  size_t bytes;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// pool x HV states of D x D FP32 (h0 transposed, dh_final scaled and its transpose) and, with
// value heads sharing q/k heads (HV > H), one [tokens, HV, D] FP32 buffer for the parts of dq
// and dk.
inline Layout layout(int64_t tokens, int H, int HV, int D, int pool, bool has_h0, bool has_dhf) {
  Layout l{};
  const size_t states = align256(static_cast<size_t>(pool) * HV * D * D * 4);
  size_t off = 0;
  l.h0t = off;
  if (has_h0) off += states;
  l.dhf = off;
  if (has_dhf) off += states;
  l.dhft = off;
  if (has_dhf) off += states;
  l.part = off;
  if (HV > H) off += align256(static_cast<size_t>(tokens) * HV * D * 4);
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

la_status check_shape(int D, int V) {
  if (D != V || (D != 128 && D != 64))
    return fail(LA_ERR_UNSUPPORTED, "the backward pass needs D == V == 128 or 64 (got D=%d, V=%d)", D, V);
  return LA_OK;
}

}  // namespace


extern "C" {

la_status la_prefill_bwd_workspace(int B, int T, int H, int HV, int D, int pool_size, int has_h0, int has_dh_final,
                                   size_t* bytes) {
  la_host::g_last_error[0] = '\0';
  if (!bytes) return fail(LA_ERR_INVALID_ARGUMENT, "bytes is null");
  if (B < 0 || T < 0 || H <= 0 || HV <= 0 || D <= 0 || pool_size < 0)
    return fail(LA_ERR_INVALID_ARGUMENT, "bad sizes");
  if (HV % H != 0) return fail(LA_ERR_UNSUPPORTED, "HV (%d) must be a multiple of H (%d)", HV, H);
  *bytes = labw::layout(static_cast<int64_t>(B) * T, H, HV, D, pool_size, has_h0 != 0, has_dh_final != 0).bytes;
  return LA_OK;
}

la_status la_prefill_bwd(const void* q, const void* k, const void* v, const float* slopes, float scale,
                         const float* h0, const void* dout, const float* dh_final, const int32_t* state_indices,
                         const int32_t* cu_seqlens, void* dq, void* dk, void* dv, float* dh0, int B, int T, int N,
                         int H, int HV, int D, int V, int pool_size, void* workspace, size_t workspace_bytes,
                         int* dev_error, void* stream) {
  la_host::g_last_error[0] = '\0';
  la_status st = check_shape(D, V);
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
  const bool grouped = HV > H;  // value heads share q/k heads: dq and dk are sums over a group
  const int pool = (h0 || dh0 || dh_final) ? pool_size : (state_indices ? 0 : N);
  const labw::Layout lay = labw::layout(tokens, H, HV, D, pool, h0 != nullptr, dh_final != nullptr);
  if (lay.bytes > 0 && (!workspace || workspace_bytes < lay.bytes))
    return fail(LA_ERR_INVALID_ARGUMENT, "workspace too small: %zu bytes given, %zu needed", workspace_bytes,
                lay.bytes);
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return fail(LA_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
  {
    // q, k, v, dout, slopes, h0, dh_final and the index arrays are read; the gradients, the
    // workspace and dev_error are written, and none of these may share memory with another
    const uint64_t tk = static_cast<uint64_t>(tokens);
    const uint64_t bq = tk * H * D * 2, bv = tk * HV * V * 2;
    const uint64_t slots = state_indices ? static_cast<uint64_t>(pool_size) : static_cast<uint64_t>(N);
    const uint64_t bst = slots * HV * static_cast<uint64_t>(V) * D * 4;
    const la_host::Span ins[] = {{q, bq, "q"},
                                 {k, bq, "k"},
                                 {v, bv, "v"},
                                 {dout, bv, "dout"},
                                 {slopes, static_cast<uint64_t>(HV) * 4, "slopes"},
                                 {h0, bst, "h0"},
                                 {dh_final, bst, "dh_final"},
                                 {state_indices, static_cast<uint64_t>(N) * 4, "state_indices"},
                                 {cu_seqlens, cu_seqlens ? static_cast<uint64_t>(N + 1) * 4 : 0, "cu_seqlens"}};
    const la_host::Span outs[] = {{dq, bq, "dq"},   {dk, bq, "dk"},
                                  {dv, bv, "dv"},   {dh0, bst, "dh0"},
                                  {workspace, lay.bytes, "workspace"}, {dev_error, 4, "dev_error"}};
    if ((st = la_host::check_disjoint(outs, 6, ins, 9)) != LA_OK) return st;
  }
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return fail(LA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(ce));

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* h0t = h0 ? reinterpret_cast<float*>(ws + lay.h0t) : nullptr;
  float* dhf = dh_final ? reinterpret_cast<float*>(ws + lay.dhf) : nullptr;
  float* dhft = dh_final ? reinterpret_cast<float*>(ws + lay.dhft) : nullptr;
  float* part = grouped ? reinterpret_cast<float*>(ws + lay.part) : nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const dim3 tgrid(static_cast<unsigned>(pool) * HV, (D / 32) * (D / 32)), tblock(32, 8);
  const int rgrid = static_cast<int>(tokens < 4096 ? (tokens > 0 ? tokens : 1) : 4096);
  labw::ReduceParams rp{};
  rp.cu_seqlens = cu_seqlens;
  rp.state_indices = state_indices;
  rp.N = N;
  rp.T = cu_seqlens ? 0 : T;
  rp.tokens = static_cast<int>(tokens);
  rp.pool = la_host::effective_pool_size(h0, dh0, state_indices, pool_size, N);
  rp.H = H;
  rp.HV = HV;
  rp.D = D;

  // 1. dq: the forward recurrence with (q, k, v) -> (dout, v, k) from h0^T; with value heads
  //    sharing a q/k head, per value head (q' and k' of HV heads, v' of H) into FP32 parts that
  //    are summed over each group
  if (h0 && pool > 0) {
    labw::la_transpose_states_kernel<<<tgrid, tblock, 0, s>>>(h0, h0t, D, nullptr, HV, 1.f, 1);
    if ((st = launched("state transpose")) != LA_OK) return st;
  }
  if (tokens > 0) {
    if (!grouped) {
      st = la_prefill_fwd(dout, v, k, slopes, scale, h0t, state_indices, cu_seqlens, dq, nullptr, B, T, N, H, HV, D,
                          V, pool_size, LA_SCHED_AUTO, dev_error, stream);
      if (st != LA_OK) return st;
    } else {
      st = la_internal::chunkwise(dout, v, k, slopes, scale, h0t, state_indices, cu_seqlens, nullptr, part, nullptr, B,
                                  T, N, HV, HV, H, D, pool_size, false, dev_error, stream);
      if (st != LA_OK) return st;
      rp.part = part;
      rp.dst = static_cast<__nv_bfloat16*>(dq);
      labw::la_group_sum_kernel<<<rgrid, labw::kCopyThreads, 0, s>>>(rp);
      if ((st = launched("group sum")) != LA_OK) return st;
    }
  }

  // 2. dh_final / (lambda scale), as it is and transposed: the reverse runs' initial states
  if (dh_final && pool > 0) {
    labw::la_transpose_states_kernel<<<tgrid, tblock, 0, s>>>(dh_final, dhf, D, slopes, HV, scale, 0);
    if ((st = launched("state scaling")) != LA_OK) return st;
    labw::la_transpose_states_kernel<<<tgrid, tblock, 0, s>>>(dh_final, dhft, D, slopes, HV, scale, 1);
    if ((st = launched("state transpose")) != LA_OK) return st;
  }

  // 3. dv (and dh0): the recurrence run backwards with (q, k, v) -> (k, q, dout), per value head
  st = la_internal::chunkwise(k, q, dout, slopes, scale, dhf, state_indices, cu_seqlens, dv, nullptr, dh0, B, T, N, H,
                              HV, HV, D, pool_size, true, dev_error, stream);
  if (st != LA_OK) return st;
  // 4. dk: the recurrence run backwards with (q, k, v) -> (v, dout, q); grouped: per value head
  //    into FP32 parts
  if (tokens > 0) {
    st = la_internal::chunkwise(v, dout, q, slopes, scale, dhft, state_indices, cu_seqlens, grouped ? nullptr : dk,
                                part, nullptr, B, T, N, HV, HV, H, D, pool_size, true, dev_error, stream);
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
    bp.dk_f32 = part;
    bp.dv = static_cast<__nv_bfloat16*>(dv);
    bp.dh0 = dh0;
    bp.scale = scale;
    bp.N = N;
    bp.T = cu_seqlens ? 0 : T;
    bp.H = H;
    bp.HV = HV;
    bp.D = D;
    bp.tokens = static_cast<int>(tokens);
    bp.pool = pool_size;
    labw::la_bwd_big_slope_kernel<<<static_cast<unsigned>(N) * HV, D, 0, s>>>(bp);
    if ((st = launched("large-slope final state")) != LA_OK) return st;
  }
  // 7. grouped: dk as the sum of its value heads' parts
  if (grouped && tokens > 0) {
    rp.part = part;
    rp.dst = static_cast<__nv_bfloat16*>(dk);
    labw::la_group_sum_kernel<<<rgrid, labw::kCopyThreads, 0, s>>>(rp);
    if ((st = launched("group sum")) != LA_OK) return st;
  }
  return LA_OK;
}

}  // extern "C"
