// la_d256_api.cu -- host side of include/la_d256.h and its helper kernels: the D = V = 256
// prefill as four independent 128 x 128 blocks of the state, run by the D = 128 chunkwise kernel.
//
// Virtual heads.  With G = HV / H, value head hv = hq G + g, value half a and key half b, the
// chunkwise kernel runs 4 HV virtual value heads per sequence,
//     u = (2 hq + b) 2G + 2g + a,
// over q and k read in place as [tokens, 2H, 128] (virtual q/k head u / 2G = 2 hq + b: the b half
// of head hq) and v as [tokens, 2HV, 128] (the kernel's value-head fold drops the digit b of u:
// v head 2 hv + a, the a half of head hv).  Virtual head u evolves the state block
// S[a half of v][b half of k] from its block of h0 and writes its part of o[.][hv][a half] in
// FP32; la_d256_sum_kernel adds the parts of b = 0 and 1 and rounds once.  Fixed-length batches
// of at most kShortMax tokens per sequence go to the tokenwise kernel's D = 256 instance instead
// (whole 256 x 256 states, BF16 outputs, no workspace).  Nothing here reads device memory on the
// host or synchronises.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/la_d256.h"
#include "../../include/la_segment.h"
#include "la_decode_kernels.cuh"
#include "la_host_common.h"
#include "la_prefill_internal.h"

namespace la256 {

constexpr int kThreads = 256;
constexpr int kHalf = 128;       // the kernel's head dimension
constexpr int kRowsPerStep = 8;  // rows of a 128 x 128 block per copy step (kThreads float4)
constexpr int kShortMax = 32;    // longest sequence taken by the tokenwise kernel
constexpr int kSplitAvg = 64;    // packed batches of at most this many tokens per sequence on average are split

// The value head hv, value half a and key half b of virtual head u (G value heads per q/k head).
struct Virt {
  int hv, a, b;
};
__device__ __forceinline__ Virt virt(int u, int G) {
  const int G2 = 2 * G, qk = u / G2, j = u - qk * G2;
  Virt x;
  x.b = qk & 1;
  x.a = j & 1;
  x.hv = (qk >> 1) * G + (j >> 1);
  return x;
}

struct TableParams {
  const float* slopes;           // [HV]
  const int32_t* state_indices;  // [N] or null
  float* slopes_q;               // [4 HV]: the slope of each virtual head's value head
  int32_t* slot_q;               // [N]: n, or -1 for a padded sequence or a bad index
  int* dev_error;
  int N, HV, G, pool;
};

__global__ void __launch_bounds__(kThreads) la_d256_tables_kernel(const TableParams t) {
  const int i = blockIdx.x * kThreads + threadIdx.x;
  if (i < 4 * t.HV) t.slopes_q[i] = __ldg(t.slopes + virt(i, t.G).hv);
  if (i < t.N) {
    int s = i;
    if (t.state_indices) {
      const int idx = __ldg(t.state_indices + i);
      if (idx >= t.pool) {
        if (t.dev_error) atomicOr(t.dev_error, 2);  // LA_DEV_ERR_BAD_INDEX: the sequence is skipped
        s = -1;
      } else if (idx < 0) {
        s = -1;
      }
    }
    t.slot_q[i] = s;
  }
}

struct BlockParams {
  const float* big_in;   // gather: h0 [P, HV, 256, 256]
  float* big_out;        // scatter: h_final [P, HV, 256, 256]
  float* blocks;         // [N, 4 HV, 128, 128] in the workspace
  const int32_t* state_indices;
  const int32_t* cu_seqlens;
  int N, HV, G, pool, tokens;
  int short_max;  // packed: sequences of at most this many tokens are skipped (-1: none)
};

// grid (N * 4 HV, y): a block's 128 rows split over y CTAs (y divides 16), one float4 per thread
// and step.  gather: blocks[n][u] <- the
// (a, b) block of h0[slot(n)][hv]; scatter: the (a, b) block of h_final[slot(n)][hv] <-
// blocks[n][u], for sequences that ran (valid slot and, packed, valid bounds).
template <bool kGather>
__global__ void __launch_bounds__(kThreads) la_d256_blocks_kernel(const BlockParams p) {
  const int HVq = 4 * p.HV;
  const int n = blockIdx.x / HVq, u = blockIdx.x - n * HVq;
  int slot = n;
  if (p.state_indices) {
    slot = __ldg(p.state_indices + n);
    if (slot < 0 || slot >= p.pool) return;
  }
  if (p.cu_seqlens && (!kGather || p.short_max >= 0)) {
    const int b = __ldg(p.cu_seqlens + n), e = __ldg(p.cu_seqlens + n + 1);
    if (!kGather && (b < 0 || e < b || e > p.tokens)) return;  // the chunkwise kernel skipped this sequence
    if (e - b <= p.short_max) return;  // a sequence of the tokenwise kernel, which reads and writes whole states
  }
  const Virt x = virt(u, p.G);
  const int c = 4 * (threadIdx.x & 31);
  const int rows = kHalf / static_cast<int>(gridDim.y), r0 = static_cast<int>(blockIdx.y) * rows;
  for (int r = r0 + static_cast<int>(threadIdx.x >> 5); r < r0 + rows; r += kRowsPerStep) {
    const size_t big = ((static_cast<size_t>(slot) * p.HV + x.hv) * 256 + x.a * kHalf + r) * 256 + x.b * kHalf + c;
    const size_t small = ((static_cast<size_t>(n) * HVq + u) * kHalf + r) * kHalf + c;
    if (kGather)
      *reinterpret_cast<float4*>(p.blocks + small) = __ldg(reinterpret_cast<const float4*>(p.big_in + big));
    else
      *reinterpret_cast<float4*>(p.big_out + big) = *reinterpret_cast<const float4*>(p.blocks + small);
  }
}

struct SumParams {
  const float* part;  // [tokens, 4 HV, 128] FP32
  __nv_bfloat16* o;   // [tokens, HV, 256]
  const int32_t* cu_seqlens;
  const int32_t* state_indices;
  int N, T, tokens, pool, HV, G;
  int short_max;  // packed: rows of sequences of at most this many tokens are skipped (-1: none)
};

// o[r][hv][128 a + c] = bf16(part[r][u(b = 0)][c] + part[r][u(b = 1)][c]) for the rows of
// sequences that ran (the others are left as they are), 8 values per thread.
__global__ void __launch_bounds__(kThreads) la_d256_sum_kernel(const SumParams p) {
  const int per_row = p.HV * 256 / 8, G2 = 2 * p.G;
  for (int r = blockIdx.x; r < p.tokens; r += gridDim.x) {
    const int n = la_internal::row_sequence(p.cu_seqlens, p.state_indices, p.N, p.T, p.tokens, p.pool, r);
    if (n < 0) continue;
    if (p.short_max >= 0 && __ldg(p.cu_seqlens + n + 1) - __ldg(p.cu_seqlens + n) <= p.short_max) continue;
    for (int i = threadIdx.x; i < per_row; i += kThreads) {
      const int hv = i >> 5, d = 8 * (i & 31);
      const int a = d >> 7, c = d & (kHalf - 1);
      const int hq = hv / p.G, g = hv - hq * p.G;
      const int u0 = 2 * hq * G2 + 2 * g + a;  // key half 0; key half 1 is u0 + 2G
      const float* row = p.part + static_cast<size_t>(r) * 4 * p.HV * kHalf;
      const float4* s0 = reinterpret_cast<const float4*>(row + static_cast<size_t>(u0) * kHalf + c);
      const float4* s1 = reinterpret_cast<const float4*>(row + static_cast<size_t>(u0 + G2) * kHalf + c);
      const float4 x0 = __ldg(s0), x1 = __ldg(s0 + 1), y0 = __ldg(s1), y1 = __ldg(s1 + 1);
      uint4 out;
      out.x = la_internal::bf16x2(x0.x + y0.x, x0.y + y0.y);
      out.y = la_internal::bf16x2(x0.z + y0.z, x0.w + y0.w);
      out.z = la_internal::bf16x2(x1.x + y1.x, x1.y + y1.y);
      out.w = la_internal::bf16x2(x1.z + y1.z, x1.w + y1.w);
      *reinterpret_cast<uint4*>(p.o + (static_cast<size_t>(r) * p.HV + hv) * 256 + d) = out;
    }
  }
}

// Workspace layout, every section 256-byte aligned.
struct Layout {
  size_t part, blocks, slopes_q, slot_q, bytes;
};
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
inline Layout layout(int64_t tokens, int N, int HV, bool has_state) {
  Layout l{};
  size_t off = 0;
  l.part = off;
  off = align256(off + static_cast<size_t>(tokens) * 4 * HV * kHalf * sizeof(float));
  l.blocks = off;
  if (has_state) off = align256(off + static_cast<size_t>(N) * 4 * HV * kHalf * kHalf * sizeof(float));
  l.slopes_q = off;
  off = align256(off + static_cast<size_t>(4) * HV * sizeof(float));
  l.slot_q = off;
  off = align256(off + static_cast<size_t>(N) * sizeof(int32_t));
  l.bytes = off;
  return l;
}

la_host::DeviceState g_dev[la_host::kMaxDevices];

cudaError_t setup_kernels() {
  return cudaFuncSetAttribute(lad::la_tokenwise_kernel<lad::kPrefill, 256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              lad::tokenwise_smem_bytes<256>());
}

la_status launched(const char* what) {
  const cudaError_t ce = cudaGetLastError();
  if (ce != cudaSuccess) return la_host::fail(LA_ERR_CUDA, "%s launch failed: %s", what, cudaGetErrorString(ce));
  return LA_OK;
}

// The tokenwise kernel's D = 256 instance in prefill mode on whole states: every sequence of a
// fixed-length batch (T <= kShortMax), or the sequences of at most kShortMax tokens of a packed one.
la_status launch_tokenwise(const void* q, const void* k, const void* v, const float* slopes, float scale,
                           const float* h0, const int32_t* state_indices, const int32_t* cu_seqlens, void* o,
                           float* h_final, int T, int N, int H, int HV, int pool, int64_t tokens,
                           la_host::DeviceState* ds, int* dev_error, void* stream) {
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
  tp.T = cu_seqlens ? 0 : T;
  tp.H = H;
  tp.HV = HV;
  tp.G = HV / H;
  tp.pool_size = pool;
  tp.num_tokens = static_cast<int>(tokens);
  tp.short_max = kShortMax;
  const int parts = N * HV * lad::split_of<256>();  // <= 4 N HV, checked by check_args
  cudaError_t ce = la_host::launch_pdl(lad::la_tokenwise_kernel<lad::kPrefill, 256>,
                                       lad::tokenwise_grid<256>(parts, ds->sms), lad::threads_of<256>(),
                                       lad::tokenwise_smem_bytes<256>(), static_cast<cudaStream_t>(stream), tp);
  if (ce == cudaSuccess) ce = cudaGetLastError();
  if (ce != cudaSuccess) return la_host::fail(LA_ERR_CUDA, "tokenwise kernel launch failed: %s", cudaGetErrorString(ce));
  return LA_OK;
}

// The checks of la_prefill_fwd_d256 and its segmented form: D = V = 256, the head counts, and
// la_prefill_fwd's checks on the same memory seen as 2 H q/k and 2 HV value heads of 128.
la_status check_args(const void* q, const void* k, const void* v, const float* slopes, const float* h0,
                     const int32_t* state_indices, const int32_t* cu_seqlens, const void* o, const float* h_final,
                     int B, int T, int N, int H, int HV, int D, int V, int pool_size, const int* dev_error,
                     bool* nothing) {
  using la_host::fail;
  if (D != 256 || V != 256) return fail(LA_ERR_UNSUPPORTED, "the D = 256 prefill needs D == V == 256 (got D=%d, V=%d)", D, V);
  if (H <= 0 || HV <= 0) return fail(LA_ERR_INVALID_ARGUMENT, "H and HV must be positive (got %d, %d)", H, HV);
  if (HV % H != 0) return fail(LA_ERR_UNSUPPORTED, "HV (%d) must be a multiple of H (%d)", HV, H);
  const la_status st = la_host::check_prefill_args(q, k, v, slopes, h0, state_indices, cu_seqlens, o, h_final, B, T,
                                                   N, 2 * H, 2 * HV, kHalf, kHalf, pool_size, dev_error, nothing);
  if (st != LA_OK || *nothing) return st;
  if (static_cast<int64_t>(N) * 4 * HV > INT32_MAX) return fail(LA_ERR_UNSUPPORTED, "4*N*HV too large");
  return LA_OK;
}

// The block path of a call whose arguments are checked: the per-virtual-head tables, the h0
// blocks, the D = 128 chunkwise kernel (segment_len < 0) or the segmented prefill
// (segment_len >= 0, its seg_bytes of workspace after the block path's) over the 4 HV virtual
// heads, the sum of the key halves and the final blocks.
la_status blocks_path(const void* q, const void* k, const void* v, const float* slopes, float scale, const float* h0,
                      const int32_t* state_indices, const int32_t* cu_seqlens, void* o, float* h_final, int B, int T,
                      int N, int H, int HV, int pool_size, int segment_len, size_t seg_bytes, void* workspace,
                      size_t workspace_bytes, int* dev_error, void* stream) {
  using la_host::fail;
  la_status st;
  const int64_t tokens = static_cast<int64_t>(B) * T;
  const int pool = la_host::effective_pool_size(h0, h_final, state_indices, pool_size, N);
  const bool has_state = h0 || h_final;
  const Layout l = layout(tokens, N, HV, has_state);
  const size_t need = l.bytes + seg_bytes;
  if (!workspace || workspace_bytes < need)
    return fail(LA_ERR_INVALID_ARGUMENT, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, need);
  if (reinterpret_cast<uintptr_t>(workspace) % 256)
    return fail(LA_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
  if ((st = la_host::check_prefill_disjoint(q, k, v, slopes, h0, state_indices, cu_seqlens, o, h_final, dev_error, B,
                                            T, N, H, HV, 256, 256, pool_size, workspace, need)) != LA_OK)
    return st;
  la_host::DeviceState* ds = nullptr;
  if ((st = la_host::current_device(g_dev, &ds, setup_kernels)) != LA_OK) return st;
  // a packed batch of mostly short sequences (not segmented): those of at most kShortMax tokens
  // run the tokenwise kernel on whole states, the block path skips them
  const bool split = segment_len < 0 && cu_seqlens && tokens <= static_cast<int64_t>(kSplitAvg) * N;
  const int short_max = split ? kShortMax : -1;
  if (split && (st = launch_tokenwise(q, k, v, slopes, scale, h0, state_indices, cu_seqlens, o, h_final, T, N, H, HV,
                                      pool, tokens, ds, dev_error, stream)) != LA_OK)
    return st;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* part = reinterpret_cast<float*>(ws + l.part);
  float* blocks = has_state ? reinterpret_cast<float*>(ws + l.blocks) : nullptr;
  float* slopes_q = reinterpret_cast<float*>(ws + l.slopes_q);
  int32_t* slot_q = reinterpret_cast<int32_t*>(ws + l.slot_q);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int G = HV / H;

  // 1. per-virtual-head slopes, the sequences that run, and the h0 blocks
  TableParams tp{slopes, state_indices, slopes_q, slot_q, dev_error, N, HV, G, pool};
  const int tgrid = static_cast<int>(((N > 4 * HV ? N : 4 * HV) + kThreads - 1) / kThreads);
  la_d256_tables_kernel<<<tgrid, kThreads, 0, s>>>(tp);
  if ((st = launched("d256 tables")) != LA_OK) return st;
  BlockParams bp{h0, h_final, blocks, state_indices, cu_seqlens, N, HV, G, pool, static_cast<int>(tokens), short_max};
  // few blocks: split each over 16 CTAs (8 rows each); many: one CTA per block, so that the
  // blocks of short sequences cost one CTA each
  const unsigned nblocks = static_cast<unsigned>(N) * 4 * HV;
  const dim3 bgrid(nblocks, nblocks < 1024 ? kHalf / kRowsPerStep : 1);
  if (h0) {
    la_d256_blocks_kernel<true><<<bgrid, kThreads, 0, s>>>(bp);
    if ((st = launched("d256 gather")) != LA_OK) return st;
  }

  // 2. the D = 128 chunkwise kernel over the 4 HV virtual heads, FP32 parts of o, states in place;
  //    or the segmented prefill of the same virtual problem, with its workspace after ours
  if (segment_len < 0)
    st = la_internal::chunkwise(q, k, v, slopes_q, scale, h0 ? blocks : nullptr, slot_q, cu_seqlens, nullptr, part,
                                h_final ? blocks : nullptr, B, T, N, 2 * H, 4 * HV, 2 * HV, kHalf, N, false,
                                dev_error, stream, 2 * G, short_max);
  else
    st = la_internal::segmented_f32(q, k, v, slopes_q, scale, h0 ? blocks : nullptr, slot_q, cu_seqlens, part,
                                    h_final ? blocks : nullptr, B, T, N, 2 * H, 4 * HV, kHalf, N, segment_len,
                                    seg_bytes ? ws + l.bytes : nullptr, seg_bytes, dev_error, stream, 2 * G);
  if (st != LA_OK) return st;

  // 3. o = the sum over the key halves, rounded once; the final blocks to h_final
  if (tokens > 0) {
    SumParams sp{part, static_cast<__nv_bfloat16*>(o), cu_seqlens, state_indices, N, cu_seqlens ? 0 : T,
                 static_cast<int>(tokens), pool, HV, G, short_max};
    const int rgrid = static_cast<int>(tokens < 16 * ds->sms ? tokens : 16 * ds->sms);
    la_d256_sum_kernel<<<rgrid, kThreads, 0, s>>>(sp);
    if ((st = launched("d256 sum")) != LA_OK) return st;
  }
  if (h_final) {
    la_d256_blocks_kernel<false><<<bgrid, kThreads, 0, s>>>(bp);
    if ((st = launched("d256 scatter")) != LA_OK) return st;
  }
  return LA_OK;
}

}  // namespace la256

extern "C" {

la_status la_prefill_d256_workspace(int B, int T, int N, int HV, int has_state, size_t* bytes) {
  la_host::g_last_error[0] = '\0';
  if (!bytes) return la_host::fail(LA_ERR_INVALID_ARGUMENT, "bytes is null");
  if (B < 0 || T < 0 || N < 0 || HV <= 0)
    return la_host::fail(LA_ERR_INVALID_ARGUMENT, "B, T, N >= 0 and HV > 0 required");
  const int64_t tokens = static_cast<int64_t>(B) * T;
  if (tokens + 64 > INT32_MAX || static_cast<int64_t>(N) * 4 * HV > INT32_MAX)
    return la_host::fail(LA_ERR_UNSUPPORTED, "B*T or 4*N*HV too large");
  *bytes = la256::layout(tokens, N, HV, has_state != 0).bytes;
  return LA_OK;
}

la_status la_prefill_fwd_d256(const void* q, const void* k, const void* v, const float* slopes, float scale,
                              const float* h0, const int32_t* state_indices, const int32_t* cu_seqlens, void* o,
                              float* h_final, int B, int T, int N, int H, int HV, int D, int V, int pool_size,
                              void* workspace, size_t workspace_bytes, int* dev_error, void* stream) {
  using la_host::fail;
  la_host::g_last_error[0] = '\0';
  bool nothing = false;
  la_status st = la256::check_args(q, k, v, slopes, h0, state_indices, cu_seqlens, o, h_final, B, T, N, H, HV, D, V,
                                   pool_size, dev_error, &nothing);
  if (st != LA_OK || nothing) return st;
  const int64_t tokens = static_cast<int64_t>(B) * T;
  la_host::DeviceState* ds = nullptr;
  const int pool = la_host::effective_pool_size(h0, h_final, state_indices, pool_size, N);

  if (!cu_seqlens && T <= la256::kShortMax) {
    // short fixed-length sequences: the tokenwise recurrence on whole states, no workspace
    if ((st = la_host::check_prefill_disjoint(q, k, v, slopes, h0, state_indices, cu_seqlens, o, h_final, dev_error,
                                              B, T, N, H, HV, D, V, pool_size)) != LA_OK)
      return st;
    if ((st = la_host::current_device(la256::g_dev, &ds, la256::setup_kernels)) != LA_OK) return st;
    return la256::launch_tokenwise(q, k, v, slopes, scale, h0, state_indices, nullptr, o, h_final, T, N, H, HV, pool,
                                   tokens, ds, dev_error, stream);
  }

  return la256::blocks_path(q, k, v, slopes, scale, h0, state_indices, cu_seqlens, o, h_final, B, T, N, H, HV,
                            pool_size, -1, 0, workspace, workspace_bytes, dev_error, stream);
}

la_status la_prefill_d256_segmented_workspace(int B, int T, int N, int HV, int packed, int segment_len, int has_state,
                                              size_t* bytes, int* resolved_segment_len) {
  using la_host::fail;
  la_host::g_last_error[0] = '\0';
  if (!bytes) return fail(LA_ERR_INVALID_ARGUMENT, "bytes is null");
  if (B < 0 || T < 0 || N < 0 || HV <= 0) return fail(LA_ERR_INVALID_ARGUMENT, "B, T, N >= 0 and HV > 0 required");
  const int64_t tokens = static_cast<int64_t>(B) * T;
  if (tokens + 64 > INT32_MAX || static_cast<int64_t>(N) * 4 * HV > INT32_MAX)
    return fail(LA_ERR_UNSUPPORTED, "B*T or 4*N*HV too large");
  size_t seg = 0;
  int resolved = 0;
  const la_status st = la_prefill_segmented_workspace(B, T, N, 4 * HV, packed, segment_len, &seg, &resolved);
  if (st != LA_OK) return st;
  *bytes = la256::layout(tokens, N, HV, has_state != 0).bytes + seg;
  if (resolved_segment_len) *resolved_segment_len = resolved;
  return LA_OK;
}

la_status la_prefill_fwd_d256_segmented(const void* q, const void* k, const void* v, const float* slopes, float scale,
                                        const float* h0, const int32_t* state_indices, const int32_t* cu_seqlens,
                                        void* o, float* h_final, int B, int T, int N, int H, int HV, int D, int V,
                                        int pool_size, int segment_len, void* workspace, size_t workspace_bytes,
                                        int* dev_error, void* stream) {
  la_host::g_last_error[0] = '\0';
  bool nothing = false;
  la_status st = la256::check_args(q, k, v, slopes, h0, state_indices, cu_seqlens, o, h_final, B, T, N, H, HV, D, V,
                                   pool_size, dev_error, &nothing);
  if (st != LA_OK || nothing) return st;
  // the segmented workspace of the virtual problem (4 HV heads of 128); 0 when the plan has no
  // segments (every chain then runs whole, as in la_prefill_fwd_d256's block path)
  size_t seg = 0;
  int resolved = 0;
  if ((st = la_prefill_segmented_workspace(B, T, N, 4 * HV, cu_seqlens != nullptr, segment_len, &seg, &resolved)) !=
      LA_OK)
    return st;
  return la256::blocks_path(q, k, v, slopes, scale, h0, state_indices, cu_seqlens, o, h_final, B, T, N, H, HV,
                            pool_size, segment_len, seg, workspace, workspace_bytes, dev_error, stream);
}

}  // extern "C"
