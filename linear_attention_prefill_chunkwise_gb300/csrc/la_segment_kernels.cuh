// la_segment_kernels.cuh -- sm_103a kernels of the segmented-sequence prefill: long
// sequences are cut into segments of S tokens so that a batch with few (sequence, value
// head) chains still spreads over every SM.
//
// The recurrence of one chain is affine in its state: a segment of length L that starts
// from state H ends in lambda^L H + Sloc, where
//     Sloc = sum_{j<L} lambda^(L-1-j) v_j^T k_j          (the segment run from a zero state)
// depends only on the segment's own tokens.  This is the segmented affine scan that page
// "linear_attention: add a Hopper (sm90) KDA prefill path - #1017" (How) pairs with short
// chunks for another decayed recurrence, applied to Lightning Attention's scalar decay.
// The pipeline:
//   plan      one CTA: sequence bounds -> segment table (bounds, state slots, which segments
//             need a local state), device-side, so the host never reads cu_seqlens
//   state     la_segment_state_kernel: Sloc of every segment that is not the last of its
//             sequence, on the tensor cores: Sloc = V^T Kt with Kt_j = lambda^(L-1-j) k_j
//             over the whole segment (one accumulation, no per-chunk state update)
//   combine   la_segment_combine_kernel: H_0 = h0 (or 0), H_{i+1} = lambda^{L_i} H_i + Sloc_i,
//             written in place of Sloc_i as segment i's initial state
//   prefill   the chunkwise prefill kernel on the segments as a packed batch whose state
//             pool is this workspace (each segment reads its initial state, writes its final)
//   final     la_segment_final_kernel: the last segment's final state -> h_final
// Every segment's output is then the unsegmented output: the same chunkwise arithmetic, from
// the exact initial state up to FP32 rounding.
// The kernels are templated on the head dimension kD = D = V (128 or 64); the states in the
// workspace are [kD v][kD k].
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace las {

using lap::bf16x2_to_f2;
using lap::f2_mul;
using lap::f2_pack;
using lap::split_bf16x2;

constexpr int kChunk = 64;
constexpr uint32_t kTileBytes = 8192;  // one 64 x 64 BF16 box, 128-byte swizzled rows

// ---------------------------------------------------------------------------- plan

struct PlanParams {
  const int32_t* cu_seqlens;     // [N + 1] or null (fixed length T)
  const int32_t* state_indices;  // [N] or null
  int* dev_error;
  int32_t* seg_cu;     // [nseg_max + 1] segment boundaries (a packed batch of segments)
  int32_t* seg_slot;   // [nseg_max] g when segment g runs, else -1
  int32_t* seg_flags;  // [nseg_max] bit 0: needs its local state (not the last of its sequence)
  int32_t* seq_seg0;   // [N + 1] first segment of each sequence
  int32_t* seq_slot;   // [N] the sequence's state slot when it runs, else -1
  int N, T, tokens, S, nseg_max, pool_size;
  int S_last;  // > 0: each sequence's last segment is its last S_last tokens, the rest cut into S
};

constexpr int kPlanThreads = 1024;

// Sequence n owns max(1, ceil(L_n / S)) consecutive segments; segment j covers tokens
// [bos + j S, min(bos + (j + 1) S, eos)).  With S_last > 0 the last segment is the sequence's
// last min(L_n, S_last) tokens and the E = L_n - S_last before it (if any) are cut into
// ceil(E / S) segments of S from the start: short segments whose local states run in parallel,
// one long one that needs none.  A skipped sequence (padded, bad bounds, bad index)
// owns one segment with slot -1 so that the segment bounds stay one contiguous prefix array.
// Segment g's end is written by g itself (seg_cu[g + 1]), so every entry has one writer.
__global__ void __launch_bounds__(kPlanThreads, 1) la_segment_plan_kernel(const PlanParams p) {
  lap::griddep_wait();  // launched with programmatic stream serialization (la_host::launch_pdl)
  lap::griddep_launch_dependents();
  // 64-bit counts: with overlapping (invalid) bounds the segment counts can exceed int32
  __shared__ long long warp_tot[kPlanThreads / 32];
  __shared__ long long s_carry;
  __shared__ int s_first_over;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_carry = 0;
    s_first_over = INT32_MAX;
    int c0 = 0;
    if (p.cu_seqlens) c0 = min(max(__ldg(p.cu_seqlens), 0), p.tokens);
    p.seg_cu[0] = c0;
  }
  __syncthreads();
  int err = 0;
  for (int base = 0; base < p.N; base += kPlanThreads) {
    const int n = base + tid;
    int cnt = 0, bos = 0, len = 0, eos = 0, slot = -1;
    bool run = false;
    if (n < p.N) {
      bool bad = false;
      if (p.cu_seqlens) {
        const int b = __ldg(p.cu_seqlens + n), e = __ldg(p.cu_seqlens + n + 1);
        bad = b < 0 || e < b || e > p.tokens;
        if (bad) err |= 1;  // LA_DEV_ERR_BAD_SEQLENS
        bos = b;
        len = bad ? 0 : e - b;
        eos = min(max(e, 0), p.tokens);
      } else {
        bos = n * p.T;
        len = p.T;
        eos = bos + p.T;
      }
      slot = n;
      if (p.state_indices) {
        slot = __ldg(p.state_indices + n);
        if (slot >= p.pool_size) err |= 2;  // LA_DEV_ERR_BAD_INDEX
      }
      run = !bad && slot >= 0 && slot < p.pool_size;
      if (p.S_last > 0)
        cnt = run ? (max(len - p.S_last, 0) + p.S - 1) / p.S + 1 : 1;
      else
        cnt = run ? max(1, (len + p.S - 1) / p.S) : 1;
    }
    // exclusive scan of cnt over the block
    long long x = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
      long long t = warp_tot[lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, t, d);
        if (lane >= d) t += y;
      }
      warp_tot[lane] = t;  // inclusive over warps
    }
    __syncthreads();
    const long long carry = s_carry;
    const long long g0 = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + x - cnt;
    if (n < p.N) {
      const bool fits = g0 + cnt <= p.nseg_max;
      p.seq_seg0[n] = static_cast<int>(min(g0, static_cast<long long>(p.nseg_max)));
      if (!fits) {
        err |= 1;  // the bounds overlap: more segments than the batch's tokens allow
        if (g0 <= p.nseg_max) atomicMin(&s_first_over, static_cast<int>(g0));
        p.seq_slot[n] = -1;
      } else {
        p.seq_slot[n] = run ? slot : -1;
        for (int j = 0; j < cnt; ++j) {
          const int g = static_cast<int>(g0) + j;
          const bool last = j == cnt - 1;
          const int early_end = p.S_last > 0 ? min((j + 1) * p.S, len - p.S_last) : (j + 1) * p.S;
          p.seg_cu[g + 1] = last ? (run ? bos + len : eos) : bos + early_end;
          p.seg_slot[g] = run ? g : -1;
          p.seg_flags[g] = (run && !last) ? 1 : 0;
        }
      }
    }
    __syncthreads();
    if (tid == 0) s_carry = carry + warp_tot[kPlanThreads / 32 - 1];
    __syncthreads();
  }
  // segments written: a prefix [0, total)
  const int total = static_cast<int>(min(s_carry, static_cast<long long>(s_first_over)));
  if (tid == 0) p.seq_seg0[p.N] = min(total, p.nseg_max);
  __syncthreads();
  const int tail = p.seg_cu[min(total, p.nseg_max)];
  for (int g = total + tid; g < p.nseg_max; g += kPlanThreads) {
    p.seg_cu[g + 1] = tail;  // empty trailing segments
    p.seg_slot[g] = -1;
    p.seg_flags[g] = 0;
  }
  if (err && p.dev_error) atomicOr(p.dev_error, err);
}

// ---------------------------------------------------------------------------- local states

struct StateParams {
  const float* slopes;
  const int32_t* seg_cu;
  const int32_t* seg_flags;
  float* states;  // [nseg_max, HV, D v, D k]
  int* dev_error;
  int HV, G, num_units;  // num_units = nseg_max * HV, unit u = g * HV + hv
  // > 0: v's head of value head hv is hv with the digit of weight vfold dropped,
  // (hv / (2 vfold)) vfold + hv % vfold (the D = 256 decomposition; as the prefill kernel's)
  int vfold;
};

constexpr int kStStages = 4;          // K/V ring depth
constexpr int kStThreads = 512;
constexpr int kStBuildThreads = 256;  // warps 4..11: Kt builders
constexpr int kStEpiThreads = 128;    // warps 12..15: accumulator -> global
constexpr uint32_t kStTmemCols = 256; // two 128-column accumulators

struct __align__(1024) StateSmem {
  uint8_t k[kStStages][2][kTileBytes];  // K [64 tokens][64 dims] x 2 halves of D (D = 64: the first)
  uint8_t v[kStStages][2][kTileBytes];  // V [64 tokens][64 dims] x 2 halves of V (D = 64: the second zero)
  uint8_t kt_hi[2][2][kTileBytes];      // Kt hi/lo, 2 buffers, same layout as K (MN-major B operand)
  uint8_t kt_lo[2][2][kTileBytes];
  uint64_t full[kStStages];
  uint64_t empty[kStStages];
  uint64_t kt_ready[2];
  uint64_t kt_free[2];
  uint64_t acc_full[2];
  uint64_t acc_free[2];
  uint64_t final_bar;
  uint32_t tmem_base;
  int abort;
};

// The units that need a local state, walked identically by every role.
struct SegUnit {
  int g, hv, bos, len, nchunks;
};
__device__ __forceinline__ bool next_seg_unit(const StateParams& p, int& u, SegUnit& w) {
  for (; u < p.num_units; u += gridDim.x) {
    const int g = u / p.HV;
    if (!(__ldg(p.seg_flags + g) & 1)) continue;
    w.g = g;
    w.hv = u - g * p.HV;
    w.bos = __ldg(p.seg_cu + g);
    w.len = __ldg(p.seg_cu + g + 1) - w.bos;
    w.nchunks = (w.len + kChunk - 1) / kChunk;
    if (w.nchunks <= 0) continue;
    return true;
  }
  return false;
}

__device__ __forceinline__ uint32_t st_swz(uint32_t r, uint32_t c) { return r * 128u + ((c ^ (r & 7u)) << 4); }

__device__ __forceinline__ bool st_warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool ok = lap::mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

// Warp 0: TMA producer of the K and V chunk tiles (kD / 64 boxes of each).
template <int kD>
__device__ __forceinline__ void st_producer(StateSmem& sm, const StateParams& p, const CUtensorMap* tm_k,
                                            const CUtensorMap* tm_v, volatile int* abort) {
  constexpr int kBoxes = kD / 64;
  uint32_t it = 0;
  SegUnit w;
  for (int u = blockIdx.x; next_seg_unit(p, u, w); u += gridDim.x) {
    const int hq = w.hv / p.G;
    const int vh = p.vfold ? (w.hv / (2 * p.vfold)) * p.vfold + w.hv % p.vfold : w.hv;
    for (int c = 0; c < w.nchunks; ++c, ++it) {
      const uint32_t s = it % kStStages;
      if (!lap::mbar_wait(&sm.empty[s], ((it / kStStages) & 1u) ^ 1u, abort)) goto drain;
      lap::mbar_arrive_expect_tx(&sm.full[s], 2 * kBoxes * kTileBytes);
#pragma unroll
      for (int h = 0; h < kBoxes; ++h) {
        lap::tma_load_2d(sm.k[s][h], tm_k, &sm.full[s], hq * kD + 64 * h, w.bos + c * kChunk);
        lap::tma_load_2d(sm.v[s][h], tm_v, &sm.full[s], vh * kD + 64 * h, w.bos + c * kChunk);
      }
    }
  }
drain:
  // no copy may still be landing in shared memory when the CTA exits
  for (uint32_t i = 0; i < kStStages && i < it; ++i) {
    const uint32_t j = it - 1 - i;
    lap::mbar_wait_drain(&sm.full[j % kStStages], (j / kStStages) & 1u);
  }
}

// Warp 1, one thread: Sloc[acc] (+)= V^T Kt_hi + V^T Kt_lo, 8 MMAs (M = 128 v, N = kD k,
// K = 16 tokens each) per chunk.  With kD = 64, rows v >= 64 of the accumulator come from V's
// zeroed second box and are not read.
template <int kD>
__device__ __forceinline__ void st_mma(StateSmem& sm, const StateParams& p, uint32_t tmem, volatile int* abort) {
  constexpr uint32_t idesc = lap::idesc_bf16_f32(128, kD, true, true);
  const uint64_t dv0 = lap::sdesc_sw128(lap::smem_u32(sm.v[0]), kTileBytes, 1024);
  const uint64_t v_step = (2 * kTileBytes) >> 4;
  const uint64_t dhi0 = lap::sdesc_sw128(lap::smem_u32(sm.kt_hi[0]), kTileBytes, 1024);
  const uint64_t dlo0 = lap::sdesc_sw128(lap::smem_u32(sm.kt_lo[0]), kTileBytes, 1024);
  const uint64_t kt_step = (2 * kTileBytes) >> 4;
  uint32_t it = 0, ui = 0;
  SegUnit w;
  for (int u = blockIdx.x; next_seg_unit(p, u, w); u += gridDim.x, ++ui) {
    const uint32_t a = ui & 1u;
    if (!lap::mbar_wait(&sm.acc_free[a], ((ui >> 1) & 1u) ^ 1u, abort)) break;
    lap::tc_fence_after();
    const uint32_t d = tmem + a * 128;
    bool ok = true;
    for (int c = 0; c < w.nchunks; ++c, ++it) {
      const uint32_t s = it % kStStages, b = it & 1u;
      if (!lap::mbar_wait(&sm.kt_ready[b], (it >> 1) & 1u, abort) ||
          !lap::mbar_wait(&sm.full[s], (it / kStStages) & 1u, abort)) {
        ok = false;
        break;
      }
      lap::tc_fence_after();
      const uint64_t v0 = dv0 + s * v_step;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const uint64_t kt0 = (part ? dlo0 : dhi0) + b * kt_step;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          lap::mma_ss(d, v0 + ((kk * 2048) >> 4), kt0 + ((kk * 2048) >> 4), idesc, (c | part | kk) != 0);
      }
      lap::mma_commit(&sm.kt_free[b]);
      lap::mma_commit(&sm.empty[s]);
    }
    if (!ok) break;
    lap::mma_commit(&sm.acc_full[a]);
  }
  lap::mma_commit(&sm.final_bar);
  lap::mbar_wait_drain(&sm.final_bar, 0);  // every MMA retired before TMEM is released, also after an abort
}

// Warps 4..11: Kt_j = lambda^(L-1-j) k_j as a BF16 hi/lo pair, in the K tile's own swizzled
// layout (an elementwise map, so each 16-byte chunk keeps its position).  Thread bt owns
// token row bt % 64 of box (bt / 64) % 2 and its 16-byte chunks 4 (bt / 128) .. + 3; with
// kD = 64 the threads of box 1 have nothing to build but still take part in every phase.
template <int kD>
__device__ __forceinline__ void st_builder(StateSmem& sm, const StateParams& p, int bt, volatile int* abort) {
  const int row = bt & 63, box = (bt >> 6) & 1, c0 = 4 * (bt >> 7);
  const bool active = box < kD / 64;
  uint32_t it = 0;
  SegUnit w;
  for (int u = blockIdx.x; next_seg_unit(p, u, w); u += gridDim.x) {
    const float slope = __ldg(p.slopes + w.hv);
    for (int c = 0; c < w.nchunks; ++c, ++it) {
      const uint32_t s = it % kStStages, b = it & 1u;
      if (!st_warp_wait(&sm.full[s], (it / kStStages) & 1u, abort) ||
          !st_warp_wait(&sm.kt_free[b], ((it >> 1) & 1u) ^ 1u, abort))
        return;
      const int j = c * kChunk + row;  // token index inside the segment
      const uint8_t* src = sm.k[s][box];
      uint8_t* dhi = sm.kt_hi[b][box];
      uint8_t* dlo = sm.kt_lo[b][box];
      if (!active) {
      } else if (j < w.len) {
        const float wj = expf(-slope * static_cast<float>(w.len - 1 - j));
        const uint64_t w2 = f2_pack(wj, wj);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const uint32_t off = st_swz(row, c0 + cc);
          const uint4 kx = *reinterpret_cast<const uint4*>(src + off);
          const uint32_t kw[4] = {kx.x, kx.y, kx.z, kx.w};
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split_bf16x2(f2_mul(w2, bf16x2_to_f2(kw[e])), hi[e], lo[e]);
          *reinterpret_cast<uint4*>(dhi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(dlo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      } else {
        // Past the segment's end (segments that need a local state are whole chunks, so this
        // is defensive): Kt and V rows are zeroed rather than multiplied by zero, so that a
        // non-finite value of a neighbouring sequence cannot reach this state (0 * inf = NaN).
        uint8_t* vrow = sm.v[s][box] + row * 128;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const uint32_t off = st_swz(row, c0 + cc);
          *reinterpret_cast<uint4*>(dhi + off) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(dlo + off) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(vrow + 16 * (c0 + cc)) = make_uint4(0, 0, 0, 0);
        }
      }
      lap::fence_proxy_async_smem();
      lap::mbar_arrive(&sm.kt_ready[b]);
    }
  }
}

// Warps 12..15: accumulator rows (lane v) -> states[g][hv][v][:], 4 kD contiguous bytes per
// thread (with kD = 64 the warps of rows v >= 64 only take part in the barriers).
template <int kD>
__device__ __forceinline__ void st_epilogue(StateSmem& sm, const StateParams& p, uint32_t tmem, int et,
                                            volatile int* abort) {
  const int qd = et >> 5, lane = et & 31;
  const int vrow = 32 * qd + lane;
  const bool active = 32 * qd < kD;  // warp-uniform
  const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
  uint32_t ui = 0;
  SegUnit w;
  for (int u = blockIdx.x; next_seg_unit(p, u, w); u += gridDim.x, ++ui) {
    const uint32_t a = ui & 1u;
    if (!st_warp_wait(&sm.acc_full[a], (ui >> 1) & 1u, abort)) return;
    lap::tc_fence_after();
    if (active) {
      float4* dst = reinterpret_cast<float4*>(p.states + ((static_cast<size_t>(w.g) * p.HV + w.hv) * kD + vrow) * kD);
#pragma unroll 1
      for (int q = 0; q < kD / 16; ++q) {
        float r[16];
        lap::tmem_ld16(tmem + lane_base + a * 128 + 16 * q, r);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[4 * q + i] = make_float4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
      }
    }
    lap::tc_fence_before();
    lap::mbar_arrive(&sm.acc_free[a]);
  }
}

template <int kD>
__global__ void __launch_bounds__(kStThreads, 1)
la_segment_state_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const StateParams p) {
  static_assert(kD == 128 || kD == 64, "head dimension");
  lap::griddep_wait();  // launched with programmatic stream serialization (la_host::launch_pdl)
  lap::griddep_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  StateSmem& sm = *reinterpret_cast<StateSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort = &sm.abort;
  if (warp == 1) {
    lap::tmem_alloc(&sm.tmem_base, kStTmemCols);
    lap::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < kStStages; ++i) {
      lap::mbar_init(&sm.full[i], 1);
      lap::mbar_init(&sm.empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      lap::mbar_init(&sm.kt_ready[b], kStBuildThreads);
      lap::mbar_init(&sm.kt_free[b], 1);
      lap::mbar_init(&sm.acc_full[b], 1);
      lap::mbar_init(&sm.acc_free[b], kStEpiThreads);
    }
    lap::mbar_init(&sm.final_bar, 1);
    sm.abort = 0;
    lap::fence_mbar_init();
    lap::tma_prefetch_desc(&tm_k);
    lap::tma_prefetch_desc(&tm_v);
  }
  if constexpr (kD == 64) {
    // The MMAs read V as an M = 128 operand; with D = 64 its second box is never loaded and
    // must hold zeros for the whole kernel.
    for (int i = tid; i < kStStages * static_cast<int>(kTileBytes / 16); i += kStThreads) {
      const int st = i / static_cast<int>(kTileBytes / 16), e = i % static_cast<int>(kTileBytes / 16);
      reinterpret_cast<uint4*>(sm.v[st][1])[e] = make_uint4(0, 0, 0, 0);
    }
    lap::fence_proxy_async_smem();
  }
  lap::tc_fence_before();
  __syncthreads();
  lap::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    if (lane == 0) st_producer<kD>(sm, p, &tm_k, &tm_v, abort);
  } else if (warp == 1) {
    if (lane == 0) st_mma<kD>(sm, p, tmem, abort);
  } else if (warp >= 4 && warp < 12) {
    st_builder<kD>(sm, p, tid - 128, abort);
  } else if (warp >= 12) {
    st_epilogue<kD>(sm, p, tmem, tid - 384, abort);
  }

  lap::tc_fence_before();
  __syncthreads();
  if (tid == 0 && sm.abort && p.dev_error) atomicOr(p.dev_error, 4);  // LA_DEV_ERR_TIMEOUT
  if (warp == 1) {
    __syncwarp();
    lap::tc_fence_after();
    lap::tmem_dealloc(tmem, kStTmemCols);
  }
}

// ---------------------------------------------------------------------------- combine / final

struct CombineParams {
  const float* slopes;
  const float* h0;  // [P, HV, D, D] or null
  float* h_final;   // [P, HV, D, D] or null (final kernel)
  const int32_t* seg_cu;
  const int32_t* seq_seg0;
  const int32_t* seq_slot;
  float* states;  // [nseg_max, HV, D, D]
  int HV;
};

constexpr int kCombThreads = 256;
// CTAs per (sequence, head): comb_split x 256 threads = the float4 of a state (16 at D = 128)
template <int kD>
__host__ __device__ constexpr int comb_split() { return kD * kD / 4 / kCombThreads; }
constexpr int kCombBatch = 8;   // segments whose local states are loaded before they are chained

// grid (N * HV, comb_split): thread owns one float4 of the [kD x kD] state.
// H <- h0 (or 0); for each segment i of the sequence: states[i] <- H, then
// H <- lambda^{L_i} H + Sloc_i (Sloc_i read from states[i] before it is overwritten).
template <int kD>
__global__ void __launch_bounds__(kCombThreads) la_segment_combine_kernel(const CombineParams p) {
  lap::griddep_wait();  // launched with programmatic stream serialization (la_host::launch_pdl)
  lap::griddep_launch_dependents();
  const int n = blockIdx.x / p.HV, hv = blockIdx.x - n * p.HV;
  const int slot = __ldg(p.seq_slot + n);
  if (slot < 0) return;
  const int g0 = __ldg(p.seq_seg0 + n), g1 = __ldg(p.seq_seg0 + n + 1);
  const size_t e = static_cast<size_t>(blockIdx.y) * kCombThreads + threadIdx.x;  // float4 index
  constexpr size_t kState4 = kD * kD / 4;
  float4 H = make_float4(0.f, 0.f, 0.f, 0.f);
  if (p.h0) H = __ldg(reinterpret_cast<const float4*>(p.h0) + (static_cast<size_t>(slot) * p.HV + hv) * kState4 + e);
  const float slope = __ldg(p.slopes + hv);
  float4* st = reinterpret_cast<float4*>(p.states);
  for (int gb = g0; gb < g1; gb += kCombBatch) {
    float4 loc[kCombBatch];
#pragma unroll
    for (int j = 0; j < kCombBatch; ++j)
      if (gb + j < g1 - 1) loc[j] = st[(static_cast<size_t>(gb + j) * p.HV + hv) * kState4 + e];
#pragma unroll
    for (int j = 0; j < kCombBatch; ++j) {
      const int g = gb + j;
      if (g >= g1) break;
      st[(static_cast<size_t>(g) * p.HV + hv) * kState4 + e] = H;
      if (g < g1 - 1) {
        const float lamL = expf(-slope * static_cast<float>(__ldg(p.seg_cu + g + 1) - __ldg(p.seg_cu + g)));
        H.x = fmaf(lamL, H.x, loc[j].x);
        H.y = fmaf(lamL, H.y, loc[j].y);
        H.z = fmaf(lamL, H.z, loc[j].z);
        H.w = fmaf(lamL, H.w, loc[j].w);
      }
    }
  }
}

// grid (N * HV, comb_split): the final state of each running sequence's last segment,
// left in the workspace by the prefill, copied to h_final[slot].
template <int kD>
__global__ void __launch_bounds__(kCombThreads) la_segment_final_kernel(const CombineParams p) {
  lap::griddep_wait();  // launched with programmatic stream serialization (la_host::launch_pdl)
  lap::griddep_launch_dependents();
  const int n = blockIdx.x / p.HV, hv = blockIdx.x - n * p.HV;
  const int slot = __ldg(p.seq_slot + n);
  if (slot < 0) return;
  const int glast = __ldg(p.seq_seg0 + n + 1) - 1;
  const size_t e = static_cast<size_t>(blockIdx.y) * kCombThreads + threadIdx.x;
  constexpr size_t kState4 = kD * kD / 4;
  const float4 x = reinterpret_cast<const float4*>(p.states)[(static_cast<size_t>(glast) * p.HV + hv) * kState4 + e];
  reinterpret_cast<float4*>(p.h_final)[(static_cast<size_t>(slot) * p.HV + hv) * kState4 + e] = x;
}

}  // namespace las
