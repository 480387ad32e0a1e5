// la_prefill_kernel.cuh -- sm_103a kernel for the Lightning Attention chunkwise prefill.
//
// What one (sequence n, value head hv) unit computes, chunk by chunk (C = 64 tokens,
// L = valid tokens of the chunk, s / j = token index inside the chunk), following the
// chunkwise form on page "[Lightning Attention] Add Hopper SM90 CuTe DSL prefill"
// (Description: FP32 recurrent state carried across 64-token chunks) and the closed
// form on page "[LA] Lightning Attention MTP decode + KVBuffer parallel verify /
// commit" (Description, term1 / term2):
//
//   A      = Q K^T                                  scores            [64 x 64]
//   P[s,j] = A[s,j] * lambda^(s-j)  (j <= s, j < L)  causal decay mask
//   O^T    = V^T P^T + (S Q^T) diag(lambda^(s+1))    intra + inter     [128 v x 64 s]
//   o      = scale * O                               stored as BF16, rows s < L
//   S     <- lambda^L S + V^T Kt,  Kt[j] = lambda^(L-1-j) k_j   state advance [128 v x 128 k]
//
// All four contractions run on the 5th-generation tensor cores (tcgen05.mma, BF16
// operands, FP32 accumulation in tensor memory).  The outputs are computed
// transposed (value dimension on the 128 TMEM lanes) so that every contraction except
// the scores has M = 128.  The decayed operands P, Kt and the FP32 state S are fed to
// the tensor cores as a BF16 pair hi + lo (hi = bf16(x), lo = bf16(x - hi)), so the
// products keep ~16 significant bits; only the final output is rounded to BF16 once.
//
// Warp-specialised pipeline, 512 threads per CTA, one CTA per SM:
//   warp 0       TMA producer: Q/K/V chunk tiles into a kStages-deep shared-memory ring
//   warp 1       TMEM allocator and the single MMA-issuing thread
//   warps 2-3    idle
//   warps 4-11   state warpgroups: thread (quadrant qd, lane) of warpgroup wg owns state
//                row v = 32 qd + lane, columns k in [64 wg, 64 wg + 64), in registers;
//                they advance the state and write the output of their half of the chunk
//   warps 12-15  operand warpgroup: builds the decayed BF16 hi/lo operands Kt and P
//
// Only the state advance and the inter-chunk MMA that reads it form a serial chain
// from chunk to chunk; scores, P, Kt, O_intra and Delta S of later chunks are built
// and multiplied ahead of it.  Per chunk i (a CTA-wide running chunk counter) the
// MMA thread issues, in order:
//   scores(i)    after stage i is loaded and the operand warpgroup read scores(i-1)
//   dS(i)        after Kt(i) is built and the state warpgroups read dS(i-1)
//   O_intra(i)   after P(i) is built and the state warpgroups read O(i-1)
//   O_inter(i)   after the state warpgroups wrote S(i) as hi/lo into TMEM
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace lap {

constexpr int kChunk = 64;        // tokens per chunk
constexpr int kDim = 128;         // D = V = 128
constexpr int kStages = 3;        // Q/K/V ring depth
constexpr int kThreads = 512;
constexpr int kStateThreads = 256;    // warps 4-11
constexpr int kOperandThreads = 128;  // warps 12-15
constexpr uint32_t kTileBytes = 8192;             // one 64 x 64 BF16 box (128-byte rows)
constexpr uint32_t kStageBytes = 6 * kTileBytes;  // Q, K, V: two boxes each

// TMEM column map (512 columns allocated, 128 lanes x 32 bit each)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColScores = 0;    // A = Q K^T, M = 64 accumulator, 64 columns
constexpr uint32_t kColOIntra = 64;   // (V^T P^T), lanes = v, 64 columns = s
constexpr uint32_t kColOInter = 128;  // (S Q^T),   lanes = v, 64 columns = s
constexpr uint32_t kColDeltaS = 256;  // V^T Kt,    lanes = v, 128 columns = k
constexpr uint32_t kColStateHi = 384; // S hi as MMA A operand: lanes = v, 64 columns = k pairs
constexpr uint32_t kColStateLo = 448; // S lo

constexpr int kLamStride = 68;  // floats per per-warp lambda^n table (65 used)

struct __align__(1024) StageTiles {
  uint8_t q[2][kTileBytes];  // [64 tokens][64 dims] x 2 halves of D, 128B-swizzled
  uint8_t k[2][kTileBytes];
  uint8_t v[2][kTileBytes];
};

struct __align__(1024) SharedStorage {
  StageTiles stage[kStages];
  uint8_t p_hi[2][kTileBytes];   // P [64 s][64 j], K-major B operand of O_intra, 2 buffers
  uint8_t p_lo[2][kTileBytes];
  uint8_t kt_hi[2][kTileBytes];  // Kt [64 j][128 k] (2 boxes of 64 k), MN-major B operand of dS
  uint8_t kt_lo[2][kTileBytes];
  float lam[12][kLamStride];     // per compute warp: lambda^n, n = 0..64, for that warp's current unit
  uint64_t full_bar[kStages];    // stage loaded (TMA transaction bytes)
  uint64_t empty_bar[kStages];   // stage consumed by every MMA that reads it
  uint64_t scores_full;          // MMA -> operand wg
  uint64_t scores_free;          // operand wg -> MMA
  uint64_t kt_ready;             // operand wg -> MMA
  uint64_t kt_free;              // MMA -> operand wg
  uint64_t p_ready[2];           // operand wg -> MMA
  uint64_t p_free[2];            // MMA -> operand wg
  uint64_t ds_full;              // MMA -> state wgs
  uint64_t ds_free;              // state wgs -> MMA
  uint64_t s_ready;              // state wgs -> MMA (S hi/lo written)
  uint64_t o_full;               // MMA -> state wgs (O_intra, O_inter done; S hi/lo free)
  uint64_t o_free;               // state wgs -> MMA
  uint64_t final_bar;            // every MMA retired (teardown)
  uint32_t tmem_base;
  int abort;
};

struct KernelParams {
  const float* slopes;
  const float* h0;
  const int32_t* state_indices;
  const int32_t* cu_seqlens;
  __nv_bfloat16* o;
  float* h_final;
  int* dev_error;
  float scale;
  int num_tokens;
  int T;          // fixed-length mode sequence length
  int N;          // sequences
  int H;          // q/k heads
  int HV;         // value heads
  int G;          // HV / H
  int pool_size;
  int num_units;  // N * HV
};

// One unit's sequence bounds, state slot and chunk count, decoded identically by every role.
struct Unit {
  int n, hv, hq;
  int bos, len, nchunks;
  int slot;   // -1: no state slot (padded sequence)
  int error;  // LA_DEV_ERR_* bits found while decoding
  bool run;   // false: skip (padded or invalid)
};

__device__ __forceinline__ Unit decode_unit(const KernelParams& p, int u) {
  Unit w;
  w.n = u / p.HV;
  w.hv = u - w.n * p.HV;
  w.hq = w.hv / p.G;
  w.error = 0;
  w.run = true;
  if (p.cu_seqlens) {
    const int b = __ldg(p.cu_seqlens + w.n), e = __ldg(p.cu_seqlens + w.n + 1);
    if (b < 0 || e < b || e > p.num_tokens) {
      w.error |= 1;  // LA_DEV_ERR_BAD_SEQLENS
      w.run = false;
      w.bos = 0;
      w.len = 0;
    } else {
      w.bos = b;
      w.len = e - b;
    }
  } else {
    w.bos = w.n * p.T;
    w.len = p.T;
  }
  w.slot = w.n;
  if (p.state_indices) {
    const int idx = __ldg(p.state_indices + w.n);
    if (idx >= p.pool_size) {
      w.error |= 2;  // LA_DEV_ERR_BAD_INDEX
      w.run = false;
    }
    if (idx < 0) w.run = false;  // padded sequence: nothing read or written
    w.slot = idx;
  }
  w.nchunks = (w.len + kChunk - 1) / kChunk;
  return w;
}

// Byte offset of 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t c) { return r * 128u + ((c ^ (r & 7u)) << 4); }

// Bounded wait whose result is the same on every lane of the warp, so the
// warp-collective tcgen05.ld / tcgen05.st that follow always see a converged warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

// lambda^n for n = 0..64 into the calling warp's own table; lambda^0 is exactly 1.
// Warp-local (two __syncwarp), so no role ever waits on another warp outside an mbarrier.
__device__ __forceinline__ void fill_lambda_table(float* tab, float slope, int lane) {
  __syncwarp();  // every lane is done with the previous unit's table
  for (int t = lane; t <= kChunk; t += 32) tab[t] = t == 0 ? 1.f : expf(-slope * static_cast<float>(t));
  __syncwarp();
}

// ------------------------------------------------------------------------------ roles

__device__ __forceinline__ void producer_loop(SharedStorage& sm, const KernelParams& p, const CUtensorMap* tm_q,
                                              const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                              volatile int* abort) {
  uint32_t it = 0;
  bool ok = true;
  for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
    const Unit w = decode_unit(p, u);
    if (!w.run) continue;
    for (int c = 0; c < w.nchunks; ++c, ++it) {
      const uint32_t st = it % kStages;
      if (!mbar_wait(&sm.empty_bar[st], ((it / kStages) & 1u) ^ 1u, abort)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(&sm.full_bar[st], kStageBytes);
      const int row = w.bos + c * kChunk;
      StageTiles& t = sm.stage[st];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        tma_load_2d(t.q[h], tm_q, &sm.full_bar[st], w.hq * kDim + 64 * h, row);
        tma_load_2d(t.k[h], tm_k, &sm.full_bar[st], w.hq * kDim + 64 * h, row);
        tma_load_2d(t.v[h], tm_v, &sm.full_bar[st], w.hv * kDim + 64 * h, row);
      }
    }
  }
  // Before leaving, make sure no load this thread issued is still writing shared memory.
  const uint32_t outstanding = it < kStages ? it : kStages;
  for (uint32_t i = 0; i < outstanding; ++i) {
    const uint32_t j = it - 1 - i;
    mbar_wait(&sm.full_bar[j % kStages], (j / kStages) & 1u, abort);
  }
}

__device__ __forceinline__ void mma_loop(SharedStorage& sm, const KernelParams& p, uint32_t tmem,
                                         volatile int* abort) {
  const uint32_t id_scores = idesc_bf16_f32(64, 64, false, false);   // Q (K-major) x K (K-major)
  const uint32_t id_ointra = idesc_bf16_f32(128, 64, true, false);   // V^T (MN-major) x P (K-major)
  const uint32_t id_ointer = idesc_bf16_f32(128, 64, false, false);  // S (TMEM) x Q (K-major)
  const uint32_t id_dstate = idesc_bf16_f32(128, 128, true, true);   // V^T (MN-major) x Kt (MN-major)
  const uint32_t kt_hi = smem_u32(sm.kt_hi), kt_lo = smem_u32(sm.kt_lo);
  uint32_t it = 0;
  bool ok = true;
  for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
    const Unit w = decode_unit(p, u);
    if (!w.run) continue;
    for (int c = 0; c < w.nchunks; ++c, ++it) {
      const uint32_t st = it % kStages;
      const uint32_t ph = it & 1u;
      const uint32_t pb = it & 1u;          // P buffer
      const uint32_t pph = (it >> 1) & 1u;  // its phase
      const uint32_t q0 = smem_u32(sm.stage[st].q), k0 = smem_u32(sm.stage[st].k);
      const uint32_t v0 = smem_u32(sm.stage[st].v);

      // scores A = Q K^T : M=64, N=64, K=128 (8 steps of 16)
      if (!mbar_wait(&sm.full_bar[st], (it / kStages) & 1u, abort) || !mbar_wait(&sm.scores_free, ph ^ 1u, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * kTileBytes + (kk & 3) * 32;
        mma_ss(tmem + kColScores, sdesc_sw128(q0 + off, 16, 1024), sdesc_sw128(k0 + off, 16, 1024), id_scores,
               kk > 0);
      }
      mma_commit(&sm.scores_full);

      // Delta S = V^T (Kt_hi + Kt_lo) : M=128, N=128, K=64
      if (!mbar_wait(&sm.kt_ready, ph, abort) || !mbar_wait(&sm.ds_free, ph ^ 1u, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const uint32_t kb = part ? kt_lo : kt_hi;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem + kColDeltaS, sdesc_sw128(v0 + kk * 2048, kTileBytes, 1024),
                 sdesc_sw128(kb + kk * 2048, kTileBytes, 1024), id_dstate, (part | kk) != 0);
      }
      mma_commit(&sm.ds_full);
      mma_commit(&sm.kt_free);

      // O_intra^T = V^T (P_hi + P_lo)^T : M=128, N=64, K=64
      if (!mbar_wait(&sm.p_ready[pb], pph, abort) || !mbar_wait(&sm.o_free, ph ^ 1u, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t p_hi = smem_u32(sm.p_hi[pb]), p_lo = smem_u32(sm.p_lo[pb]);
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const uint32_t pbase = part ? p_lo : p_hi;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem + kColOIntra, sdesc_sw128(v0 + kk * 2048, kTileBytes, 1024),
                 sdesc_sw128(pbase + kk * 32, 16, 1024), id_ointra, (part | kk) != 0);
      }

      // O_inter^T = (S_hi + S_lo) Q^T : M=128, N=64, K=128, A from TMEM
      if (!mbar_wait(&sm.s_ready, ph, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const uint32_t a0 = tmem + (part ? kColStateLo : kColStateHi);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kTileBytes + (kk & 3) * 32;
          mma_ts(tmem + kColOInter, a0 + kk * 8, sdesc_sw128(q0 + off, 16, 1024), id_ointer, (part | kk) != 0);
        }
      }
      mma_commit(&sm.o_full);
      mma_commit(&sm.p_free[pb]);
      mma_commit(&sm.empty_bar[st]);
    }
  }
  // Retire every MMA before the accumulators are released.
  mma_commit(&sm.final_bar);
  mbar_wait(&sm.final_bar, 0, abort);
}

// Operand warpgroup: Kt = lambda^(L-1-j) k_j and P = A * lambda^(s-j) (causal, tail masked), as BF16 hi/lo.
__device__ __forceinline__ void operand_loop(SharedStorage& sm, const KernelParams& p, uint32_t tmem, int otid,
                                             volatile int* abort) {
  const int warp = otid >> 5, lane = otid & 31;
  const int qd = warp & 3;  // TMEM lane quadrant (warps 12..15 -> 0..3)
  const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
  uint32_t it = 0;
  bool ok = true;
  for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
    const Unit w = decode_unit(p, u);
    if (!w.run) continue;
    float* lam = sm.lam[8 + warp];
    fill_lambda_table(lam, __ldg(p.slopes + w.hv), lane);
    for (int c = 0; c < w.nchunks; ++c, ++it) {
      const uint32_t st = it % kStages;
      const uint32_t ph = it & 1u;
      const uint32_t pb = it & 1u, pph = (it >> 1) & 1u;
      const int L = min(kChunk, w.len - c * kChunk);

      // ---- Kt: same swizzled layout as the K tile; thread -> row j, one of the two 64-column boxes
      if (!warp_wait(&sm.full_bar[st], (it / kStages) & 1u, abort) || !warp_wait(&sm.kt_free, ph ^ 1u, abort)) {
        ok = false;
        break;
      }
      {
        const int j = otid >> 1, box = otid & 1;
        const float wj = (j < L) ? lam[L - 1 - j] : 0.f;
        const uint8_t* ksrc = sm.stage[st].k[box];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          const uint32_t off = swz(j, cc);
          const uint4 kx = *reinterpret_cast<const uint4*>(ksrc + off);
          const uint32_t kw[4] = {kx.x, kx.y, kx.z, kx.w};
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split_bf16x2(wj * bf16lo_to_f32(kw[e]), wj * bf16hi_to_f32(kw[e]), hi[e], lo[e]);
          *reinterpret_cast<uint4*>(sm.kt_hi[box] + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(sm.kt_lo[box] + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&sm.kt_ready);

      // ---- P from the scores (M = 64 layout: row s in lane 32*(s/16) + s%16, lanes 16..31 unused)
      if (!warp_wait(&sm.scores_full, ph, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (!warp_wait(&sm.p_free[pb], pph ^ 1u, abort)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int gh = 0; gh < 2; ++gh) {  // columns j = 32 gh .. 32 gh + 31
        float a[2][16];
        tmem_ld16(tmem + lane_base + kColScores + 32 * gh, a[0]);
        tmem_ld16(tmem + lane_base + kColScores + 32 * gh + 16, a[1]);
        if (gh == 1) {
          tc_fence_before();
          mbar_arrive(&sm.scores_free);
        }
        if (lane < 16) {
          const int s = 16 * qd + lane;
#pragma unroll
          for (int g2 = 0; g2 < 2; ++g2) {  // 16 columns -> 16-byte chunks 2g, 2g+1
            const int g = 2 * gh + g2;
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int j0 = 16 * g + 2 * i, j1 = j0 + 1;
              const float p0 = (j0 <= s && j0 < L) ? a[g2][2 * i] * lam[max(s - j0, 0)] : 0.f;
              const float p1 = (j1 <= s && j1 < L) ? a[g2][2 * i + 1] * lam[max(s - j1, 0)] : 0.f;
              split_bf16x2(p0, p1, hi[i], lo[i]);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t off = swz(s, 2 * g + h);
              *reinterpret_cast<uint4*>(sm.p_hi[pb] + off) =
                  make_uint4(hi[4 * h], hi[4 * h + 1], hi[4 * h + 2], hi[4 * h + 3]);
              *reinterpret_cast<uint4*>(sm.p_lo[pb] + off) =
                  make_uint4(lo[4 * h], lo[4 * h + 1], lo[4 * h + 2], lo[4 * h + 3]);
            }
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&sm.p_ready[pb]);
    }
  }
}

// State warpgroups: own S in registers, advance it, feed it to the MMA as hi/lo, write the output.
__device__ __forceinline__ int state_loop(SharedStorage& sm, const KernelParams& p, uint32_t tmem, int ctid,
                                          volatile int* abort) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const int wg = warp >> 2;         // which half of k (state) and of s (output)
  const int qd = warp & 3;          // TMEM lane quadrant
  const int vrow = 32 * qd + lane;  // state row / output column v
  const int kbase = 64 * wg;
  const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
  float S[64];
  uint32_t it = 0;
  bool ok = true;
  int err = 0;

  auto write_state_operand = [&]() {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) split_bf16x2(S[32 * half + 2 * i], S[32 * half + 2 * i + 1], hi[i], lo[i]);
      tmem_st16(tmem + lane_base + kColStateHi + 32 * wg + 16 * half, hi);
      tmem_st16(tmem + lane_base + kColStateLo + 32 * wg + 16 * half, lo);
    }
  };

  for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
    const Unit w = decode_unit(p, u);
    err |= w.error;
    if (!w.run) continue;
    float* lam = sm.lam[warp];
    fill_lambda_table(lam, __ldg(p.slopes + w.hv), lane);

    // state gather
    const size_t state_off = ((static_cast<size_t>(w.slot) * p.HV + w.hv) * kDim + vrow) * kDim + kbase;
    if (p.h0) {
      const float4* src = reinterpret_cast<const float4*>(p.h0 + state_off);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 x = __ldg(src + i);
        S[4 * i] = x.x;
        S[4 * i + 1] = x.y;
        S[4 * i + 2] = x.z;
        S[4 * i + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 64; ++i) S[i] = 0.f;
    }
    if (w.nchunks > 0) {
      // S hi/lo is free: the previous unit's last O_inter was waited on (o_full) below
      write_state_operand();
      tc_fence_before();
      mbar_arrive(&sm.s_ready);
    }

    __nv_bfloat16* obase =
        p.o + static_cast<size_t>(w.bos) * p.HV * kDim + static_cast<size_t>(w.hv) * kDim + vrow;
    const size_t ostride = static_cast<size_t>(p.HV) * kDim;
    for (int c = 0; c < w.nchunks; ++c, ++it) {
      const uint32_t ph = it & 1u;
      const int L = min(kChunk, w.len - c * kChunk);

      // ---- S <- lambda^L S + Delta S
      if (!warp_wait(&sm.ds_full, ph, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        const float lamL = lam[L];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          float d[16];
          tmem_ld16(tmem + lane_base + kColDeltaS + kbase + 16 * q4, d);
#pragma unroll
          for (int i = 0; i < 16; ++i) S[16 * q4 + i] = fmaf(lamL, S[16 * q4 + i], d[i]);
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.ds_free);

      // ---- O(c) is complete and S(c) hi/lo has been read: publish S(c+1)
      if (!warp_wait(&sm.o_full, ph, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (c + 1 < w.nchunks) {
        write_state_operand();
        tc_fence_before();
        mbar_arrive(&sm.s_ready);
      }

      // ---- o = scale (O_intra + lambda^(s+1) O_inter), this warpgroup's 32 rows s
      {
        const float sc = p.scale;
        __nv_bfloat16* orow = obase + static_cast<size_t>(c) * kChunk * ostride;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float oi[16], oe[16];
          tmem_ld16(tmem + lane_base + kColOIntra + 32 * wg + 16 * half, oi);
          tmem_ld16(tmem + lane_base + kColOInter + 32 * wg + 16 * half, oe);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int s = 32 * wg + 16 * half + i;
            if (s < L) orow[s * ostride] = __float2bfloat16_rn(sc * fmaf(lam[s + 1], oe[i], oi[i]));
          }
        }
        tc_fence_before();
        mbar_arrive(&sm.o_free);
      }
    }
    if (!ok) break;
    // state scatter
    if (p.h_final) {
      float4* dst = reinterpret_cast<float4*>(p.h_final + state_off);
#pragma unroll
      for (int i = 0; i < 16; ++i) dst[i] = make_float4(S[4 * i], S[4 * i + 1], S[4 * i + 2], S[4 * i + 3]);
    }
  }
  return err;
}

__global__ void __launch_bounds__(kThreads, 1)
la_prefill_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const KernelParams p) {
  extern __shared__ uint8_t smem_raw[];
  SharedStorage& sm =
      *reinterpret_cast<SharedStorage*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  volatile int* abort = &sm.abort;

  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.full_bar[i], 1);
      mbar_init(&sm.empty_bar[i], 1);
    }
    mbar_init(&sm.scores_full, 1);
    mbar_init(&sm.scores_free, kOperandThreads);
    mbar_init(&sm.kt_ready, kOperandThreads);
    mbar_init(&sm.kt_free, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.p_ready[b], kOperandThreads);
      mbar_init(&sm.p_free[b], 1);
    }
    mbar_init(&sm.ds_full, 1);
    mbar_init(&sm.ds_free, kStateThreads);
    mbar_init(&sm.s_ready, kStateThreads);
    mbar_init(&sm.o_full, 1);
    mbar_init(&sm.o_free, kStateThreads);
    mbar_init(&sm.final_bar, 1);
    sm.abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    if (lane == 0) producer_loop(sm, p, &tm_q, &tm_k, &tm_v, abort);
  } else if (warp == 1) {
    if (lane == 0) mma_loop(sm, p, tmem, abort);
  } else if (warp >= 4 && warp < 12) {
    const int err = state_loop(sm, p, tmem, tid - 128, abort);
    if (err && tid == 128 && p.dev_error) atomicOr(p.dev_error, err);
  } else if (warp >= 12) {
    operand_loop(sm, p, tmem, tid - 384, abort);
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0 && sm.abort && p.dev_error) atomicOr(p.dev_error, 4);  // LA_DEV_ERR_TIMEOUT
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace lap
