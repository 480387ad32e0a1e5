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
// All four contractions run on the 5th-generation tensor cores (tcgen05.mma, FP32
// accumulation in tensor memory).  The outputs are computed transposed (value
// dimension on the 128 TMEM lanes) so that every contraction except the scores has
// M = 128.  The inter-chunk decay lambda^(s+1) and the output scale are folded into a
// converted copy of Q, Qt[s] = scale lambda^(s+1) q_s, and the scale into P, so that
// O_inter and O_intra accumulate into one accumulator that already holds o.
// Operand precision:
//   scores   Q K^T           BF16 x BF16 (the inputs, exact)
//   O_inter  S Qt^T          TF32 x TF32: the FP32 state and Qt as stored (the tensor core
//                            reads the top 10 mantissa bits of each FP32 operand)
//   O_intra  V^T P^T         BF16 x (P_hi + P_lo): P as a BF16 pair, ~16 significant bits
//   dS       V^T Kt          BF16 x (Kt_hi + Kt_lo)
// Only the final output is rounded to BF16; the state itself stays FP32 throughout.
//
// Warp-specialised pipeline, 512 threads per CTA, one CTA per SM:
//   warp 0       TMA and MMA thread B, one polling loop: Q/K chunk tiles into a 2-stage ring,
//                V tiles into a 3-stage ring (the two rings refill independently), and the
//                scores and dS MMAs, each issued as soon as its operands are ready
//   warp 1       TMEM allocator and MMA thread A: O_inter(i) then O_intra(i), chunk by chunk
//                (tcgen05.mma issue stalls its thread while the tensor pipe is busy; with two
//                issuing threads one keeps the pipe fed while the other waits, tests a
//                barrier or commits, and the small MMAs of the two streams overlap)
//   warps 2-3    Q converter: BF16 Q tile -> Qt = scale lambda^(s+1) q in TF32 (B operand of
//                O_inter), 2 buffers
//   warps 4-11   state warpgroups: thread (quadrant qd, lane) of warpgroup wg owns state
//                row v = 32 qd + lane, columns k in [64 wg, 64 wg + 64), in registers;
//                they advance the state, publish it to TMEM and write the output: each warp
//                stages its 32 x 32 block of o as BF16 in the chunk's V stage (stmatrix) and
//                stores it with one TMA store (16-byte rows of the tile, not 2-byte scalars)
//   warps 12-15  operand warpgroup: builds the decayed BF16 hi/lo operands Kt and P
//
// Per chunk i (a CTA-wide running chunk counter) the MMA groups and their operands:
//   scores(i)    thread B, after stage i is loaded and scores(i-1) was read
//   dS(i)        thread B, after Kt(i) is built and the state warpgroups read dS(i-1)
//   O_inter(i)   thread A, into O[i%2], after S(i) is published, Qt(i) converted, O(i-2) read
//   O_intra(i)   thread A, accumulated into O[i%2], after P(i) is built
// The Q/K stage of chunk i is released as soon as its three readers (the scores MMAs, the
// Kt builders and the Qt converter) are done; a V stage after dS, O_intra and the output
// stores staged in it.
// Sequence isolation: the rows of a ragged chunk's tiles past the sequence's end belong to the
// next packed sequence; the operand warpgroup zeroes those K and V rows before any MMA that
// could mix them into this sequence reads them, and P is masked by a select.
// The serial chain from chunk to chunk is only: O_inter(i) done -> S(i+1) written to
// TMEM -> O_inter(i+1); everything else is built ahead of it.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace lap {

constexpr int kChunk = 64;        // tokens per chunk
constexpr int kDim = 128;         // largest head dimension D = V (the tile and TMEM layout)
constexpr int kQKStages = 2;      // Q/K ring depth (released early: after scores, Kt, Qt)
constexpr int kVStages = 3;       // V ring depth (held until O_intra)
constexpr int kThreads = 512;
constexpr int kConvThreads = 64;      // warps 2-3
constexpr int kStateThreads = 256;    // warps 4-11
constexpr int kOperandThreads = 128;  // warps 12-15
constexpr uint32_t kTileBytes = 8192;  // one 64 x 64 BF16 box (128-byte rows)

// TMEM column map (512 columns allocated, 128 lanes x 32 bit each)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColScores = 0;    // A = Q K^T, M = 64 accumulator, 64 columns
constexpr uint32_t kColO = 64;        // O^T = S Qt^T + V^T P^T, 2 buffers of 64 columns (lanes = v, columns = s)
constexpr uint32_t kColDeltaS = 256;  // V^T Kt, lanes = v, 128 columns = k
constexpr uint32_t kColState = 384;   // S (TF32) as the A operand of O_inter: lanes = v, 128 columns = k

constexpr int kTabStride = 68;  // per operand warp: lambda^n for n = 0..64

// Unit schedule of a packed batch (the kernel's kListed instance): sequences ranked by length
// at kernel start and their units dealt out longest first (see build_schedule).  The host uses
// it for batches of at most kSchedSeqMax sequences whose CTAs get at most kSchedMax units each;
// the other instance deals units out round robin.
constexpr int kSchedMax = 128;
constexpr int kSchedSeqMax = 256;

struct __align__(1024) QKTiles {
  uint8_t q[2][kTileBytes];  // [64 tokens][64 dims] x 2 halves of D, 128B-swizzled
  uint8_t k[2][kTileBytes];
};

struct __align__(1024) SharedStorage {
  QKTiles qk[kQKStages];
  uint8_t v[kVStages][2][kTileBytes];  // V [64 tokens][64 dims] x 2 halves, 128B-swizzled
  uint8_t qt[2][4][kTileBytes];  // Qt, TF32 [64 s][128 d] (4 boxes of 32 d), K-major B of O_inter; 2 buffers
  uint8_t p_hi[kTileBytes];      // P [64 s][64 j], K-major B operand of O_intra
  uint8_t p_lo[kTileBytes];
  uint8_t kt_hi[2][kTileBytes];  // Kt [64 j][128 k] (2 boxes of 64 k), MN-major B operand of dS
  uint8_t kt_lo[2][kTileBytes];
  float tab[4][kTabStride];      // per operand warp: lambda^n for its current unit
  uint64_t qk_full[kQKStages];   // Q/K stage loaded (TMA transaction bytes)
  uint64_t qk_empty[kQKStages];  // Q/K stage consumed: scores MMA commit + every Kt and Qt builder thread
  uint64_t v_full[kVStages];     // V stage loaded
  uint64_t v_empty[kVStages];    // V stage consumed: one commit from each MMA thread (dS, O_intra)
  uint64_t scores_full;          // MMA -> operand wg
  uint64_t scores_free;          // operand wg -> MMA
  uint64_t kt_ready;             // operand wg -> MMA
  uint64_t kt_free;              // MMA -> operand wg
  uint64_t p_ready;              // operand wg -> MMA
  uint64_t p_free;               // MMA -> operand wg
  uint64_t qt_ready[2];          // converter -> MMA
  uint64_t qt_free[2];           // MMA -> converter (O_inter done reading Qt)
  uint64_t ds_full;              // MMA -> state wgs
  uint64_t ds_free;              // state wgs -> MMA
  uint64_t s_ready;              // state wgs -> MMA (S written to TMEM)
  uint64_t s_free;               // MMA -> state wgs (O_inter done reading S)
  uint64_t o_full[2];            // MMA -> state wgs (O(i) complete)
  uint64_t o_free[2];            // state wgs -> MMA
  uint64_t final_bar[2];         // every MMA of thread A / B retired (teardown)            // every MMA retired (teardown)
  uint32_t tmem_base;
  int abort;
  int sched_n;                   // kListed: units listed in sched
  int32_t sched[kSchedMax];      // kListed: this CTA's units in processing order
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
  int HV;         // value heads (units, states and outputs per sequence)
  int G;          // HV / H
  int pool_size;
  int num_units;  // N * HV
  int short_max;  // sequences of at most this many tokens belong to the tokenwise kernel (-1: none)
  // kF32Out instance only: the FP32 output ([tokens, HV, D], the layout of o), and v's head of
  // value head hv: hv / vdiv (v then has HV / vdiv heads), or with vfold > 0 the index hv
  // with the digit of weight vfold dropped, (hv / (2 vfold)) vfold + hv % vfold (v then has
  // HV / 2 heads; the D = 256 decomposition, where that digit is the half of the key dimension)
  float* o_f32;
  int vdiv;
  int vfold;
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
      if (w.len <= p.short_max) w.run = false;  // run by the tokenwise kernel
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

// The calling warp's lambda^n table (n = 0..64, lambda^0 exactly 1) for a new unit.
// Warp-local (two __syncwarp), so no role ever waits on another warp outside an mbarrier.
__device__ __forceinline__ float* fill_lambda_table(SharedStorage& sm, int warp, int lane, float slope) {
  float* tab = sm.tab[warp];
  __syncwarp();  // every lane is done with the previous unit's table
  for (int t = lane; t <= kChunk; t += 32) tab[t] = t == 0 ? 1.f : expf(-slope * static_cast<float>(t));
  __syncwarp();
  return tab;
}

// The walk over this CTA's units, taken identically by every role: round robin (units
// blockIdx.x, blockIdx.x + gridDim.x, ...) or, in the kListed instance, the CTA's list.
template <bool kListed>
struct UnitWalk;
template <>
struct UnitWalk<false> {
  int u;
  __device__ __forceinline__ UnitWalk(const SharedStorage&, const KernelParams&) : u(blockIdx.x) {}
  __device__ __forceinline__ bool valid(const SharedStorage&, const KernelParams& p) const { return u < p.num_units; }
  __device__ __forceinline__ int unit(const SharedStorage&) const { return u; }
  __device__ __forceinline__ void next() { u += gridDim.x; }
};
template <>
struct UnitWalk<true> {
  int j, n;
  __device__ __forceinline__ UnitWalk(const SharedStorage& sm, const KernelParams&) : j(0), n(sm.sched_n) {}
  __device__ __forceinline__ bool valid(const SharedStorage&, const KernelParams&) const { return j < n; }
  __device__ __forceinline__ int unit(const SharedStorage& sm) const { return sm.sched[j]; }
  __device__ __forceinline__ void next() { ++j; }
};

// Number of chunks this CTA processes.
template <bool kListed>
__device__ __forceinline__ uint32_t cta_chunk_count(const SharedStorage& sm, const KernelParams& p) {
  uint32_t n = 0;
  for (UnitWalk<kListed> wk(sm, p); wk.valid(sm, p); wk.next()) {
    const Unit w = decode_unit(p, wk.unit(sm));
    if (w.run) n += w.nchunks;
  }
  return n;
}

// The packed batch's schedule (kListed instance), built by the whole CTA before the roles start
// (with CTA-wide barriers, before any role waits on anything).  Round robin over (sequence,
// head) units leaves some CTAs with the long sequences of a batch of random lengths; instead the
// sequences are ranked by length (ties by index; a sequence that will not run counts as empty)
// and the units in that order are dealt out in a snake: round j gives CTA b the unit of rank
// j G + b for even j and j G + G - 1 - b for odd j (G = gridDim.x).  Every CTA computes the
// same ranking from the same cu_seqlens, so each unit runs exactly once, and each unit's
// arithmetic does not depend on which CTA runs it.  The ranking's scratch is the Q conversion
// buffer, unused until the roles start.
__device__ __forceinline__ void build_schedule(SharedStorage& sm, const KernelParams& p, int tid) {
  const int G = gridDim.x, b = blockIdx.x;
  const int rounds = (p.num_units + G - 1) / G;  // <= kSchedMax (the host's condition)
  int32_t* len = reinterpret_cast<int32_t*>(sm.qt[0][0]);
  int32_t* by_rank = len + kSchedSeqMax;
  if (tid < p.N) {
    const int bb = __ldg(p.cu_seqlens + tid), ee = __ldg(p.cu_seqlens + tid + 1);
    int l = (bb >= 0 && ee >= bb && ee <= p.num_tokens) ? ee - bb : 0;
    if (l <= p.short_max) l = 0;
    if (p.state_indices && __ldg(p.state_indices + tid) < 0) l = 0;
    len[tid] = l;
  }
  __syncthreads();
  if (tid < p.N) {
    const int l = len[tid];
    int r = 0;
    for (int m = 0; m < p.N; ++m) {
      const int lm = len[m];
      r += (lm > l || (lm == l && m < tid)) ? 1 : 0;
    }
    by_rank[r] = tid;
  }
  __syncthreads();
  for (int j = tid; j < rounds; j += blockDim.x) {
    const int k = j * G + ((j & 1) ? G - 1 - b : b);
    sm.sched[j] = k < p.num_units ? by_rank[k / p.HV] * p.HV + k % p.HV : -1;
  }
  if (tid == 0) {
    const int jl = rounds - 1;
    const int kl = jl * G + ((jl & 1) ? G - 1 - b : b);
    sm.sched_n = kl < p.num_units ? rounds : rounds - 1;  // only the last round can run past the end
  }
}

// ------------------------------------------------------------------------------ roles

__device__ __forceinline__ uint64_t desc_at(uint64_t base, uint32_t byte_off) { return base + (byte_off >> 4); }

// Index in its sequence of a unit's c-th processed chunk: the chunks of a sequence run in order
// or, in the reverse instance (kRev), from the last to the first.  The partition into 64-token
// chunks is the same either way: only the sequence's last chunk can be ragged.
template <bool kRev>
__device__ __forceinline__ int seq_chunk(int c, int nchunks) { return kRev ? nchunks - 1 - c : c; }
template <bool kRev>
__device__ __forceinline__ int chunk_rows(const Unit& w, int c) {
  return min(kChunk, w.len - seq_chunk<kRev>(c, w.nchunks) * kChunk);
}

// The walk of this CTA's chunks by a role that runs ahead of the others.
template <bool kListed, bool kRev>
struct ChunkCursor {
  UnitWalk<kListed> wk;
  int c, row, hq, hv, nchunks;
  int tail;  // valid rows of the unit's last chunk (1..64)
  bool valid;
  // The current chunk ends inside its 64-row tiles: rows past the sequence's end are there.
  __device__ __forceinline__ bool ragged() const { return seq_chunk<kRev>(c, nchunks) == nchunks - 1 && tail < kChunk; }
};
template <bool kListed, bool kRev>
__device__ __forceinline__ void cursor_seek(const SharedStorage& sm, const KernelParams& p,
                                            ChunkCursor<kListed, kRev>& k) {
  for (; k.wk.valid(sm, p); k.wk.next()) {
    const Unit w = decode_unit(p, k.wk.unit(sm));
    if (w.run && w.nchunks > 0) {
      k.c = 0;
      k.row = w.bos + (kRev ? kChunk * (w.nchunks - 1) : 0);
      k.hq = w.hq;
      k.hv = w.hv;
      k.nchunks = w.nchunks;
      k.tail = w.len - kChunk * (w.nchunks - 1);
      k.valid = true;
      return;
    }
  }
  k.valid = false;
}
template <bool kListed, bool kRev>
__device__ __forceinline__ void cursor_next(const SharedStorage& sm, const KernelParams& p,
                                            ChunkCursor<kListed, kRev>& k) {
  if (++k.c < k.nchunks) {
    k.row += kRev ? -kChunk : kChunk;
  } else {
    k.wk.next();
    cursor_seek(sm, p, k);
  }
}

// TMA and MMA thread B, one polling loop: each pass issues, in this order, every job whose
// inputs are ready (mbarrier.test_wait, no blocking): dS(i) = V(i)^T Kt(i), scores(i) =
// Q(i) K(i)^T, and the next Q/K and V loads once their ring slots have been released.
template <bool kListed, int kD, bool kRev, bool kF32Out>
__device__ __forceinline__ void tma_mma_loop(SharedStorage& sm, const KernelParams& p, const CUtensorMap* tm_q,
                                             const CUtensorMap* tm_k, const CUtensorMap* tm_v, uint32_t tmem,
                                             volatile int* abort) {
  static_assert(kD == 64 || kD == 128, "head dimension");
  constexpr int kHalves = kD / 64;  // 64-wide boxes per head row
  constexpr uint32_t id_scores = idesc_bf16_f32(64, 64, false, false);
  constexpr uint32_t id_dstate = idesc_bf16_f32(128, kD, true, true);
  const uint64_t dq0 = sdesc_sw128(smem_u32(sm.qk[0].q), 16, 1024);
  const uint64_t dk0 = sdesc_sw128(smem_u32(sm.qk[0].k), 16, 1024);
  const uint64_t qk_step = sizeof(QKTiles) >> 4;
  const uint64_t dv0 = sdesc_sw128(smem_u32(sm.v[0]), kTileBytes, 1024);
  const uint64_t v_step = (2 * kTileBytes) >> 4;
  const uint64_t dkt_hi = sdesc_sw128(smem_u32(sm.kt_hi), kTileBytes, 1024);
  const uint64_t dkt_lo = sdesc_sw128(smem_u32(sm.kt_lo), kTileBytes, 1024);
  const uint32_t t_scores = tmem + kColScores, t_ds = tmem + kColDeltaS;
  const uint32_t total = cta_chunk_count<kListed>(sm, p);
  uint32_t n_ds = 0, n_sc = 0, nqk = 0, nv = 0;
  ChunkCursor<kListed, kRev> cq{UnitWalk<kListed>(sm, p)};
  cursor_seek(sm, p, cq);
  ChunkCursor<kListed, kRev> cv = cq;
  uint64_t last = globaltimer_ns();
  while (n_ds < total || n_sc < total || cq.valid || cv.valid) {
    bool progressed = false;
    if (n_ds < total) {
      const uint32_t j = n_ds, sv = j % kVStages;
      if (mbar_test(&sm.kt_ready, j & 1u) && mbar_test(&sm.v_full[sv], (j / kVStages) & 1u) &&
          mbar_test(&sm.ds_free, (j & 1u) ^ 1u)) {
        tc_fence_after();
        const uint64_t v0 = dv0 + sv * v_step;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(t_ds, desc_at(v0, kk * 2048), desc_at(part ? dkt_lo : dkt_hi, kk * 2048), id_dstate,
                   (part | kk) != 0);
        }
        mma_commit(&sm.ds_full);
        mma_commit(&sm.kt_free);
        mma_commit(&sm.v_empty[sv]);
        ++n_ds;
        progressed = true;
      }
    }
    if (n_sc < total) {
      const uint32_t j = n_sc, sq = j % kQKStages;
      if (mbar_test(&sm.qk_full[sq], (j / kQKStages) & 1u) && (j == 0 || mbar_test(&sm.scores_free, (j - 1) & 1u))) {
        tc_fence_after();
        const uint64_t q0 = dq0 + sq * qk_step, k0 = dk0 + sq * qk_step;
#pragma unroll
        for (int kk = 0; kk < 4 * kHalves; ++kk) {
          const uint32_t off = (kk >> 2) * kTileBytes + (kk & 3) * 32;
          mma_ss(t_scores, desc_at(q0, off), desc_at(k0, off), id_scores, kk > 0);
        }
        mma_commit(&sm.scores_full);
        mma_commit(&sm.qk_empty[sq]);
        ++n_sc;
        progressed = true;
      }
    }
    if (cq.valid) {
      const uint32_t sq = nqk % kQKStages;
      if (mbar_test(&sm.qk_empty[sq], ((nqk / kQKStages) & 1u) ^ 1u)) {
        // a ragged chunk's V tile lands on this stage's barrier as well (see the V load)
        mbar_arrive_expect_tx(&sm.qk_full[sq], (cq.ragged() ? 3 : 2) * kHalves * kTileBytes);
#pragma unroll
        for (int h = 0; h < kHalves; ++h) {
          tma_load_2d(sm.qk[sq].q[h], tm_q, &sm.qk_full[sq], cq.hq * kD + 64 * h, cq.row);
          tma_load_2d(sm.qk[sq].k[h], tm_k, &sm.qk_full[sq], cq.hq * kD + 64 * h, cq.row);
        }
        ++nqk;
        cursor_next(sm, p, cq);
        progressed = true;
      }
    }
    if (cv.valid) {
      const uint32_t sv = nv % kVStages;
      // The V tile of a ragged chunk holds rows of the next packed sequence past the end.  The
      // operand warpgroup zeroes them before any MMA reads the tile: the tile lands on the Q/K
      // stage's barrier, which the operand warpgroup waits on anyway (so its Q/K load must have
      // been issued, with these bytes in its expected count), and v_full's phase is completed
      // by a plain arrival; dS and O_intra read the tile only after kt_ready / p_ready, which
      // the operand warpgroup gives after the zeroing.
      const bool ragged = cv.ragged();
      if (mbar_test(&sm.v_empty[sv], ((nv / kVStages) & 1u) ^ 1u) && (!ragged || nqk > nv)) {
        uint64_t* bar = &sm.v_full[sv];
        if (ragged) {
          mbar_arrive(bar);
          bar = &sm.qk_full[nv % kQKStages];
        } else {
          mbar_arrive_expect_tx(bar, kHalves * kTileBytes);
        }
        // (the kF32Out instance may share a V head among vdiv value heads, or fold two onto one)
        const int vh = !kF32Out ? cv.hv : p.vfold ? (cv.hv / (2 * p.vfold)) * p.vfold + cv.hv % p.vfold : cv.hv / p.vdiv;
#pragma unroll
        for (int h = 0; h < kHalves; ++h) tma_load_2d(sm.v[sv][h], tm_v, bar, vh * kD + 64 * h, cv.row);
        ++nv;
        cursor_next(sm, p, cv);
        progressed = true;
      }
    }
    if (progressed) {
      last = globaltimer_ns();
    } else {
      if (*abort) break;
      if (globaltimer_ns() - last > kWaitLimitNs) {
        *abort = 1;
        break;
      }
      __nanosleep(32);
    }
  }
  // Teardown, also after an abort: every load issued has landed and every MMA issued has
  // retired before the CTA releases its shared and tensor memory.  A load is issued only
  // after the previous one into its slot was consumed, so the last loads of each ring are the
  // only ones that can still be in flight.
  for (uint32_t i = 0; i < kQKStages && i < nqk; ++i) {
    const uint32_t j = nqk - 1 - i;
    mbar_wait_drain(&sm.qk_full[j % kQKStages], (j / kQKStages) & 1u);
  }
  for (uint32_t i = 0; i < kVStages && i < nv; ++i) {
    const uint32_t j = nv - 1 - i;
    mbar_wait_drain(&sm.v_full[j % kVStages], (j / kVStages) & 1u);
  }
  mma_commit(&sm.final_bar[1]);
  mbar_wait_drain(&sm.final_bar[1], 0);
}

// MMA thread A: the output accumulator, in chunk order, with blocking waits (this is the
// serial chain of the pipeline):
//   O_inter(i) = S(i) Qt(i)^T     into O[i%2]: needs Qt(i), O(i-2) read out, S(i) published
//   O_intra(i) += V(i)^T P(i)^T   needs V(i) and P(i); after O_inter(i) (same thread, in order)
template <bool kListed, int kD>
__device__ __forceinline__ void mma_o_loop(SharedStorage& sm, const KernelParams& p, uint32_t tmem,
                                           volatile int* abort) {
  constexpr uint32_t id_ointer = idesc_tf32_f32(128, 64, false, false);
  constexpr uint32_t id_ointra = idesc_bf16_f32(128, 64, true, false);
  const uint64_t dv0 = sdesc_sw128(smem_u32(sm.v[0]), kTileBytes, 1024);
  const uint64_t v_step = (2 * kTileBytes) >> 4;
  const uint64_t dqt0 = sdesc_sw128(smem_u32(sm.qt[0]), 16, 1024);
  const uint64_t qt_step = (4 * kTileBytes) >> 4;
  const uint64_t dp_hi = sdesc_sw128(smem_u32(sm.p_hi), 16, 1024);
  const uint64_t dp_lo = sdesc_sw128(smem_u32(sm.p_lo), 16, 1024);
  const uint32_t t_state = tmem + kColState;
  const uint32_t total = cta_chunk_count<kListed>(sm, p);
  for (uint32_t it = 0; it < total; ++it) {
    const uint32_t sv = it % kVStages, ph = it & 1u, b = it & 1u, bph = (it >> 1) & 1u;
    if (!mbar_wait(&sm.qt_ready[b], bph, abort) || !mbar_wait(&sm.o_free[b], bph ^ 1u, abort) ||
        !mbar_wait(&sm.s_ready, ph, abort))
      break;
    tc_fence_after();
    const uint32_t t_o = tmem + kColO + 64 * b;
    const uint64_t qt0 = dqt0 + b * qt_step;
#pragma unroll 4
    for (int kk = 0; kk < kD / 8; ++kk) {
      const uint32_t off = (kk >> 2) * kTileBytes + (kk & 3) * 32;
      mma_tf32_ts(t_o, t_state + kk * 8, desc_at(qt0, off), id_ointer, kk > 0);
    }
    mma_commit(&sm.s_free);
    mma_commit(&sm.qt_free[b]);
    if (!mbar_wait(&sm.v_full[sv], (it / kVStages) & 1u, abort) || !mbar_wait(&sm.p_ready, ph, abort)) break;
    tc_fence_after();
    const uint64_t v0 = dv0 + sv * v_step;
#pragma unroll
    for (int part = 0; part < 2; ++part) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ss(t_o, desc_at(v0, kk * 2048), desc_at(part ? dp_lo : dp_hi, kk * 32), id_ointra, 1);
    }
    mma_commit(&sm.o_full[b]);
    mma_commit(&sm.p_free);
    mma_commit(&sm.v_empty[sv]);
  }
  mma_commit(&sm.final_bar[0]);
  mbar_wait_drain(&sm.final_bar[0], 0);  // every MMA of this thread retired, also after an abort
}

// Q converter (warps 2-3): the BF16 Q tile (K-major, 128B-swizzled, 2 boxes of 64 d) into
// Qt = scale lambda^(s+1) q in FP32 (K-major, 128B-swizzled, 4 boxes of 32 d), which the
// tensor core reads as TF32, i.e. truncated to 10 mantissa bits; rounding it here instead
// would cost two more instructions per element on the critical conversion and changes the
// output by far less than its BF16 step.  Thread t owns token row s = t of the chunk.
template <bool kListed, int kD, bool kRev>
__device__ __forceinline__ void convert_loop(SharedStorage& sm, const KernelParams& p, int ctid,
                                             volatile int* abort) {
  const int s = ctid;
  uint32_t it = 0;
  bool ok = true;
  for (UnitWalk<kListed> wk(sm, p); wk.valid(sm, p) && ok; wk.next()) {
    const Unit w = decode_unit(p, wk.unit(sm));
    if (!w.run) continue;
    // scale lambda^(s+1): row s is s + 1 tokens past the state; in the reverse instance the state
    // enters a chunk of L tokens after its last one, L - s tokens from row s (rows s >= L are
    // never stored: 0)
    const float slope = __ldg(p.slopes + w.hv);
    const float f = p.scale * expf(-slope * static_cast<float>(kRev ? kChunk - s : s + 1));
    const float ftail = kRev && s < w.len - kChunk * (w.nchunks - 1)
                            ? p.scale * expf(-slope * static_cast<float>(w.len - kChunk * (w.nchunks - 1) - s))
                            : 0.f;
    for (int c = 0; c < w.nchunks; ++c, ++it) {
      const float fc = (kRev && chunk_rows<kRev>(w, c) < kChunk) ? ftail : f;
      const uint64_t ff = f2_pack(fc, fc);
      const uint32_t sq = it % kQKStages, qph = (it / kQKStages) & 1u;
      const uint32_t b = it & 1u, bph = (it >> 1) & 1u;
      if (!warp_wait(&sm.qk_full[sq], qph, abort) || !warp_wait(&sm.qt_free[b], bph ^ 1u, abort)) {
        ok = false;
        break;
      }
#pragma unroll 1
      for (int h = 0; h < kD / 64; ++h) {
#pragma unroll 2
        for (int cc = 0; cc < 8; ++cc) {
          const uint4 x = *reinterpret_cast<const uint4*>(sm.qk[sq].q[h] + swz(s, cc));
          uint8_t* dst = sm.qt[b][2 * h + (cc >> 2)];
          const uint32_t fc = 2 * (cc & 3);
          const float2 q0 = f2_unpack(f2_mul(ff, bf16x2_to_f2(x.x))), q1 = f2_unpack(f2_mul(ff, bf16x2_to_f2(x.y)));
          const float2 q2 = f2_unpack(f2_mul(ff, bf16x2_to_f2(x.z))), q3 = f2_unpack(f2_mul(ff, bf16x2_to_f2(x.w)));
          *reinterpret_cast<float4*>(dst + swz(s, fc)) = make_float4(q0.x, q0.y, q1.x, q1.y);
          *reinterpret_cast<float4*>(dst + swz(s, fc + 1)) = make_float4(q2.x, q2.y, q3.x, q3.y);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&sm.qt_ready[b]);
      mbar_arrive(&sm.qk_empty[sq]);
    }
  }
}

// Operand warpgroup: Kt = lambda^(L-1-j) k_j and P = A * lambda^(s-j) (causal, tail masked), as BF16 hi/lo;
// in the reverse instance Kt = lambda^j k_j and P = A * lambda^(j-s) for j >= s (the recurrence
// run from a chunk's last token to its first).
template <bool kListed, int kD, bool kRev>
__device__ __forceinline__ void operand_loop(SharedStorage& sm, const KernelParams& p, uint32_t tmem, int otid,
                                             volatile int* abort) {
  const int warp = otid >> 5, lane = otid & 31;
  const int qd = warp;                     // TMEM lane quadrant (warps 12..15 -> 0..3)
  const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
  const int prow = 16 * qd + (lane & 15);  // P: score row s of this thread
  const int pcol = 32 * (lane >> 4);       //    and its first column j
  const int krow = otid & 63;              // Kt: token row j of this thread
  const int kbox = otid >> 6;              //     and its 64-column box of k
  uint32_t it = 0;
  bool ok = true;
  for (UnitWalk<kListed> wk(sm, p); wk.valid(sm, p) && ok; wk.next()) {
    const Unit w = decode_unit(p, wk.unit(sm));
    if (!w.run) continue;
    const float* lam = fill_lambda_table(sm, warp, lane, __ldg(p.slopes + w.hv));
    // decay row of P for this thread: scale lambda^(s-j) for j <= s, 0 above the diagonal
    float drow[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (kRev)
        drow[i] = (pcol + i >= prow) ? p.scale * lam[max(pcol + i - prow, 0)] : 0.f;
      else
        drow[i] = (pcol + i <= prow) ? p.scale * lam[max(prow - pcol - i, 0)] : 0.f;
    }
    for (int c = 0; c < w.nchunks; ++c, ++it) {
      const uint32_t sq = it % kQKStages, qph = (it / kQKStages) & 1u;
      const uint32_t ph = it & 1u;
      const int L = chunk_rows<kRev>(w, c);

      // ---- Kt: same swizzled layout as the K tile
      if (!warp_wait(&sm.qk_full[sq], qph, abort) || !warp_wait(&sm.kt_free, ph ^ 1u, abort)) {
        ok = false;
        break;
      }
      // (with D = 64 the second 64-column box of K, V and Kt is unused: V's stays zero, see the
      // kernel's prologue, and the dS MMA has N = 64)
      if (kD == 128 || kbox == 0) {
        if (krow >= L) {
          // Rows j >= L of a ragged chunk belong to the next packed sequence (or are the TMA's zero
          // fill): this thread's K row and V row are zeroed, so that a non-finite value there cannot
          // reach this sequence (0 * inf is NaN); the V tile of a ragged chunk has landed with the
          // Q/K stage.
          uint8_t* kr = sm.qk[sq].k[kbox] + krow * 128;
          uint8_t* vr = sm.v[it % kVStages][kbox] + krow * 128;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            *reinterpret_cast<uint4*>(kr + 16 * cc) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(vr + 16 * cc) = make_uint4(0, 0, 0, 0);
          }
        }
        {
          const float wjf = (krow < L) ? lam[kRev ? krow : L - 1 - krow] : 0.f;
          const uint64_t wj = f2_pack(wjf, wjf);
          const uint8_t* ksrc = sm.qk[sq].k[kbox];
#pragma unroll 2
          for (int cc = 0; cc < 8; ++cc) {
            const uint32_t off = swz(krow, cc);
            const uint4 kx = *reinterpret_cast<const uint4*>(ksrc + off);
            const uint32_t kw[4] = {kx.x, kx.y, kx.z, kx.w};
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) split_bf16x2(f2_mul(wj, bf16x2_to_f2(kw[e])), hi[e], lo[e]);
            *reinterpret_cast<uint4*>(sm.kt_hi[kbox] + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(sm.kt_lo[kbox] + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&sm.kt_ready);
      mbar_arrive(&sm.qk_empty[sq]);

      // ---- P from the scores: row prow, columns pcol .. pcol + 31 (16x32bx2 loads use all 32 lanes)
      if (!warp_wait(&sm.scores_full, ph, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float a[2][16];
      tmem_ld16_x2split32(tmem + lane_base + kColScores, a[0]);
      tmem_ld16_x2split32(tmem + lane_base + kColScores + 16, a[1]);
      tc_fence_before();
      mbar_arrive(&sm.scores_free);
      if (!warp_wait(&sm.p_free, ph ^ 1u, abort)) {
        ok = false;
        break;
      }
      {
        const bool full = (L == kChunk);
#pragma unroll
        for (int g = 0; g < 2; ++g) {  // 16 columns -> 16-byte chunks (pcol/8) + 2g, +1
          uint32_t hi[8], lo[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int i0 = 16 * g + 2 * i;
            uint64_t pp = f2_mul(f2_pack(a[g][2 * i], a[g][2 * i + 1]), f2_pack(drow[i0], drow[i0 + 1]));
            if (!full) {
              const float2 v = f2_unpack(pp);
              pp = f2_pack((pcol + i0 < L) ? v.x : 0.f, (pcol + i0 + 1 < L) ? v.y : 0.f);
            }
            split_bf16x2(pp, hi[i], lo[i]);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t off = swz(prow, (pcol >> 3) + 2 * g + h);
            *reinterpret_cast<uint4*>(sm.p_hi + off) = make_uint4(hi[4 * h], hi[4 * h + 1], hi[4 * h + 2], hi[4 * h + 3]);
            *reinterpret_cast<uint4*>(sm.p_lo + off) = make_uint4(lo[4 * h], lo[4 * h + 1], lo[4 * h + 2], lo[4 * h + 3]);
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&sm.p_ready);
    }
  }
}

// State warpgroups: own S in registers, advance it, publish it to TMEM, write the output.
template <bool kListed, int kD, bool kRev, bool kF32Out>
__device__ __forceinline__ int state_loop(SharedStorage& sm, const KernelParams& p, const CUtensorMap* tm_o,
                                          uint32_t tmem, int ctid, volatile int* abort) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const int wg = warp >> 2;         // which half of k (state) and of s (output)
  const int qd = warp & 3;          // TMEM lane quadrant
  const int vrow = 32 * qd + lane;  // state row / output column v
  const int kbase = 64 * wg;
  // With D = 64 only rows v < 64 and columns k < 64 of the 128 x 128 layout hold the state: the
  // second warpgroup's columns are never read (O_inter has K = 64), rows v >= 64 stay zero.
  const bool k_live = kD == 128 || wg == 0;
  const bool state_live = kD == 128 || (wg == 0 && qd < 2);
  const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
  float S[64];
  uint32_t it = 0;
  bool ok = true;
  int err = 0;

  // S into its TMEM columns (the TF32 MMA reads its top 10 mantissa bits), then tell the MMA thread.
  auto publish_state = [&]() {
    if (k_live) {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t u[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) u[i] = __float_as_uint(S[16 * q4 + i]);
        tmem_st16(tmem + lane_base + kColState + kbase + 16 * q4, u);
      }
    }
    tc_fence_before();
    mbar_arrive(&sm.s_ready);
  };

  for (UnitWalk<kListed> wk(sm, p); wk.valid(sm, p) && ok; wk.next()) {
    const Unit w = decode_unit(p, wk.unit(sm));
    err |= w.error;
    if (!w.run) continue;
    const float slope = __ldg(p.slopes + w.hv);
    const float lam_chunk = expf(-slope * static_cast<float>(kChunk));  // lambda^64

    // state gather
    const size_t state_off = ((static_cast<size_t>(w.slot) * p.HV + w.hv) * kD + vrow) * kD + kbase;
    if (p.h0 && state_live) {
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
    // The state's TMEM columns are free: the previous chunk's s_free was waited on below.
    if (w.nchunks > 0) publish_state();

    const size_t ostride = static_cast<size_t>(p.HV) * kD;
    for (int c = 0; c < w.nchunks; ++c, ++it) {
      const uint32_t ph = it & 1u;
      const uint32_t b = it & 1u, bph = (it >> 1) & 1u;
      const int L = chunk_rows<kRev>(w, c);

      // ---- S(i+1) = lambda^L S(i) + Delta S(i), in registers
      if (!warp_wait(&sm.ds_full, ph, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        const float lamLf = (L == kChunk) ? lam_chunk : expf(-slope * static_cast<float>(L));
        const uint64_t lamL = f2_pack(lamLf, lamLf);
        if (k_live) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            float d[16];
            tmem_ld16(tmem + lane_base + kColDeltaS + kbase + 16 * q4, d);
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              const float2 r =
                  f2_unpack(f2_fma(lamL, f2_pack(S[16 * q4 + i], S[16 * q4 + i + 1]), f2_pack(d[i], d[i + 1])));
              S[16 * q4 + i] = r.x;
              S[16 * q4 + i + 1] = r.y;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.ds_free);

      // ---- O_inter(i) has read S(i): publish S(i+1)
      if (!warp_wait(&sm.s_free, ph, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (c + 1 < w.nchunks) publish_state();

      // ---- o = O (the scale is folded into Qt and P): this warp's 32 rows s x 32 values v of the
      //      chunk, staged as BF16 in the chunk's V stage (dS and O_intra, its readers, are done:
      //      ds_full and o_full were waited on) and stored by one TMA store of a 32 x 32 box.
      if (!warp_wait(&sm.o_full[b], bph, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if constexpr (kF32Out) {
        // FP32 output (per-value-head partial sums that the caller adds up): each thread stores the
        // values tcgen05.ld 16x256b gives it, value rows v = 32 qd + 16 g + lane / 4 (+ 8) and
        // token rows s = 32 wg + 8 r + 2 (lane % 4) (+ 1) of the chunk, rows s < L only
        const int ybase = w.bos + seq_chunk<kRev>(c, w.nchunks) * kChunk;
        const bool vlive = kD == 128 || qd < 2;
        float* obase = p.o_f32 + static_cast<size_t>(w.hv) * kD;
#pragma unroll 1
        for (int g = 0; g < 2; ++g) {
          uint32_t rg[16];
          tmem_ld_16x256b_x4(tmem + lane_base + (static_cast<uint32_t>(16 * g) << 16) + kColO + 64 * b + 32 * wg, rg);
          if (g == 1) {
            tc_fence_before();
            mbar_arrive(&sm.o_free[b]);
          }
          if (vlive) {
            const int v1 = 32 * qd + 16 * g + (lane >> 2);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int sl = 32 * wg + 8 * r + 2 * (lane & 3) + e;
                if (sl < L) {
                  float* orow = obase + static_cast<size_t>(ybase + sl) * ostride;
                  orow[v1] = __uint_as_float(rg[4 * r + e]);
                  orow[v1 + 8] = __uint_as_float(rg[4 * r + 2 + e]);
                }
              }
            }
          }
        }
        if (lane == 0) mbar_arrive(&sm.v_empty[it % kVStages]);
      } else {
        const uint32_t sv = it % kVStages;
        // 32 rows of 64 bytes, 64-byte swizzle (D = 64: the four warps with v < 64, in the half of
        // the stage the V loads use)
        uint8_t* stage = sm.v[sv][0] + (wg * (kD / 32) + qd) * 2048;
        // valid rows of this warp's box (may be <= 0 or > 32); none for values v >= D
        const int rows = (kD == 128 || qd < 2) ? L - 32 * wg : 0;
        // stmatrix.trans: lane l gives row j = l % 8 of matrix m = l / 8; the matrices of one call
        // are (repetition rr, value half h) = (2 k2 + m / 2, m % 2): row sl = 8 rr + j of the box,
        // 16-byte chunk 2 g + h (lanes 16 g .. 16 g + 15 of this warp's quadrant)
        const int m = lane >> 3, j = lane & 7;
#pragma unroll 1
        for (int g = 0; g < 2; ++g) {
          uint32_t rg[16];
          tmem_ld_16x256b_x4(tmem + lane_base + (static_cast<uint32_t>(16 * g) << 16) + kColO + 64 * b + 32 * wg, rg);
          if (g == 1) {
            tc_fence_before();
            mbar_arrive(&sm.o_free[b]);
          }
          if (rows > 0) {
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
              const uint32_t sl = 8 * (2 * k2 + (m >> 1)) + j, ch = 2 * g + (m & 1);
              const uint32_t addr = smem_u32(stage) + sl * 64 + ((ch ^ ((sl >> 1) & 3u)) << 4);
              const int ra = 8 * k2, rb = 8 * k2 + 4;
              stmatrix_x4_trans(addr, pack_bf16x2(__uint_as_float(rg[ra]), __uint_as_float(rg[ra + 1])),
                                pack_bf16x2(__uint_as_float(rg[ra + 2]), __uint_as_float(rg[ra + 3])),
                                pack_bf16x2(__uint_as_float(rg[rb]), __uint_as_float(rg[rb + 1])),
                                pack_bf16x2(__uint_as_float(rg[rb + 2]), __uint_as_float(rg[rb + 3])));
            }
          }
        }
        if (rows > 0) {
          const int y0 = w.bos + seq_chunk<kRev>(c, w.nchunks) * kChunk + 32 * wg;
          if (rows >= 32) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(tm_o, stage, w.hv * kD + 32 * qd, y0);
              bulk_commit();
              bulk_wait_read_all();  // the stage is handed back to the V loads below
            }
          } else {
            // a ragged chunk's last rows: copy the valid ones, 16 bytes per lane
            __syncwarp();
            __nv_bfloat16* orow0 = p.o + static_cast<size_t>(y0) * ostride + static_cast<size_t>(w.hv) * kD + 32 * qd;
#pragma unroll
            for (int pass = 0; pass < 4; ++pass) {
              const int sl = pass * 8 + (lane >> 2), ch = lane & 3;
              if (sl < rows) {
                const uint4 x = *reinterpret_cast<const uint4*>(stage + sl * 64 + ((ch ^ ((sl >> 1) & 3)) << 4));
                *reinterpret_cast<uint4*>(orow0 + static_cast<size_t>(sl) * ostride + 8 * ch) = x;
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
        }
        if (lane == 0) mbar_arrive(&sm.v_empty[sv]);
      }
    }
    if (!ok) break;
    // state scatter
    if (p.h_final && state_live) {
      float4* dst = reinterpret_cast<float4*>(p.h_final + state_off);
#pragma unroll
      for (int i = 0; i < 16; ++i) dst[i] = make_float4(S[4 * i], S[4 * i + 1], S[4 * i + 2], S[4 * i + 3]);
    }
  }
  return err;
}

template <bool kListed, int kD, bool kRev = false, bool kF32Out = false>
__global__ void __launch_bounds__(kThreads, 1)
la_prefill_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                      const KernelParams p) {
  extern __shared__ uint8_t smem_raw[];
  SharedStorage& sm =
      *reinterpret_cast<SharedStorage*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  volatile int* abort = &sm.abort;
  // Launched with programmatic stream serialization: no global memory is touched before the
  // previous grid in the stream has completed, and the next grid may be placed once every CTA
  // of this one is running (it waits the same way).
  griddep_wait();
  griddep_launch_dependents();

  if (p.short_max >= 0) {
    // Launched beside the tokenwise kernel for a packed batch of short sequences: unless some
    // sequence is longer than short_max (or has bounds this kernel must report), every CTA
    // leaves before taking any resource.
    bool work = false;
    for (int n = tid; n < p.N && !work; n += kThreads) {
      const int b = __ldg(p.cu_seqlens + n), e = __ldg(p.cu_seqlens + n + 1);
      const bool bad = b < 0 || e < b || e > p.num_tokens;
      work = bad || (e - b > p.short_max && (!p.state_indices || __ldg(p.state_indices + n) >= 0));
    }
    if (!__syncthreads_or(work)) return;
  }

  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < kQKStages; ++i) {
      mbar_init(&sm.qk_full[i], 1);
      mbar_init(&sm.qk_empty[i], 1 + kOperandThreads + kConvThreads);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&sm.v_full[i], 1);
      mbar_init(&sm.v_empty[i], 2 + kStateThreads / 32);
    }
    mbar_init(&sm.scores_full, 1);
    mbar_init(&sm.scores_free, kOperandThreads);
    mbar_init(&sm.kt_ready, kOperandThreads);
    mbar_init(&sm.kt_free, 1);
    mbar_init(&sm.p_ready, kOperandThreads);
    mbar_init(&sm.p_free, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.qt_ready[b], kConvThreads);
      mbar_init(&sm.qt_free[b], 1);
      mbar_init(&sm.o_full[b], 1);
      mbar_init(&sm.o_free[b], kStateThreads);
    }
    mbar_init(&sm.ds_full, 1);
    mbar_init(&sm.ds_free, kStateThreads);
    mbar_init(&sm.s_ready, kStateThreads);
    mbar_init(&sm.s_free, 1);
    mbar_init(&sm.final_bar[0], 1);
    mbar_init(&sm.final_bar[1], 1);
    sm.abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
  }
  if constexpr (kD == 64) {
    // The MMAs that read V (dS, O_intra) have M = 128 value rows; with D = 64 the V tile's second
    // 64-column box is never loaded and must hold zeros for the whole kernel.
    for (int i = tid; i < kVStages * static_cast<int>(kTileBytes / 16); i += kThreads) {
      const int st = i / static_cast<int>(kTileBytes / 16), e = i % static_cast<int>(kTileBytes / 16);
      reinterpret_cast<uint4*>(sm.v[st][1])[e] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  if constexpr (kListed) {
    build_schedule(sm, p, tid);
    __syncthreads();
  }

  if (warp == 0) {
    if (lane == 0) tma_mma_loop<kListed, kD, kRev, kF32Out>(sm, p, &tm_q, &tm_k, &tm_v, tmem, abort);
  } else if (warp == 1) {
    if (lane == 0) mma_o_loop<kListed, kD>(sm, p, tmem, abort);
  } else if (warp < 4) {
    convert_loop<kListed, kD, kRev>(sm, p, tid - 64, abort);
  } else if (warp < 12) {
    const int err = state_loop<kListed, kD, kRev, kF32Out>(sm, p, &tm_o, tmem, tid - 128, abort);
    if (err && tid == 128 && p.dev_error) atomicOr(p.dev_error, err);
    if ((tid & 31) == 0) bulk_wait_all();  // this warp's output stores have completed
  } else {
    operand_loop<kListed, kD, kRev>(sm, p, tmem, tid - 384, abort);
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
