// la_decode_kernels.cuh -- sm_103a kernels for Lightning Attention speculative decoding:
// multi-token (MTP) decode, parallel verify with an optional KV buffer, and commit
// (page "[LA] Lightning Attention MTP decode + KVBuffer parallel verify / commit",
// Description).
//
// A request carries a handful of draft tokens (T <= 8 in the pages' workloads), so each
// (request, value head) unit costs one read of its 64 KB FP32 state, T token updates and,
// for decode and commit, one write of the state: the work is bound by the state traffic.
// Each row of the state evolves, and gives its output, independently of the others, so a
// unit is split over D / 64 parts of 64 state rows, each held in the registers of one
// 128-thread CTA (256 threads at D = 256).  The CTAs are persistent (ctas_per_sm per SM) and
// walk their parts; while a CTA applies the tokens of one part, a single bulk copy brings the
// next part's state slice (32 KB at D = 128, 16 KB at D = 64, 64 KB at D = 256) into shared
// memory, so every state load but the first overlaps arithmetic.  At D = 128 thread t owns state
// rows v = 64 h + 4 (t / 8) .. +3 and, of each, the four 16-byte column chunks
// k = 32 m + 4 (t % 8) .. +3 (m = 0..3) (two chunks at D = 64; at D = 256 rows 4 (t / 16) .. +3
// and chunks 64 m + 4 (t % 16), the row group's 16 lanes folded to 8 first), and for every token
//     S[v][k] = lambda S[v][k] + v_t[v] k_t[k]              (FP32, fused multiply-add)
//     o_t[v]  = scale sum_k S[v][k] q_t[k]                    (the 8 lanes of a row group hold
//                                                             partial sums of 4 rows; a reduce-
//                                                             scatter over lanes t^4, t^2, t^1
//                                                             leaves each row's total in 2 lanes)
// with the tokens' q, k, v staged in shared memory as FP32, 8 tokens at a time.  Where
// lambda^-8 stays small (slope <= 2.5) the registers hold, within a tile of 8 tokens starting
// at t0, S'_i = S_(t0 + i) / lambda^(i+1): then S'_i = S'_(i-1) + (lambda^-(i+1) v_i[v]) k_i[k]
// is one fused multiply-add per element and token, o_i = scale lambda^(i+1) S'_i q_i, and the
// tile ends with S = lambda^nt S'.  (The same sum, in another rounding order.)  Each staged k
// or q value feeds four rows, which keeps the shared-memory traffic per FMA low; the strided
// column chunks make a warp read 128 contiguous bytes of a row at a time, from the staged
// tokens and from the state slice alike, without bank conflicts.
// The three operations run this same per-token code, so a commit of all T tokens leaves
// bitwise the state a decode leaves, and verify's outputs (requests of more than 8 tokens; the
// shorter ones go to the tensor-core closed form of la_verify_kernel.cuh) are bitwise decode's.
//
// A fourth mode serves the prefill of short sequences (at most short_max tokens; the
// chunkwise prefill kernel takes the others): bounds from cu_seqlens or n T, the initial
// state from h0 (or zero), the final state to h_final.  For a few tokens the tokenwise
// recurrence costs one state read and write plus a little arithmetic, while a chunkwise
// unit pays its whole pipeline for one partial chunk.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace lad {

using lap::f2_fma;
using lap::f2_mul;
using lap::f2_pack;
using lap::f2_unpack;

constexpr int kDim = 128;                 // the default D = V
constexpr int kRows = 64;                 // state rows per CTA (D = 128 and 64)
constexpr int kSplit = kDim / kRows;      // CTAs per (request, value head) at D = 128
constexpr int kThreads = 128;             // threads per CTA at D = 128 and 64
// Lanes per row group and threads per CTA for head dimension kD (D = V = 64, 128 or 256): at
// D = 256 a row group of 4 rows spans 16 lanes, so that a thread still owns 4 rows x 16
// columns, and a CTA of 256 threads holds its 64 rows.
template <int kD>
__host__ __device__ constexpr int rows_of() { return kRows; }
template <int kD>
__host__ __device__ constexpr int lanes_of() { return kD == 256 ? 16 : 8; }
template <int kD>
__host__ __device__ constexpr int threads_of() { return kD == 256 ? 256 : kThreads; }
// CTAs per (request, value head)
template <int kD>
__host__ __device__ constexpr int split_of() { return kD / rows_of<kD>(); }

enum Mode : int { kDecode = 0, kVerify = 1, kCommit = 2, kPrefill = 3 };

struct Params {  // (D = V = 128 or 64)
  const __nv_bfloat16* q;  // [B*T, H, D]   (decode, verify)
  const __nv_bfloat16* k;  // [B*T, H, D]   (decode, verify)
  const __nv_bfloat16* v;  // [B*T, HV, D]  (decode, verify)
  const float* slopes;     // [HV]
  float* state;            // [P, HV, D, D]
  const int32_t* state_indices;
  __nv_bfloat16* o;        // [B*T, HV, D]  (decode, verify)
  __nv_bfloat16* kbuf;     // [P, T, H, D]  (written by verify when given, read by commit)
  __nv_bfloat16* vbuf;     // [P, T, HV, D]
  const int32_t* accepted_len;  // [B] (commit)
  const float* h0;              // [P, HV, D, D] or null (prefill: initial states)
  float* h_final;               // [P, HV, D, D] or null (prefill: final states)
  const int32_t* cu_seqlens;    // [B + 1] or null (prefill: packed sequence bounds)
  int* dev_error;
  float scale;
  int B, T, H, HV, G, pool_size;
  int num_tokens;  // prefill: rows of q, k, v, o
  int short_max;   // prefill: longer sequences are left to the chunkwise kernel
};

// Eight BF16 values (one 16-byte word) as FP32.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& x, float (&f)[8]) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Persistent form: a CTA walks its units (unit u = blockIdx.x + j gridDim.x; unit = (request,
// value head, part)) and, while it applies the tokens of one unit, a single bulk copy brings the
// next unit's state slice into shared memory, so the state load of every unit but the first
// overlaps the arithmetic of the previous one.  Thread t of a CTA owns rows
// vbase + 4 (t / 8) .. + 3 and, of each row, the D / 32 16-byte chunks of columns
// 32 m + 4 (t % 8) .. + 3: a warp then reads 128 contiguous bytes per row from the
// staged slice, the staged k and q, and writes 128 contiguous bytes per row of the state, all
// without bank conflicts.
constexpr int kTileTok = 8;  // tokens staged in shared memory per pass
// Resident CTAs per SM: the D = 64 instance holds half the registers and shared memory.
template <int kD>
__host__ __device__ constexpr int ctas_per_sm() { return kD == 64 ? 6 : kD == 256 ? 2 : 4; }

template <int kD>
struct __align__(128) TokSmem {
  float pre[rows_of<kD>() * kD]; // the next unit's state slice (bulk copy)
  float ks[kTileTok][kD];        // staged k (commit: from the KV buffer)
  float qs[kTileTok][kD];        // staged q
  float vs[kTileTok][rows_of<kD>()];  // staged v, this CTA's rows
  float linv[kTileTok];          // lambda^-(i+1) of the tile's token i (rescaled update)
  float lpow[kTileTok];          // lambda^(i+1)
  uint64_t bar;                  // slice landed (transaction bytes)
  int abort;
};

template <int kD>
__host__ __device__ constexpr int tokenwise_smem_bytes() { return static_cast<int>(sizeof(TokSmem<kD>)) + 128; }
// Persistent grid: every unit of work, or ctas_per_sm CTAs per SM when there are more units.
template <int kD>
inline int tokenwise_grid(int units, int sms) {
  return units < sms * ctas_per_sm<kD>() ? units : sms * ctas_per_sm<kD>();
}

// One unit's decoded description, identical for every thread of the CTA.
struct TokUnit {
  int b, hv, hq, part, slot, ntok;
  size_t row0;
  bool run, load, bad_index;
};

template <int kMode, int kD>
__device__ __forceinline__ TokUnit tok_unit(const Params& p, int u) {
  TokUnit w;
  const int unit = u / split_of<kD>();
  w.part = u - unit * split_of<kD>();
  w.b = unit / p.HV;
  w.hv = unit - w.b * p.HV;
  w.hq = w.hv / p.G;
  w.run = true;
  w.bad_index = false;
  w.slot = w.b;
  if (p.state_indices) {
    w.slot = __ldg(p.state_indices + w.b);
    w.bad_index = w.slot >= p.pool_size;
    if (w.slot < 0 || w.bad_index) w.run = false;  // padded (nothing read or written), or a bad index
  }
  w.ntok = p.T;
  w.row0 = static_cast<size_t>(w.b) * p.T;
  if (kMode == kPrefill) {
    if (p.cu_seqlens) {
      const int bb = __ldg(p.cu_seqlens + w.b), ee = __ldg(p.cu_seqlens + w.b + 1);
      if (bb < 0 || ee < bb || ee > p.num_tokens) w.run = false;  // flagged by the chunkwise kernel
      w.row0 = bb;
      w.ntok = ee - bb;
    }
    if (w.ntok > p.short_max) w.run = false;  // the chunkwise kernel's unit
  }
  if (kMode == kCommit && w.run) {
    w.ntok = min(max(__ldg(p.accepted_len + w.b), 0), p.T);
    if (w.ntok == 0) w.run = false;  // nothing accepted: the state stays as it is
  }
  w.load = w.run && (kMode != kPrefill || p.h0 != nullptr);
  return w;
}

// kD = D = V: 128 (two CTAs of 64 state rows per unit, 16 columns of each row per thread), 64
// (one CTA per unit, 8 columns per thread, more CTAs per SM) or 256 (four CTAs of 256 threads
// and 64 rows per unit, 16 columns of each row per thread, row groups of 16 lanes).
template <int kMode, int kD = kDim>
__global__ void __launch_bounds__(threads_of<kD>(), ctas_per_sm<kD>()) la_tokenwise_kernel(const Params p) {
  static_assert(kD == 128 || kD == 64 || kD == 256, "head dimension");
  constexpr int kR = rows_of<kD>();       // state rows of this CTA
  constexpr int kLanes = lanes_of<kD>();  // lanes of a row group
  constexpr int kLaneBits = kLanes == 16 ? 4 : 3;
  constexpr int kColStride = 4 * kLanes;  // columns between a thread's 16-byte chunks
  constexpr int kM = kD / kColStride;     // 16-byte column chunks of a row per thread
  constexpr int kChunks = kD / 8;         // 8-value chunks of a token row
  constexpr uint32_t kSlice = kR * kD * 4;
  extern __shared__ uint8_t tok_raw[];
  TokSmem<kD>& sm = *reinterpret_cast<TokSmem<kD>*>((reinterpret_cast<uintptr_t>(tok_raw) + 127) & ~uintptr_t(127));
  const int t = threadIdx.x;
  const int cg = t & (kLanes - 1), rg = t >> kLaneBits;  // chunks kColStride m + 4 cg, rows vbase + 4 rg .. +3
  const int units = p.B * p.HV * split_of<kD>();
  const float* s_in = (kMode == kPrefill) ? p.h0 : p.state;
  float* s_out = (kMode == kPrefill) ? p.h_final : p.state;
  volatile int* abort = &sm.abort;
  // launched with programmatic stream serialization (see la_prefill_fwd_kernel)
  lap::griddep_wait();
  lap::griddep_launch_dependents();
  if (t == 0) {
    lap::mbar_init(&sm.bar, 1);
    sm.abort = 0;
    lap::fence_mbar_init();
  }
  __syncthreads();

  auto slice_of = [&](const TokUnit& w) {
    return (static_cast<size_t>(w.slot) * p.HV + w.hv) * kD * kD + static_cast<size_t>(w.part) * kR * kD;
  };
  auto prefetch = [&](const TokUnit& w) {  // thread 0
    lap::mbar_arrive_expect_tx(&sm.bar, kSlice);
    lap::bulk_copy_g2s(sm.pre, s_in + slice_of(w), kSlice, &sm.bar);
  };
  // the first unit from u on (this CTA's stride) that runs; a bad state index is flagged
  auto seek = [&](int u, TokUnit& w) {
    for (; u < units; u += gridDim.x) {
      w = tok_unit<kMode, kD>(p, u);
      if (w.bad_index && t == 0 && p.dev_error) atomicOr(p.dev_error, 2);  // LA_DEV_ERR_BAD_INDEX
      if (w.run) return u;
    }
    return units;
  };

  TokUnit cur;
  int u = seek(blockIdx.x, cur);
  uint32_t phase = 0;
  bool pending = false;  // a slice copy is in flight
  if (u < units && cur.load && t == 0) prefetch(cur);
  pending = u < units && cur.load;
  while (u < units) {
    TokUnit nxt;
    const int un = seek(u + gridDim.x, nxt);
    const int vbase = cur.part * kR;
    const float slope = __ldg(p.slopes + cur.hv);
    const float lam = expf(-slope);
    const uint64_t lam2 = f2_pack(lam, lam);
    const bool resc = slope * kTileTok <= 20.f;  // the rescaled update (lambda^-8 <= e^20)

    // ---- this unit's state slice: S[r][2 m + h] = the pair (e = 2 h, 2 h + 1) of chunk m of row r
    uint64_t S[4][2 * kM];
    if (cur.load) {
      // a bounded wait, its outcome agreed by the whole CTA before anyone leaves the loop
      if (!__syncthreads_and(lap::mbar_wait(&sm.bar, phase, abort))) break;
      phase ^= 1u;
      pending = false;
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int m = 0; m < kM; ++m) {
          const float4 x = *reinterpret_cast<const float4*>(&sm.pre[(4 * rg + r) * kD + kColStride * m + 4 * cg]);
          S[r][2 * m] = f2_pack(x.x, x.y);
          S[r][2 * m + 1] = f2_pack(x.z, x.w);
        }
    } else {
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int j = 0; j < 2 * kM; ++j) S[r][j] = f2_pack(0.f, 0.f);
    }
    __syncthreads();  // every thread holds its part of the slice: the buffer is free
    if (un < units && nxt.load) {
      if (t == 0) prefetch(nxt);
      pending = true;
    }

    const size_t qk_tok = static_cast<size_t>(p.H) * kD;
    const size_t v_tok = static_cast<size_t>(p.HV) * kD;
    for (int t0 = 0; t0 < cur.ntok; t0 += kTileTok) {
      const int nt = min(kTileTok, cur.ntok - t0);
      __syncthreads();  // the previous tile has been consumed
      // stage tokens t0 .. t0 + nt - 1: 16 bytes (8 values) per thread and array per step
      for (int e = t; e < nt * kChunks; e += threads_of<kD>()) {
        const int i = e / kChunks, c = e % kChunks;  // token, 8-value chunk
        const bool vmine = c / (kR / 8) == cur.part;  // values 8c .. 8c + 7 are rows of this CTA
        uint4 kx, vx = make_uint4(0u, 0u, 0u, 0u);
        if (kMode == kCommit) {
          const size_t brow = static_cast<size_t>(cur.slot) * p.T + t0 + i;
          kx = __ldg(reinterpret_cast<const uint4*>(p.kbuf + (brow * p.H + cur.hq) * kD) + c);
          if (vmine) vx = __ldg(reinterpret_cast<const uint4*>(p.vbuf + (brow * p.HV + cur.hv) * kD) + c);
        } else {
          const size_t row = cur.row0 + t0 + i;
          kx = __ldg(reinterpret_cast<const uint4*>(p.k + row * qk_tok + static_cast<size_t>(cur.hq) * kD) + c);
          if (vmine)
            vx = __ldg(reinterpret_cast<const uint4*>(p.v + row * v_tok + static_cast<size_t>(cur.hv) * kD) + c);
          const uint4 qx =
              __ldg(reinterpret_cast<const uint4*>(p.q + row * qk_tok + static_cast<size_t>(cur.hq) * kD) + c);
          float f[8];
          bf16x8_to_f32(qx, f);
          reinterpret_cast<float4*>(&sm.qs[i][8 * c])[0] = make_float4(f[0], f[1], f[2], f[3]);
          reinterpret_cast<float4*>(&sm.qs[i][8 * c])[1] = make_float4(f[4], f[5], f[6], f[7]);
          if (kMode == kVerify && p.kbuf) {  // the KV buffer copy (k once per q/k head, by part 0)
            const size_t brow = static_cast<size_t>(cur.slot) * p.T + t0 + i;
            if (cur.hv % p.G == 0 && cur.part == 0)
              reinterpret_cast<uint4*>(p.kbuf + (brow * p.H + cur.hq) * kD)[c] = kx;
            if (vmine) reinterpret_cast<uint4*>(p.vbuf + (brow * p.HV + cur.hv) * kD)[c] = vx;
          }
        }
        float f[8];
        bf16x8_to_f32(kx, f);
        reinterpret_cast<float4*>(&sm.ks[i][8 * c])[0] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4*>(&sm.ks[i][8 * c])[1] = make_float4(f[4], f[5], f[6], f[7]);
        if (vmine) {
          bf16x8_to_f32(vx, f);
          reinterpret_cast<float4*>(&sm.vs[i][8 * c - vbase])[0] = make_float4(f[0], f[1], f[2], f[3]);
          reinterpret_cast<float4*>(&sm.vs[i][8 * c - vbase])[1] = make_float4(f[4], f[5], f[6], f[7]);
        }
      }
      if (t < nt) {
        sm.linv[t] = resc ? expf(slope * (t + 1)) : 1.f;
        sm.lpow[t] = resc ? expf(-slope * (t + 1)) : 1.f;
      }
      __syncthreads();

      for (int i = 0; i < nt; ++i) {
        const float4 vv = *reinterpret_cast<const float4*>(&sm.vs[i][4 * rg]);
        const float vf = sm.linv[i];
        const float vr[4] = {vv.x * vf, vv.y * vf, vv.z * vf, vv.w * vf};
        uint64_t kk[2 * kM];
#pragma unroll
        for (int m = 0; m < kM; ++m) {
          const float4 x = *reinterpret_cast<const float4*>(&sm.ks[i][kColStride * m + 4 * cg]);
          kk[2 * m] = f2_pack(x.x, x.y);
          kk[2 * m + 1] = f2_pack(x.z, x.w);
        }
        // S = lambda S + v_t[v] k_t
        if (!resc) {
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int j = 0; j < 2 * kM; ++j) S[r][j] = f2_mul(lam2, S[r][j]);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const uint64_t v2 = f2_pack(vr[r], vr[r]);
#pragma unroll
          for (int j = 0; j < 2 * kM; ++j) S[r][j] = f2_fma(v2, kk[j], S[r][j]);
        }
        if (kMode != kCommit) {
          // o_t[v] = scale S[v] . q_t over this thread's 4 kM columns, then across the 8 lanes of the row group
          uint64_t qq[2 * kM];
#pragma unroll
          for (int m = 0; m < kM; ++m) {
            const float4 x = *reinterpret_cast<const float4*>(&sm.qs[i][kColStride * m + 4 * cg]);
            qq[2 * m] = f2_pack(x.x, x.y);
            qq[2 * m + 1] = f2_pack(x.z, x.w);
          }
          float dot[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            uint64_t acc = f2_pack(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 2 * kM; ++j) acc = f2_fma(S[r][j], qq[j], acc);
            const float2 a2 = f2_unpack(acc);
            dot[r] = a2.x + a2.y;
          }
          // (16-lane row groups: fold the upper 8 lanes onto the lower first)
          if constexpr (kLanes == 16) {
#pragma unroll
            for (int r = 0; r < 4; ++r) dot[r] += __shfl_xor_sync(0xffffffffu, dot[r], 8);
          }
          // reduce-scatter over 8 lanes of the row group: lanes with bit 2 of cg keep rows
          // {2, 3} (else {0, 1}), bit 1 picks one of the two, bit 0 pairs lanes; lane cg ends
          // with the total of row 2 (cg >> 2) + ((cg >> 1) & 1), written by the even lanes
          // (of the lower 8, with 16-lane groups)
          const bool b2 = cg & 4, b1 = cg & 2;
          const float s0 = b2 ? dot[0] : dot[2], s1 = b2 ? dot[1] : dot[3];
          float k0 = (b2 ? dot[2] : dot[0]) + __shfl_xor_sync(0xffffffffu, s0, 4);
          float k1 = (b2 ? dot[3] : dot[1]) + __shfl_xor_sync(0xffffffffu, s1, 4);
          float kx = (b1 ? k1 : k0) + __shfl_xor_sync(0xffffffffu, b1 ? k0 : k1, 2);
          kx += __shfl_xor_sync(0xffffffffu, kx, 1);
          if (!(cg & 1) && (kLanes == 8 || cg < 8))
            p.o[(cur.row0 + t0 + i) * v_tok + static_cast<size_t>(cur.hv) * kD + vbase + 4 * rg +
                (2 * (cg >> 2) + ((cg >> 1) & 1))] = __float2bfloat16_rn(p.scale * sm.lpow[i] * kx);
        }
      }
      if (resc) {
        const float ln = sm.lpow[nt - 1];
        const uint64_t ln2 = f2_pack(ln, ln);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int j = 0; j < 2 * kM; ++j) S[r][j] = f2_mul(ln2, S[r][j]);
      }
    }

    if (kMode != kVerify && (kMode != kPrefill || s_out)) {
      float* dst = s_out + slice_of(cur);
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int m = 0; m < kM; ++m) {
          const float2 a = f2_unpack(S[r][2 * m]), c = f2_unpack(S[r][2 * m + 1]);
          *reinterpret_cast<float4*>(dst + (4 * rg + r) * kD + kColStride * m + 4 * cg) = make_float4(a.x, a.y, c.x, c.y);
        }
    }
    u = un;
    cur = nxt;
  }
  // no copy may still be landing in shared memory when the CTA exits
  if (pending) lap::mbar_wait_drain(&sm.bar, phase);
  __syncthreads();
  if (t == 0 && sm.abort && p.dev_error) atomicOr(p.dev_error, 4);  // LA_DEV_ERR_TIMEOUT
}

}  // namespace lad
