// la_decode_kernels.cuh -- sm_103a kernels for Lightning Attention speculative decoding:
// multi-token (MTP) decode, parallel verify with an optional KV buffer, and commit
// (page "[LA] Lightning Attention MTP decode + KVBuffer parallel verify / commit",
// Description).
//
// A request carries a handful of draft tokens (T <= 8 in the pages' workloads), so each
// (request, value head) unit costs one read of its 64 KB FP32 state, T token updates and,
// for decode and commit, one write of the state: the work is bound by the state traffic.
// Each row of the state evolves, and gives its output, independently of the others, so a
// unit is split over kSplit CTAs of 128 threads that each keep 64 state rows in registers
// (more, smaller CTAs per SM overlap one CTA's state load with another's arithmetic).
// Thread t of part h owns the 4 x 16 block of state rows v = 64 h + 4 (t / 8) .. +3 and
// columns k = 16 (t % 8) .. +15, and for every token
//     S[v][k] = lambda S[v][k] + v_t[v] k_t[k]              (FP32, fused multiply-add)
//     o_t[v]  = scale sum_k S[v][k] q_t[k]                    (8 column-group partial sums,
//                                                             added across lanes t^1, t^2, t^4)
// with the tokens' q, k, v staged in shared memory as FP32, 16 tokens at a time.  Each staged
// k or q value feeds four rows, which keeps the shared-memory traffic per FMA low; the column
// groups are padded to 20 floats so that the 8 groups a warp reads sit in distinct banks.
// The three operations run this same per-token code, so a commit of all T tokens leaves
// bitwise the state a decode leaves, and verify's outputs are bitwise decode's.
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

constexpr int kDim = 128;   // D = V = 128
constexpr int kSplit = 2;                 // CTAs per (request, value head)
constexpr int kRows = kDim / kSplit;      // state rows per CTA
constexpr int kThreads = kRows / 4 * 8;   // 4 rows x 16 columns per thread
constexpr int kTileT = 16;  // tokens staged in shared memory per pass

enum Mode : int { kDecode = 0, kVerify = 1, kCommit = 2, kPrefill = 3 };

struct Params {
  const __nv_bfloat16* q;  // [B*T, H, 128]   (decode, verify)
  const __nv_bfloat16* k;  // [B*T, H, 128]   (decode, verify)
  const __nv_bfloat16* v;  // [B*T, HV, 128]  (decode, verify)
  const float* slopes;     // [HV]
  float* state;            // [P, HV, 128, 128]
  const int32_t* state_indices;
  __nv_bfloat16* o;        // [B*T, HV, 128]  (decode, verify)
  __nv_bfloat16* kbuf;     // [P, T, H, 128]  (written by verify when given, read by commit)
  __nv_bfloat16* vbuf;     // [P, T, HV, 128]
  const int32_t* accepted_len;  // [B] (commit)
  const float* h0;              // [P, HV, 128, 128] or null (prefill: initial states)
  float* h_final;               // [P, HV, 128, 128] or null (prefill: final states)
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

constexpr int kGroupStride = 20;  // floats per staged 16-column group (16 + 4 padding)

template <int kMode>
__global__ void __launch_bounds__(kThreads, 2 * kSplit) la_tokenwise_kernel(const Params p) {
  __shared__ __align__(16) float ks[kTileT][8 * kGroupStride];
  __shared__ __align__(16) float qs[kTileT][8 * kGroupStride];
  __shared__ __align__(16) float vs[kTileT][kRows];

  const int unit = blockIdx.x / kSplit;  // b * HV + hv
  const int part = blockIdx.x - unit * kSplit;
  const int vbase = part * kRows;        // first state row (value index) of this CTA
  const int b = unit / p.HV;
  const int hv = unit - b * p.HV;
  const int hq = hv / p.G;
  int slot = b;
  if (p.state_indices) {
    slot = __ldg(p.state_indices + b);
    if (slot < 0) return;  // padded request: nothing read or written
    if (slot >= p.pool_size) {
      if (threadIdx.x == 0 && p.dev_error) atomicOr(p.dev_error, 2);  // LA_DEV_ERR_BAD_INDEX
      return;
    }
  }
  int ntok = p.T;
  size_t row0 = static_cast<size_t>(b) * p.T;  // first token row of this unit
  if (kMode == kPrefill) {
    if (p.cu_seqlens) {
      const int bb = __ldg(p.cu_seqlens + b), ee = __ldg(p.cu_seqlens + b + 1);
      if (bb < 0 || ee < bb || ee > p.num_tokens) return;  // flagged by the chunkwise kernel
      row0 = bb;
      ntok = ee - bb;
    }
    if (ntok > p.short_max) return;  // the chunkwise kernel's unit
  }
  if (kMode == kCommit) {
    ntok = min(max(__ldg(p.accepted_len + b), 0), p.T);
    if (ntok == 0) return;  // nothing accepted: the state stays as it is
  }

  const int t = threadIdx.x;
  const int cg = t & 7, rg = t >> 3;  // columns 16 cg .. +15, rows vbase + 4 rg .. +3
  const float lam = expf(-__ldg(p.slopes + hv));
  const uint64_t lam2 = f2_pack(lam, lam);

  // ---- state block: S[r][j] pairs = (S[v + r][16 cg + 2 j], S[v + r][16 cg + 2 j + 1]), v = vbase + 4 rg
  uint64_t S[4][8];
  const size_t soff = ((static_cast<size_t>(slot) * p.HV + hv) * kDim + vbase + 4 * rg) * kDim + 16 * cg;
  const float* s_in = (kMode == kPrefill) ? p.h0 : p.state;
  float* s_out = (kMode == kPrefill) ? p.h_final : p.state;
  if (kMode != kPrefill || s_in) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 x = __ldg(reinterpret_cast<const float4*>(s_in + soff + r * kDim) + i);
        S[r][2 * i] = f2_pack(x.x, x.y);
        S[r][2 * i + 1] = f2_pack(x.z, x.w);
      }
  } else {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int j = 0; j < 8; ++j) S[r][j] = f2_pack(0.f, 0.f);
  }

  const size_t qk_tok = static_cast<size_t>(p.H) * kDim;   // elements between tokens of q / k
  const size_t v_tok = static_cast<size_t>(p.HV) * kDim;   // ... of v / o
  for (int t0 = 0; t0 < ntok; t0 += kTileT) {
    const int nt = min(kTileT, ntok - t0);
    __syncthreads();  // the previous tile has been consumed
    // Stage tokens t0 .. t0 + nt - 1: 16 bytes (8 values) per thread and array per step.
    for (int e = t; e < nt * (kDim / 8); e += kThreads) {
      const int i = e >> 4, c = e & 15;              // token, 8-value chunk (column group c / 2)
      const int kpos = (c >> 1) * kGroupStride + 8 * (c & 1);
      const bool vmine = c / (kRows / 8) == part;    // values 8c .. 8c + 7 are rows of this CTA
      uint4 kx, vx = make_uint4(0u, 0u, 0u, 0u);
      if (kMode == kCommit) {
        const size_t brow = static_cast<size_t>(slot) * p.T + t0 + i;
        kx = __ldg(reinterpret_cast<const uint4*>(p.kbuf + (brow * p.H + hq) * kDim) + c);
        if (vmine) vx = __ldg(reinterpret_cast<const uint4*>(p.vbuf + (brow * p.HV + hv) * kDim) + c);
      } else {
        const size_t row = row0 + t0 + i;
        kx = __ldg(reinterpret_cast<const uint4*>(p.k + row * qk_tok + static_cast<size_t>(hq) * kDim) + c);
        if (vmine) vx = __ldg(reinterpret_cast<const uint4*>(p.v + row * v_tok + static_cast<size_t>(hv) * kDim) + c);
        const uint4 qx = __ldg(reinterpret_cast<const uint4*>(p.q + row * qk_tok + static_cast<size_t>(hq) * kDim) + c);
        float f[8];
        bf16x8_to_f32(qx, f);
        reinterpret_cast<float4*>(&qs[i][kpos])[0] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4*>(&qs[i][kpos])[1] = make_float4(f[4], f[5], f[6], f[7]);
        if (kMode == kVerify && p.kbuf) {  // the KV buffer copy (k once per q/k head, by part 0)
          const size_t brow = static_cast<size_t>(slot) * p.T + t0 + i;
          if (hv % p.G == 0 && part == 0)
            reinterpret_cast<uint4*>(p.kbuf + (brow * p.H + hq) * kDim)[c] = kx;
          if (vmine) reinterpret_cast<uint4*>(p.vbuf + (brow * p.HV + hv) * kDim)[c] = vx;
        }
      }
      float f[8];
      bf16x8_to_f32(kx, f);
      reinterpret_cast<float4*>(&ks[i][kpos])[0] = make_float4(f[0], f[1], f[2], f[3]);
      reinterpret_cast<float4*>(&ks[i][kpos])[1] = make_float4(f[4], f[5], f[6], f[7]);
      if (vmine) {
        bf16x8_to_f32(vx, f);
        reinterpret_cast<float4*>(&vs[i][8 * c - vbase])[0] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4*>(&vs[i][8 * c - vbase])[1] = make_float4(f[4], f[5], f[6], f[7]);
      }
    }
    __syncthreads();

    for (int i = 0; i < nt; ++i) {
      const float4 vv = *reinterpret_cast<const float4*>(&vs[i][4 * rg]);
      const float vr[4] = {vv.x, vv.y, vv.z, vv.w};
      uint64_t kk[8];
      {
        const float4* kr = reinterpret_cast<const float4*>(&ks[i][cg * kGroupStride]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 x = kr[j];
          kk[2 * j] = f2_pack(x.x, x.y);
          kk[2 * j + 1] = f2_pack(x.z, x.w);
        }
      }
      // S = lambda S + v_t[v] k_t
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint64_t v2 = f2_pack(vr[r], vr[r]);
#pragma unroll
        for (int j = 0; j < 8; ++j) S[r][j] = f2_fma(v2, kk[j], f2_mul(lam2, S[r][j]));
      }
      if (kMode != kCommit) {
        // o_t[v] = scale S[v] . q_t over this thread's 16 columns, then across the 8 groups
        uint64_t qq[8];
        const float4* qr = reinterpret_cast<const float4*>(&qs[i][cg * kGroupStride]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 x = qr[j];
          qq[2 * j] = f2_pack(x.x, x.y);
          qq[2 * j + 1] = f2_pack(x.z, x.w);
        }
        float dot[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          uint64_t acc = f2_pack(0.f, 0.f);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc = f2_fma(S[r][j], qq[j], acc);
          const float2 a2 = f2_unpack(acc);
          dot[r] = a2.x + a2.y;
        }
#pragma unroll
        for (int m = 1; m < 8; m <<= 1)
#pragma unroll
          for (int r = 0; r < 4; ++r) dot[r] += __shfl_xor_sync(0xffffffffu, dot[r], m);
        if (cg < 4)  // lane group cg writes row vbase + 4 rg + cg
          p.o[(row0 + t0 + i) * v_tok + static_cast<size_t>(hv) * kDim + vbase + 4 * rg + cg] =
              __float2bfloat16_rn(p.scale * (cg == 0 ? dot[0] : cg == 1 ? dot[1] : cg == 2 ? dot[2] : dot[3]));
      }
    }
  }

  if (kMode != kVerify && (kMode != kPrefill || s_out)) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 a = f2_unpack(S[r][2 * i]), c = f2_unpack(S[r][2 * i + 1]);
        reinterpret_cast<float4*>(s_out + soff + r * kDim)[i] = make_float4(a.x, a.y, c.x, c.y);
      }
  }
}

}  // namespace lad
