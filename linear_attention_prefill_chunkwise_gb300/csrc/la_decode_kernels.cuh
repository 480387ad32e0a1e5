// la_decode_kernels.cuh -- sm_103a kernels for Lightning Attention speculative decoding:
// multi-token (MTP) decode, parallel verify with an optional KV buffer, and commit
// (page "[LA] Lightning Attention MTP decode + KVBuffer parallel verify / commit",
// Description).
//
// A request carries a handful of draft tokens (T <= 8 in the pages' workloads), so each
// (request, value head) unit costs one read of its 64 KB FP32 state, T token updates and,
// for decode and commit, one write of the state: the work is bound by the state traffic,
// and the state fits the registers of one CTA.  One CTA of 256 threads per unit: thread t
// owns state row v = t / 2, columns k in [64 (t % 2), 64 (t % 2) + 64), and for every token
//     S[v][k] = lambda S[v][k] + v_t[v] k_t[k]              (FP32, fused multiply-add)
//     o_t[v]  = scale sum_k S[v][k] q_t[k]                    (two half-row partial sums)
// with the tokens' q, k, v staged in shared memory as FP32, 16 tokens at a time.  The three
// operations run this same per-token code, so a commit of all T tokens leaves bitwise the
// state a decode leaves, and verify's outputs are bitwise decode's.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace lad {

constexpr int kDim = 128;   // D = V = 128
constexpr int kThreads = 256;
constexpr int kTileT = 16;  // tokens staged in shared memory per pass

enum Mode : int { kDecode = 0, kVerify = 1, kCommit = 2 };

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
  int* dev_error;
  float scale;
  int B, T, H, HV, G, pool_size;
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

template <int kMode>
__global__ void __launch_bounds__(kThreads, 2) la_tokenwise_kernel(const Params p) {
  __shared__ __align__(16) float ks[kTileT][kDim];
  __shared__ __align__(16) float qs[kTileT][kDim];
  __shared__ __align__(16) float vs[kTileT][kDim];

  const int unit = blockIdx.x;  // b * HV + hv
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
  if (kMode == kCommit) {
    ntok = min(max(__ldg(p.accepted_len + b), 0), p.T);
    if (ntok == 0) return;  // nothing accepted: the state stays as it is
  }

  const int t = threadIdx.x;
  const int vrow = t >> 1, kh = t & 1;
  const float lam = expf(-__ldg(p.slopes + hv));

  // ---- state row v, columns 64 kh .. 64 kh + 63
  float S[64];
  float* srow = p.state + ((static_cast<size_t>(slot) * p.HV + hv) * kDim + vrow) * kDim + 64 * kh;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(srow) + i);
    S[4 * i] = x.x;
    S[4 * i + 1] = x.y;
    S[4 * i + 2] = x.z;
    S[4 * i + 3] = x.w;
  }

  const size_t qk_tok = static_cast<size_t>(p.H) * kDim;   // elements between tokens of q / k
  const size_t v_tok = static_cast<size_t>(p.HV) * kDim;   // ... of v / o
  for (int t0 = 0; t0 < ntok; t0 += kTileT) {
    const int nt = min(kTileT, ntok - t0);
    __syncthreads();  // the previous tile has been consumed
    // Stage tokens t0 .. t0 + nt - 1: 16 bytes (8 values) per thread and array per step.
    for (int e = t; e < nt * (kDim / 8); e += kThreads) {
      const int i = e >> 4, c = e & 15;
      uint4 kx, vx;
      if (kMode == kCommit) {
        kx = __ldg(reinterpret_cast<const uint4*>(p.kbuf + ((static_cast<size_t>(slot) * p.T + t0 + i) * p.H + hq) *
                                                               kDim) + c);
        vx = __ldg(reinterpret_cast<const uint4*>(p.vbuf + ((static_cast<size_t>(slot) * p.T + t0 + i) * p.HV + hv) *
                                                               kDim) + c);
      } else {
        const size_t row = static_cast<size_t>(b) * p.T + t0 + i;
        kx = __ldg(reinterpret_cast<const uint4*>(p.k + row * qk_tok + static_cast<size_t>(hq) * kDim) + c);
        vx = __ldg(reinterpret_cast<const uint4*>(p.v + row * v_tok + static_cast<size_t>(hv) * kDim) + c);
        const uint4 qx = __ldg(reinterpret_cast<const uint4*>(p.q + row * qk_tok + static_cast<size_t>(hq) * kDim) + c);
        float f[8];
        bf16x8_to_f32(qx, f);
        reinterpret_cast<float4*>(&qs[i][8 * c])[0] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4*>(&qs[i][8 * c])[1] = make_float4(f[4], f[5], f[6], f[7]);
        if (kMode == kVerify && p.kbuf) {  // the KV buffer copy (k once per q/k head)
          const size_t brow = static_cast<size_t>(slot) * p.T + t0 + i;
          if (hv % p.G == 0)
            reinterpret_cast<uint4*>(p.kbuf + (brow * p.H + hq) * kDim)[c] = kx;
          reinterpret_cast<uint4*>(p.vbuf + (brow * p.HV + hv) * kDim)[c] = vx;
        }
      }
      float f[8];
      bf16x8_to_f32(kx, f);
      reinterpret_cast<float4*>(&ks[i][8 * c])[0] = make_float4(f[0], f[1], f[2], f[3]);
      reinterpret_cast<float4*>(&ks[i][8 * c])[1] = make_float4(f[4], f[5], f[6], f[7]);
      bf16x8_to_f32(vx, f);
      reinterpret_cast<float4*>(&vs[i][8 * c])[0] = make_float4(f[0], f[1], f[2], f[3]);
      reinterpret_cast<float4*>(&vs[i][8 * c])[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
    __syncthreads();

    for (int i = 0; i < nt; ++i) {
      const float vv = vs[i][vrow];
      const float4* kr = reinterpret_cast<const float4*>(&ks[i][64 * kh]);
      // S = lambda S + v_t[v] k_t
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float4 kk = kr[j];
        S[4 * j] = fmaf(vv, kk.x, lam * S[4 * j]);
        S[4 * j + 1] = fmaf(vv, kk.y, lam * S[4 * j + 1]);
        S[4 * j + 2] = fmaf(vv, kk.z, lam * S[4 * j + 2]);
        S[4 * j + 3] = fmaf(vv, kk.w, lam * S[4 * j + 3]);
      }
      if (kMode != kCommit) {
        // o_t[v] = scale S[v] . q_t: four partial sums per half row, then the two halves
        const float4* qr = reinterpret_cast<const float4*>(&qs[i][64 * kh]);
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float4 qq = qr[j];
          a0 = fmaf(S[4 * j], qq.x, a0);
          a1 = fmaf(S[4 * j + 1], qq.y, a1);
          a2 = fmaf(S[4 * j + 2], qq.z, a2);
          a3 = fmaf(S[4 * j + 3], qq.w, a3);
        }
        float dot = (a0 + a1) + (a2 + a3);
        dot += __shfl_xor_sync(0xffffffffu, dot, 1);
        if (kh == 0)
          p.o[(static_cast<size_t>(b) * p.T + t0 + i) * v_tok + static_cast<size_t>(hv) * kDim + vrow] =
              __float2bfloat16_rn(p.scale * dot);
      }
    }
  }

  if (kMode != kVerify) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      reinterpret_cast<float4*>(srow)[i] = make_float4(S[4 * i], S[4 * i + 1], S[4 * i + 2], S[4 * i + 3]);
  }
}

}  // namespace lad
