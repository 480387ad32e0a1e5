// la_verify_kernel.cuh -- sm_103a kernel of la_verify for requests of at most 8 draft tokens:
// the closed form of page "[LA] Lightning Attention MTP decode + KVBuffer parallel verify /
// commit" (Description, "Closed form used by verify"),
//     o_t = lambda^(t+1) scale (S q_t) + sum_(j <= t) lambda^(t-j) scale (q_t . k_j) v_j,
// evaluated without materialising any intermediate state.  Per (request, value head) the work
// is one read of the 64 KB FP32 state S and one small product S [q_0 .. q_(T-1)], which runs on
// the tensor cores: S is the A operand (M = 128 value rows, K = 128), the request's q rows part of
// the B operand (N = 32 columns, T of the unit's 8 used), both as TF32 (the pages' verify kernel also
// multiplies h0 by q in TF32), accumulated in FP32 in tensor memory.
//
// One persistent CTA per SM walks the units u = blockIdx.x + n gridDim.x:
//   warp 12 (one thread)  TMA loads: each unit's state slice as four 128 x 32 FP32 boxes,
//                         128-byte swizzled (the canonical K-major operand layout), into a
//                         2-stage ring, and the request's q, k, v rows (8 x 128 BF16 each)
//                         into the 2-stage ring of the group that takes the unit;
//   warps 0-3, 4-7, 8-11  three compute groups, group g on the units n with n % 3 == g: per
//                         unit, q to FP32 in the group's 8 rows of the B operand (swizzled); one thread
//                         issues the 16 MMAs (K = 8 each); meanwhile the scores
//                         A[i][j] = scale lambda^(i-j) q_i . k_j (j <= i) on the CUDA cores;
//                         then thread v (= TMEM lane v) reads row v of S q, adds the intra
//                         terms and stores o_t[v]; the draft k, v go to the KV buffer.  Each
//                         group's chain of waits is long next to its arithmetic; three of them
//                         keep three units' state loads in flight (one group: 0.123 ms, two:
//                         0.107, three: 0.103 on 128 requests x 8 tokens x 64 heads; four: no
//                         better).
// Every wait is bounded (sm103_ptx.cuh); a timeout sets LA_DEV_ERR_TIMEOUT, drains this CTA's
// copies and MMAs in flight and frees tensor memory before the CTA exits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace lav {

constexpr int kDim = 128;
constexpr int kMaxTok = 8;        // draft tokens per request on this path
constexpr int kN = 32;            // the MMA's N: the groups' q rows (rows kGroups * kMaxTok .. 31 stay zero)
constexpr int kGroups = 3;        // compute groups, each on its own units (in turn)
constexpr int kStStages = 2;      // state ring (shared by the groups, in unit order)
constexpr int kTkStages = 2;      // token ring of each group
constexpr int kCompute = 128;     // threads of a group: 4 warps, one TMEM lane per thread
constexpr int kThreads = kGroups * kCompute + 32;
constexpr uint32_t kStateBox = 128 * 32 * 4;  // 128 rows x 32 FP32 columns
constexpr uint32_t kStateBytes = 4 * kStateBox;
constexpr uint32_t kBBox = kN * 128;          // kN rows x 32 FP32 columns
constexpr uint32_t kTokBytes = kMaxTok * kDim * 2;
constexpr uint32_t kTmemCols = 128;  // group g's accumulator: columns kN g .. kN g + kN - 1 (power of 2)

struct Params {
  const float* slopes;           // [HV]
  const int32_t* state_indices;  // [B] or null
  __nv_bfloat16* o;              // [B*T, HV, 128]
  __nv_bfloat16* kbuf;           // [P, T, H, 128] or null
  __nv_bfloat16* vbuf;           // [P, T, HV, 128]
  int* dev_error;
  float scale;
  int B, T, H, HV, G, pool_size;
};

struct __align__(1024) Smem {
  uint8_t st[kStStages][kStateBytes];                     // state slices: box c = columns 32c .. 32c+31
  uint8_t bt[4][kBBox];                                   // q as FP32, [kN t][128 k] in 4 boxes of 32 k:
                                                          // rows 8g .. 8g+7 are group g's tokens
  __nv_bfloat16 tk[kGroups][kTkStages][3][kMaxTok][kDim];  // q, k, v rows of a request's tokens
  float A[kGroups][kMaxTok][kMaxTok];                     // scale lambda^(i-j) q_i . k_j, j <= i
  float dec[kGroups][kMaxTok + 1];                        // lambda^m, m = 0 .. kMaxTok
  uint64_t st_full[kStStages], st_empty[kStStages];
  uint64_t tk_full[kGroups][kTkStages], tk_empty[kGroups][kTkStages];
  uint64_t mma_bar[kGroups], final_bar[kGroups];
  uint32_t tmem_base;
  int abort;
};
static_assert(kGroups * kMaxTok <= kN, "the groups' q rows fit the MMA's N");

__host__ __device__ constexpr int verify_smem_bytes() { return static_cast<int>(sizeof(Smem)) + 1024; }

// D[tmem] (+)= A[smem] * B[smem], TF32 operands (K = 8 per instruction)
__device__ __forceinline__ void mma_tf32_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Descriptor of the same operand `byte_off` bytes further on (the start address field counts
// 16-byte units).
__device__ __forceinline__ uint64_t desc_at(uint64_t base, uint32_t byte_off) { return base + (byte_off >> 4); }

// Barrier over `n` threads (a multiple of 32) that also ANDs `pred` over them.
__device__ __forceinline__ bool bar_and(uint32_t id, uint32_t n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}\n"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// The next unit from u on (this CTA's stride) that runs: a padded request (negative slot) is
// skipped, a slot >= pool_size is skipped and, when `flag`, reported.
__device__ __forceinline__ int seek(const Params& p, int u, int units, bool flag, int& slot) {
  for (; u < units; u += gridDim.x) {
    const int b = u / p.HV;
    slot = p.state_indices ? __ldg(p.state_indices + b) : b;
    if (slot >= p.pool_size) {
      if (flag && p.dev_error) atomicOr(p.dev_error, 2);  // LA_DEV_ERR_BAD_INDEX
      continue;
    }
    if (slot >= 0) return u;
  }
  return units;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& x, float (&f)[8]) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// The load thread: every unit's state slice (ring stage n % kStStages for the CTA's n-th unit) and
// token rows (group n % kGroups's ring, stage (n / kGroups) % kTkStages), in the consumers' order.
__device__ __forceinline__ void load_loop(Smem& sm, const Params& p, const CUtensorMap* tm_s,
                                          const CUtensorMap* tm_q, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                          volatile int* abort) {
  const int units = p.B * p.HV;
  uint32_t n_st = 0, n_tk[kGroups] = {};  // units loaded, in all and per group
  int slot = 0;
  for (int u = seek(p, blockIdx.x, units, true, slot); u < units; u = seek(p, u + gridDim.x, units, true, slot)) {
    const int b = u / p.HV, hv = u - b * p.HV, hq = hv / p.G;
    const int g = n_st % kGroups;
    const uint32_t s = n_st % kStStages;
    if (!lap::mbar_wait(&sm.st_empty[s], ((n_st / kStStages) & 1u) ^ 1u, abort)) break;
    lap::mbar_arrive_expect_tx(&sm.st_full[s], kStateBytes);
    const int32_t y = (slot * p.HV + hv) * kDim;
#pragma unroll
    for (int c = 0; c < 4; ++c) lap::tma_load_2d(sm.st[s] + c * kStateBox, tm_s, &sm.st_full[s], 32 * c, y);
    ++n_st;
    const uint32_t j = n_tk[g], s2 = j % kTkStages;
    if (!lap::mbar_wait(&sm.tk_empty[g][s2], ((j / kTkStages) & 1u) ^ 1u, abort)) break;
    uint64_t* bar = &sm.tk_full[g][s2];
    lap::mbar_arrive_expect_tx(bar, 3 * kTokBytes);
    const int32_t row = b * p.T;
    lap::tma_load_2d(sm.tk[g][s2][0], tm_q, bar, hq * kDim, row);
    lap::tma_load_2d(sm.tk[g][s2][1], tm_k, bar, hq * kDim, row);
    lap::tma_load_2d(sm.tk[g][s2][2], tm_v, bar, hv * kDim, row);
    ++n_tk[g];
  }
  // Teardown, also after an abort: a load is issued only after the previous one into its slot
  // was consumed, so the last loads of each ring are the only ones that can still be in flight.
  for (uint32_t i = 0; i < kStStages && i < n_st; ++i) {
    const uint32_t j = n_st - 1 - i;
    lap::mbar_wait_drain(&sm.st_full[j % kStStages], (j / kStStages) & 1u);
  }
  for (int g = 0; g < kGroups; ++g) {
    const uint32_t n_tkg = n_tk[g];
    for (uint32_t i = 0; i < kTkStages && i < n_tkg; ++i) {
      const uint32_t j = n_tkg - 1 - i;
      lap::mbar_wait_drain(&sm.tk_full[g][j % kTkStages], (j / kTkStages) & 1u);
    }
  }
}

// Compute group g (warps 4g .. 4g+3): thread t is TMEM lane t and value row t of the group's
// units, the CTA's units n with n % kGroups == g.  The groups meet only in the state ring and in the
// B operand, of which each writes its own 8 rows (the other groups' rows give MMA columns that
// are not read).
__device__ __forceinline__ void compute_loop(Smem& sm, const Params& p, uint32_t tmem_base, int g,
                                             volatile int* abort) {
  const int t = threadIdx.x - kCompute * g;
  const uint32_t bar_id = 1 + g;  // the group's named barrier
  const int units = p.B * p.HV;
  const int T = p.T;
  const uint32_t tmem = tmem_base + kN * g;
  constexpr uint32_t idesc = lap::idesc_tf32_f32(128, kN, false, false);
  const uint64_t da0 = lap::sdesc_sw128(lap::smem_u32(sm.st[0]), 16, 1024);
  const uint64_t db0 = lap::sdesc_sw128(lap::smem_u32(sm.bt[0]), 16, 1024);
  const size_t v_tok = static_cast<size_t>(p.HV) * kDim;
  uint32_t n = 0, j = 0;  // the CTA's unit count, this group's unit count
  int slot = 0;
  for (int u = seek(p, blockIdx.x, units, false, slot); u < units;
       u = seek(p, u + gridDim.x, units, false, slot), ++n) {
    if (static_cast<int>(n % kGroups) != g) continue;
    const int b = u / p.HV, hv = u - b * p.HV, hq = hv / p.G;
    const uint32_t s = n % kStStages, s2 = j % kTkStages;
    const bool got = lap::mbar_wait(&sm.tk_full[g][s2], (j / kTkStages) & 1u, abort);
    if (!bar_and(bar_id, kCompute, got)) break;
    const __nv_bfloat16(*tk)[kMaxTok][kDim] = sm.tk[g][s2];

    // q rows as FP32 into rows 8g .. 8g+7 of the B operand: thread t converts 8 values (token
    // t / 16, chunk t % 16) and writes them as two 16-byte chunks of box (t % 16) / 4, swizzled by
    // the operand row.
    {
      const int i = t >> 4, ch = t & 15, row = kMaxTok * g + i;
      float f[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(&tk[0][i][8 * ch]), f);
      uint8_t* rp = sm.bt[ch >> 2] + row * 128;
      const int c0 = 2 * (ch & 3);
      *reinterpret_cast<float4*>(rp + ((c0 ^ (row & 7)) << 4)) = make_float4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<float4*>(rp + (((c0 + 1) ^ (row & 7)) << 4)) = make_float4(f[4], f[5], f[6], f[7]);
    }
    const float slope = __ldg(p.slopes + hv);
    if (t <= kMaxTok) sm.dec[g][t] = t == 0 ? 1.f : expf(-slope * t);
    lap::fence_proxy_async_smem();
    lap::named_bar_sync(bar_id, kCompute);

    if (t == 0) {
      // S q for the unit's tokens: 16 MMAs along K (8 columns each; 4 per 32-column box)
      if (lap::mbar_wait(&sm.st_full[s], (n / kStStages) & 1u, abort)) {
        lap::tc_fence_after();
        const uint64_t da = da0 + ((s * kStateBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
          mma_tf32_ss(tmem, desc_at(da, (kk >> 2) * kStateBox + (kk & 3) * 32),
                      desc_at(db0, (kk >> 2) * kBBox + (kk & 3) * 32), idesc, kk > 0);
        lap::mma_commit(&sm.st_empty[s]);
        lap::mma_commit(&sm.mma_bar[g]);
      }
    }

    // scores while the MMAs run: two threads per pair (i, j) = (t / 16, t / 2 % 8), 64 columns
    // each, their 16-byte chunks rotated by t so that a shared-memory phase hits 8 bank groups
    {
      const int i = t >> 4, jj = (t >> 1) & 7, h = t & 1;
      const bool live = jj <= i && i < T;
      float d0 = 0.f, d1 = 0.f;
      if (live) {
        const __nv_bfloat16* qr = &tk[0][i][64 * h];
        const __nv_bfloat16* kr = &tk[1][jj][64 * h];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          const int c = 8 * ((cc + t) & 7);
          float a[8], bk[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(qr + c), a);
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(kr + c), bk);
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            d0 = fmaf(a[e], bk[e], d0);
            d1 = fmaf(a[e + 1], bk[e + 1], d1);
          }
        }
      }
      float d = d0 + d1;
      d += __shfl_xor_sync(0xffffffffu, d, 1);
      if (live && h == 0) sm.A[g][i][jj] = p.scale * sm.dec[g][i - jj] * d;
    }

    const bool done = lap::mbar_wait(&sm.mma_bar[g], j & 1u, abort);
    if (!bar_and(bar_id, kCompute, done)) break;
    lap::tc_fence_after();
    float acc[16];
    const uint32_t col0 = (kMaxTok * g) & ~15u;  // the 16 columns holding this group's 8
    lap::tmem_ld16(tmem + ((static_cast<uint32_t>(t) & ~31u) << 16) + col0, acc);  // row t: (S q_c)[t], c = 0..15
    float vj[kMaxTok];
#pragma unroll
    for (int jj = 0; jj < kMaxTok; ++jj) vj[jj] = __bfloat162float(tk[2][jj][t]);
    __nv_bfloat16* orow = p.o + static_cast<size_t>(b) * T * v_tok + static_cast<size_t>(hv) * kDim + t;
#pragma unroll
    for (int i = 0; i < kMaxTok; ++i) {
      if (i < T) {
        float o = p.scale * sm.dec[g][i + 1] * (kMaxTok * g - col0 ? acc[kMaxTok + i] : acc[i]);
#pragma unroll
        for (int jj = 0; jj <= i; ++jj) o = fmaf(sm.A[g][i][jj], vj[jj], o);
        orow[static_cast<size_t>(i) * v_tok] = __float2bfloat16_rn(o);
      }
    }
    if (p.kbuf) {  // the KV buffer copy: k once per q/k head, v per value head
      for (int e = t; e < T * 16; e += kCompute) {
        const int i = e >> 4, c = e & 15;
        const size_t brow = static_cast<size_t>(slot) * T + i;
        if (hv % p.G == 0)
          reinterpret_cast<uint4*>(p.kbuf + (brow * p.H + hq) * kDim)[c] =
              *reinterpret_cast<const uint4*>(&tk[1][i][8 * c]);
        reinterpret_cast<uint4*>(p.vbuf + (brow * p.HV + hv) * kDim)[c] =
            *reinterpret_cast<const uint4*>(&tk[2][i][8 * c]);
      }
    }
    // the token stage and the accumulator are free once every thread is past this point
    lap::tc_fence_before();
    lap::named_bar_sync(bar_id, kCompute);
    if (t == 0) lap::mbar_arrive(&sm.tk_empty[g][s2]);
    ++j;
  }
  if (t == 0) {  // every MMA this group issued has retired before tensor memory is released
    lap::mma_commit(&sm.final_bar[g]);
    lap::mbar_wait_drain(&sm.final_bar[g], 0);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
la_verify_tc_kernel(const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const Params p) {
  extern __shared__ uint8_t verify_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(verify_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5;
  volatile int* abort = &sm.abort;
  // launched with programmatic stream serialization (see la_prefill_fwd_kernel)
  lap::griddep_wait();
  lap::griddep_launch_dependents();
  if (warp == 0) {
    lap::tmem_alloc(&sm.tmem_base, kTmemCols);
    lap::tmem_relinquish();
  }
  if (tid == kGroups * kCompute) {
    for (int i = 0; i < kStStages; ++i) {
      lap::mbar_init(&sm.st_full[i], 1);
      lap::mbar_init(&sm.st_empty[i], 1);
    }
    for (int g = 0; g < kGroups; ++g) {
      for (int i = 0; i < kTkStages; ++i) {
        lap::mbar_init(&sm.tk_full[g][i], 1);
        lap::mbar_init(&sm.tk_empty[g][i], 1);
      }
      lap::mbar_init(&sm.mma_bar[g], 1);
      lap::mbar_init(&sm.final_bar[g], 1);
    }
    sm.abort = 0;
    lap::fence_mbar_init();
    lap::tma_prefetch_desc(&tm_s);
    lap::tma_prefetch_desc(&tm_q);
    lap::tma_prefetch_desc(&tm_k);
    lap::tma_prefetch_desc(&tm_v);
  }
  // the B operand starts at zero (a group's MMAs read the other group's rows too)
  for (int i = tid; i < static_cast<int>(sizeof(sm.bt) / 16); i += kThreads)
    reinterpret_cast<uint4*>(&sm.bt[0][0])[i] = make_uint4(0u, 0u, 0u, 0u);
  lap::fence_proxy_async_smem();
  lap::tc_fence_before();
  __syncthreads();
  lap::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp < 4 * kGroups) {
    compute_loop(sm, p, tmem, warp >> 2, abort);
  } else if ((tid & 31) == 0) {
    load_loop(sm, p, &tm_s, &tm_q, &tm_k, &tm_v, abort);
  }

  lap::tc_fence_before();
  __syncthreads();
  if (tid == 0 && sm.abort && p.dev_error) atomicOr(p.dev_error, 4);  // LA_DEV_ERR_TIMEOUT
  if (warp == 0) {
    __syncwarp();
    lap::tc_fence_after();
    lap::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace lav
