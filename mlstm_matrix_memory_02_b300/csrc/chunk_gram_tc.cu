// chunk_gram_tc.cu -- the backward's per-chunk L x L matrices on tensor cores (L = 64).
//
// Page "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural Networks"
// (llms.blog), section 3 "The Parallel Dual Form": inside a chunk every pair of tokens (u, t <= u)
// meets through the decay weight E_ut = exp(i~_t + sum_{t < tau <= u} log f_tau - m_u), which in
// the chunk's prefix sums is exp(x_t - mr_u).  The backward of h needs two such matrices per chunk:
//   mode 0: P_ut  = E_ut (q_u . k_t) / sqrt(d)             and n^(k) . q_u per row
//   mode 1: M1_ut = E_ut (g_u . v_t + c_u), g_u = dh_u / D_u
// both zero above the diagonal, written [P, NC, 64, 64] fp32 (row u, column t).  The raw products
// q . k and dh . v are bf16 x bf16 with fp32 sums on the tensor cores (exact products); the
// decay, the scale, 1/D_u and c_u are applied in fp32 as the accumulator is read.
//
// CTA = (chunk, head), 256 threads: thread 0 loads the chunk's x and y rows by TMA, thread 32
// issues the K / 16 products (M = 64, N = 64) into 64 tensor-memory columns, warps 0-3 read the
// accumulator (M = 64 layout: row 16 w + l in lane l < 16 of warp w's quarter) and write the
// rows, warps 4-7 form n . q_u from the q rows in shared memory (mode 0).
#include <cuda_bf16.h>

#include "common.cuh"
#include "f2math.cuh"
#include "kernels.cuh"
#include "sm100.cuh"
#include "tmap.cuh"

namespace mlstm {
namespace {

using namespace sm100;

constexpr int kLg = 64;
constexpr int kGramThreads = 256;

struct GramSmem {
  uint64_t full, done;
  uint32_t tmem_base;
  float xg[kLg], mr[kLg], w[kLg], c[kLg];
};

template <int K>
__global__ void __launch_bounds__(kGramThreads, 1) chunk_gram_kernel(
    const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapY, int mode,
    const float *__restrict__ invD, const float *__restrict__ cc, const float *__restrict__ gx,
    const float *__restrict__ gu, const float *__restrict__ cm, const float *__restrict__ ns, int S, int DQK,
    float *__restrict__ out, float *__restrict__ nq, int *__restrict__ err) {
  constexpr int TB = K * 128;  // bytes of a [64 x K] bf16 tile: K / 64 swizzled blocks of 8 KB
  static_assert(K % 64 == 0 && K <= 512, "K");
  extern __shared__ uint8_t gram_dyn[];
  __shared__ GramSmem sm;
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(gram_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t *const sx = base, *const sy = base + TB;
  const int kc = blockIdx.x, p = blockIdx.y, NC = S / kLg;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t tok0 = (size_t)p * S + (size_t)kc * kLg;

  if (tid == 0) {
    mbar_init(&sm.full, 1);
    mbar_init(&sm.done, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = sm.tmem_base;
  if (tid == 0) {
    prefetch_tensormap(&mapX);
    prefetch_tensormap(&mapY);
    mbar_arrive_expect_tx(&sm.full, 2u * TB);
#pragma unroll 1
    for (int b = 0; b < K / 64; ++b) {
      tma_load_2d(sx + b * 8192, &mapX, b * 64, (int)tok0, &sm.full);
      tma_load_2d(sy + b * 8192, &mapY, b * 64, (int)tok0, &sm.full);
    }
  }
  const float m_in = cm[(size_t)p * (NC + 1) + kc];
  if (tid < kLg) {
    sm.xg[tid] = gx[tok0 + tid];
    sm.mr[tid] = fmaxf(m_in, gu[tok0 + tid]);
    sm.w[tid] = mode == 1 ? invD[tok0 + tid] : rsqrtf((float)DQK);
    sm.c[tid] = mode == 1 ? cc[tok0 + tid] : 0.f;
  }
  const bool landed = __syncthreads_and(mbar_wait(&sm.full, 0, err, 131)) != 0;
  if (landed) {
    if (tid == 32) {
      tc_fence_after();
      const uint32_t id = idesc_f16(64, kLg, /*bf16*/ 1, 0, 0);
      const uint64_t dx = smem_desc(smem_u32(sx), 16, 1024, kSwizzle128B);
      const uint64_t dy = smem_desc(smem_u32(sy), 16, 1024, kSwizzle128B);
#pragma unroll 1
      for (int c = 0; c < K / 16; ++c) {
        const uint64_t off = (uint64_t)(((c >> 2) * 8192 + (c & 3) * 32) >> 4);
        mma_f16_ss(tm, dx + off, dy + off, id, c > 0);
      }
      mma_commit(&sm.done);
    }
    if (warp < 4) {
      const bool got = __all_sync(0xffffffffu, mbar_wait(&sm.done, 0, err, 132));
      if (got) {
        tc_fence_after();
        uint32_t u[2][32];
        const uint32_t lb = (uint32_t)(warp * 32) << 16;
        tmem_ld32(tm + lb, u[0]);
        tmem_ld32(tm + lb + 32, u[1]);
        tmem_wait_ld();
        if (lane < 16) {
          const int r = 16 * warp + lane;
          const float wr = sm.w[r], cr = sm.c[r], mrr = sm.mr[r];
          float4 *orow = reinterpret_cast<float4 *>(out + (((size_t)p * NC + kc) * kLg + r) * kLg);
#pragma unroll
          for (int t4 = 0; t4 < kLg / 4; ++t4) {
            float o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int t = 4 * t4 + e;
              const float sv = __uint_as_float(u[t >> 5][t & 31]);
              o[e] = t <= r ? (sv * wr + cr) * expf(sm.xg[t] - mrr) : 0.f;
            }
            orow[t4] = make_float4(o[0], o[1], o[2], o[3]);
          }
        }
      }
    } else if (mode == 0) {
      // n^(k) . q_u: two threads per row, each half of the columns (16-byte chunks of the
      // swizzled q rows)
      const int t = tid - 128, r = t >> 1, hf = t & 1;
      const float *nv = ns + ((size_t)p * (NC + 1) + kc) * (size_t)DQK;
      float a = 0.f;
#pragma unroll 4
      for (int ch = hf * (K / 16); ch < (hf + 1) * (K / 16); ++ch) {
        const uint4 w4 = *reinterpret_cast<const uint4 *>(sx + (ch >> 3) * 8192 + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
        const float4 n0 = *reinterpret_cast<const float4 *>(nv + 8 * ch);
        const float4 n1 = *reinterpret_cast<const float4 *>(nv + 8 * ch + 4);
        a += bf16_lo(w4.x) * n0.x + bf16_hi(w4.x) * n0.y + bf16_lo(w4.y) * n0.z + bf16_hi(w4.y) * n0.w;
        a += bf16_lo(w4.z) * n1.x + bf16_hi(w4.z) * n1.y + bf16_lo(w4.w) * n1.z + bf16_hi(w4.w) * n1.w;
      }
      a += __shfl_xor_sync(0xffffffffu, a, 1);
      if (hf == 0) nq[tok0 + r] = a;
    }
  } else if (tid == 0) {
    mbar_wait(&sm.full, 0, err, 133);  // nothing may leave while its loads are still landing
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tm, 64);
  }
}

template <int K>
cudaError_t launch_gram_k(int mode, const void *x, const void *y, const float *invD, const float *cc, const float *gx,
                          const float *gu, const float *cm, const float *ns, int P, int S, int DQK, float *out,
                          float *nq, int *err, cudaStream_t stream) {
  CUtensorMap mx, my;
  if (!make_tmap_2d_b16(&mx, x, true, (uint64_t)P * S, K, K, 64, kLg)) return cudaErrorInvalidValue;
  if (!make_tmap_2d_b16(&my, y, true, (uint64_t)P * S, K, K, 64, kLg)) return cudaErrorInvalidValue;
  const size_t smem = (size_t)2 * K * 128 + 1024;
  auto kern = chunk_gram_kernel<K>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(S / kLg, P), kGramThreads, smem, stream>>>(mx, my, mode, invD, cc, gx, gu, cm, ns, S, DQK, out, nq, err);
  return cudaGetLastError();
}

}  // namespace

bool chunk_gram_tc_supported(int L, int K) { return L == kLg && (K == 64 || K == 128 || K == 256 || K == 512); }

cudaError_t launch_chunk_gram_tc(int mode, const void *x, const void *y, int K, const float *invD, const float *cc,
                                 const float *gx, const float *gu, const float *cm, const float *ns, int P, int S,
                                 int DQK, float *out, float *nq, int *err, cudaStream_t stream) {
  if (P == 0 || S == 0) return cudaSuccess;
  switch (K) {
    case 64: return launch_gram_k<64>(mode, x, y, invD, cc, gx, gu, cm, ns, P, S, DQK, out, nq, err, stream);
    case 128: return launch_gram_k<128>(mode, x, y, invD, cc, gx, gu, cm, ns, P, S, DQK, out, nq, err, stream);
    case 256: return launch_gram_k<256>(mode, x, y, invD, cc, gx, gu, cm, ns, P, S, DQK, out, nq, err, stream);
    case 512: return launch_gram_k<512>(mode, x, y, invD, cc, gx, gu, cm, ns, P, S, DQK, out, nq, err, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace mlstm
