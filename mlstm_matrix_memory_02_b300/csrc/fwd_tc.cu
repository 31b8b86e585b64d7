// fwd_tc.cu -- tensor-core chunkwise forward of the mLSTM cell: the inter-chunk recurrence and the
// intra-chunk output in one pass per (head, 128-row d_v tile[, d_qk half]), the matrix state
// resident in tensor memory for the whole sequence.
//
// Page "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural Networks"
// (llms.blog): section 3 "The Parallel Dual Form" (H = ((Q K^T) o D) V inside a chunk, the state
// unrolled across chunks), section 3 "Associative Matrix Cell State" (C and n updates, the
// retrieval h = C q / max(|n^T q|, .), k scaled by 1/sqrt(d)), section 2 (the max stabiliser).
// Per chunk k, entering state (C, n, m_in), and the gate kernel's per-token b, x = i~ - b and
// running max u (so the row stabiliser is m_r = b_r + mr_r with mr_r = max(m_in, u_r)):
//   S   = Q K^T                                   bf16 inputs, fp32 accumulate
//   P   = S / sqrt(d) * exp(x_j - mr_r), j <= r   fp32, rounded to fp16 for the next product
//   H^T = C (beta q)^T + V^T P^T,  beta_r = exp(m_in - mr_r)
//   h_r = H_r / max(|sum_j P_rj + beta_r n.q_r|, exp(-m_r))
//   C  <- alpha C + V^T diag(w) K / sqrt(d),  n <- alpha n + K^T w / sqrt(d)
//
// Work split.  A CTA owns 128 rows of d_v (MMA M) and DH columns of d_qk.  With PAIR, two CTAs of
// a cluster split d_qk in halves (DH = d_qk / 2): each holds its half of the state, computes
// partial Q K^T, n.q and C q sums over its half and exchanges them through distributed shared
// memory; CTA rank rho finalises output rows r in [32 rho, 32 rho + 32).  This fits d_qk = 512
// (a 128 x 256 fp32 state tile fills half of tensor memory) and doubles the SMs used per head.
//
// Tensor memory (512 columns): [0, DH) fp32 state T, [DH, 3 DH / 2) its fp16 copy (A operand of
// the C q product), [384, 448) S (M = 64 layout), [448, 512) H^T.  The state is kept in a lazily
// rescaled frame C = exp(sigma) T: the chunk decay is folded into sigma and into the scale of the
// update's k operand, and T is multiplied back only when exp(-sigma) would exceed 2^8.
//
// Warp roles (512 threads): warp 0 issues TMA loads of the q, k, v tiles (two stages); warp 1
// allocates tensor memory and issues every MMA; warp 2 computes the per-chunk gate factors;
// warpgroup 1 (warps 4-7) forms P and writes h; warpgroup 2 (warps 8-11) copies the state to
// fp16 (the serial chain of the recurrence); warpgroup 3 (warps 12-15) converts q, k, v in place
// to the scaled fp16 operands and keeps n.  Hand-offs use mbarriers; every wait is bounded in
// time and reports through an error word.
//
// Operand precision: q, k, v arrive as bf16 and convert to fp16 exactly; the computed operands
// (P, beta q, w k and the state copy) are rounded to fp16 (11 significant bits); sums are fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.cuh"
#include "sm100.cuh"
#include "tmap.cuh"

// Optional timeline trace for performance analysis (build with -DMLSTM_TRACE): the SM clock at
// fixed points of every role of CTA (0, 0), per chunk; read back with mlstm_trace_read.
#ifdef MLSTM_TRACE
__device__ long long g_trace[8][512][8];
#define TRACE(role, k, ev)                                                              \
  do {                                                                                  \
    if (blockIdx.x == 0 && blockIdx.y == 0 && (k) < 512) g_trace[role][k][ev] = clock64(); \
  } while (0)
extern "C" int mlstm_trace_read(long long *dst, size_t bytes) {
  return (int)cudaMemcpyFromSymbol(dst, g_trace, bytes < sizeof(g_trace) ? bytes : sizeof(g_trace));
}
#else
#define TRACE(role, k, ev) \
  do {                     \
  } while (0)
#endif

namespace mlstm {
namespace {

using namespace sm100;

constexpr int kL = 64;        // chunk length
constexpr int kTile = 128;    // d_v rows per CTA (MMA M)
constexpr int kThreads = 512;
constexpr float kRescaleLog = 5.545177444479562f;  // ln(2^8): largest lazy frame factor
constexpr uint32_t kColS = 384, kColH = 448;

// Per-chunk gate factors (written by warp 2, read by the other roles).
struct Gate {
  float mr[kL];      // max(m_in, u_r)
  float floor_[kL];  // exp(-(b_r + mr_r)) = exp(-m_r)
  float beta[kL];    // exp(m_in - mr_r)
  float xg[kL];      // x_j
  float wk[kL];      // w_j exp(-sigma_next) / sqrt(d): scale of k in the update (frame of T)
  float wt[kL];      // w_j / sqrt(d): scale of k in the n update
  float alpha;       // chunk decay exp(b_L + m_in - m_out)
  float fr_c;        // T -> C factor of the entering state (exp(sigma))
  float fr_w;        // eager write-back factor (exp(sigma) alpha)
  float sig_next;    // frame of T after this chunk's update
  int lazy;
  int pad_[3];
};

struct Smem {
  uint64_t full[2], empty[2], bar_S[2], bar_nq[2];
  uint64_t sfree, bar_U, bar_H, hfree, cready, opready, pready, fin;
  uint64_t sx_full[2], sx_free[2], hx_full, hx_free;
  uint64_t grp[3];  // bounded group barriers of warpgroups 1, 2 and 3
  uint32_t tmem_base;
  int abort_flag;
  Gate g[2];
  float n[256];          // normaliser, this CTA's d_qk columns
  float npart[1024];     // n-update partial sums of warpgroup 3
  float nq[2][kL];       // n . q_r over this CTA's columns
  float nqx[2][32];      // partner's n . q_r for the rows finalised here (written remotely)
  float inv[2][kL];      // 1 / max(|den_r|, exp(-m_r))
};

__device__ __forceinline__ bool aborted(const Smem &sm) { return *(volatile const int *)&sm.abort_flag != 0; }
__device__ __forceinline__ void set_abort(Smem &sm) { *(volatile int *)&sm.abort_flag = 1; }

// Barrier over the 128 threads of one warpgroup, bounded like every other wait (a plain
// bar.sync would hang if a warp of the group had given up).  `phase` counts completed uses.
__device__ __forceinline__ bool group_sync(uint64_t *bar, uint32_t &phase, int *err, int code, const int *abort) {
  mbar_arrive(bar);
  const bool ok = mbar_wait(bar, phase & 1, err, code, abort);
  ++phase;
  return ok;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int DH, bool PAIR, typename TO>
__global__ void __launch_bounds__(kThreads, 1) fwd_tc_kernel(
    const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
    const __grid_constant__ CUtensorMap mapV, const float *__restrict__ gb, const float *__restrict__ gx,
    const float *__restrict__ gu, const float *__restrict__ cm, int S, int DV, float scale,
    const float *__restrict__ C_init, const float *__restrict__ n_init, TO *__restrict__ h,
    float *__restrict__ C_last, float *__restrict__ n_last, float *__restrict__ m_last, int *__restrict__ err) {
  constexpr int D = PAIR ? 2 * DH : DH;  // d_qk
  constexpr int QB = DH * 128;           // bytes of a [64 x DH] 2-byte tile (DH / 64 swizzled blocks)
  constexpr int STAGE = 2 * QB + 16384;  // q, k, v tiles of one chunk
  constexpr uint32_t kColC16 = DH;
  constexpr int NR = PAIR ? 32 : 64;     // output rows finalised per CTA
  static_assert(DH == 64 || DH == 128 || DH == 256, "DH");

  extern __shared__ uint8_t smem_dyn[];
  __shared__ Smem sm;
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t *const sP = base + 2 * STAGE;                                // fp16 P [64 x 64], K-major
  float *const SX = reinterpret_cast<float *>(sP + 8192);              // [2][32][64] partner's S rows
  float *const HX = reinterpret_cast<float *>(sP + 8192 + 16384);      // [128][32] partner's H^T cols
#define STQ(s_) (base + (s_) * STAGE)
#define STK(s_) (base + (s_) * STAGE + QB)
#define STV(s_) (base + (s_) * STAGE + 2 * QB)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = PAIR ? (int)cluster_ctarank() : 0;
  const int atile = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int a0 = atile * kTile, c0 = rank * DH, p = blockIdx.y;
  const int NC = S / kL;
  const int *abort_ptr = &sm.abort_flag;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.full[i], 2);
      mbar_init(&sm.empty[i], 1);
      mbar_init(&sm.bar_S[i], 1);
      mbar_init(&sm.bar_nq[i], 128);
      mbar_init(&sm.sx_full[i], 1);
      mbar_init(&sm.sx_free[i], 2);
    }
    mbar_init(&sm.sfree, 128);
    mbar_init(&sm.bar_U, 1);
    mbar_init(&sm.bar_H, 1);
    mbar_init(&sm.hfree, 128);
    mbar_init(&sm.cready, 128);
    mbar_init(&sm.opready, 128);
    mbar_init(&sm.pready, 128);
    mbar_init(&sm.fin, 1);
    mbar_init(&sm.hx_full, 1);
    mbar_init(&sm.hx_free, 4);
    for (int i = 0; i < 3; ++i) mbar_init(&sm.grp[i], 128);
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (PAIR) cluster_sync();  // the partner's barriers are initialised before any remote access
  const uint32_t tm = sm.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&mapQ);
      prefetch_tensormap(&mapK);
      prefetch_tensormap(&mapV);
      int issued = 0;
      for (int k = 0; k < NC; ++k) {
        const int s = k & 1;
        if (k >= 2 && !mbar_wait(&sm.empty[s], ((k >> 1) - 1) & 1, err, 11, abort_ptr)) { set_abort(sm); break; }
        if (aborted(sm)) break;
        TRACE(0, k, 0);
        mbar_arrive_expect_tx(&sm.full[s], (uint32_t)STAGE);
        const int row = p * S + k * kL;
#pragma unroll
        for (int kb = 0; kb < DH / 64; ++kb) {
          tma_load_2d(STQ(s) + kb * 8192, &mapQ, c0 + kb * 64, row, &sm.full[s]);
          tma_load_2d(STK(s) + kb * 8192, &mapK, c0 + kb * 64, row, &sm.full[s]);
        }
        tma_load_2d(STV(s), &mapV, a0, row, &sm.full[s]);
        tma_load_2d(STV(s) + 8192, &mapV, a0 + 64, row, &sm.full[s]);
        issued = k + 1;
      }
      // the copies of the last stages land before the CTA may leave
      for (int k = issued >= 2 ? issued - 2 : 0; k < issued; ++k) mbar_wait(&sm.full[k & 1], (k >> 1) & 1, err, 19);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_S = idesc_f16(64, kL, /*bf16*/ 1, 0, 0);
      const uint32_t id_X = idesc_f16(kTile, kL, 0, 0, 0);
      const uint32_t id_U = idesc_f16(kTile, DH, 0, /*a MN-major*/ 1, /*b MN-major*/ 1);
      const uint32_t id_P = idesc_f16(kTile, NR, 0, 1, 0);
      const uint32_t sP_own = smem_u32(sP) + (PAIR ? rank * 32 * 128 : 0);
      int k = 0;
      for (; k < NC; ++k) {
        const int s = k & 1;
        // S_k = Q K^T over this CTA's d_qk columns
        if (!mbar_wait(&sm.full[s], (k >> 1) & 1, err, 12, abort_ptr)) break;
        if (k >= 1 && !mbar_wait(&sm.sfree, (k - 1) & 1, err, 13, abort_ptr)) break;
        tc_fence_after();
        TRACE(1, k, 0);
        const uint32_t q_s = smem_u32(STQ(s)), k_s = smem_u32(STK(s)), v_s = smem_u32(STV(s));
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
          mma_f16_ss(tm + kColS, smem_desc(q_s + off, 16, 1024, kSwizzle128B),
                     smem_desc(k_s + off, 16, 1024, kSwizzle128B), id_S, kk > 0);
        }
        mma_commit(&sm.bar_S[s]);
        // H^T = C16 (beta q)^T and T += V^T (w k): need the state copy, the scaled operands and a free H
        if (!mbar_wait(&sm.cready, k & 1, err, 14, abort_ptr)) break;
        TRACE(1, k, 1);
        if (!mbar_wait(&sm.opready, k & 1, err, 15, abort_ptr)) break;
        TRACE(1, k, 2);
        if (k >= 1 && !mbar_wait(&sm.hfree, (k - 1) & 1, err, 16, abort_ptr)) break;
        TRACE(1, k, 3);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
          mma_f16_ts(tm + kColH, tm + kColC16 + kk * 8, smem_desc(q_s + off, 16, 1024, kSwizzle128B), id_X,
                     kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < kL / 16; ++kk)
          mma_f16_ss(tm, smem_desc(v_s + kk * 2048, 8192, 1024, kSwizzle128B),
                     smem_desc(k_s + kk * 2048, 8192, 1024, kSwizzle128B), id_U, 1);
        mma_commit(&sm.bar_U);
        // H^T[:, own rows] += V^T P^T
        if (!mbar_wait(&sm.pready, k & 1, err, 17, abort_ptr)) break;
        TRACE(1, k, 4);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kL / 16; ++kk)
          mma_f16_ss(tm + kColH + (PAIR ? rank * 32 : 0), smem_desc(v_s + kk * 2048, 8192, 1024, kSwizzle128B),
                     smem_desc(sP_own + kk * 32, 16, 1024, kSwizzle128B), id_P, 1);
        mma_commit(&sm.bar_H);
        mma_commit(&sm.empty[s]);
      }
      if (k < NC) set_abort(sm);
      mma_commit(&sm.fin);  // completes once every MMA issued above has finished
      mbar_wait(&sm.fin, 0, err, 18);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------------ gate factors
    float sigma = 0.f;  // frame of T entering the chunk: C = exp(sigma) T
    for (int k = 0; k < NC; ++k) {
      const int s = k & 1;
      if (k >= 2 && !mbar_wait(&sm.empty[s], ((k >> 1) - 1) & 1, err, 41, abort_ptr)) { set_abort(sm); break; }
      if (aborted(sm)) break;
      const size_t tok0 = (size_t)p * S + (size_t)k * kL;
      const float m_in = cm[(size_t)p * (NC + 1) + k], m_out = cm[(size_t)p * (NC + 1) + k + 1];
      float bb[2], xx[2], uu[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        bb[i] = gb[tok0 + 32 * i + lane];
        xx[i] = gx[tok0 + 32 * i + lane];
        uu[i] = gu[tok0 + 32 * i + lane];
      }
      const float bl = __shfl_sync(0xffffffffu, bb[1], 31);
      const float log_alpha = bl + m_in - m_out;  // <= 0
      const bool lazy = -(sigma + log_alpha) <= kRescaleLog;
      const float sig_next = lazy ? sigma + log_alpha : 0.f;
      Gate &g = sm.g[s];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = 32 * i + lane;
        const float mr = fmaxf(m_in, uu[i]);
        g.mr[r] = mr;
        g.floor_[r] = __expf(-(bb[i] + mr));
        g.beta[r] = __expf(m_in - mr);
        g.xg[r] = xx[i];
        g.wk[r] = __expf(bl + xx[i] - m_out - sig_next) * scale;
        g.wt[r] = __expf(bl + xx[i] - m_out) * scale;
      }
      if (lane == 0) {
        g.alpha = __expf(log_alpha);
        g.fr_c = __expf(sigma);
        g.fr_w = __expf(sigma + log_alpha);
        g.sig_next = sig_next;
        g.lazy = lazy ? 1 : 0;
      }
      sigma = sig_next;
      __syncwarp();
      if (lane == 0) {
        TRACE(2, k, 0);
        mbar_arrive(&sm.full[s]);
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------------ warpgroup 1: P and h
    const int t = threadIdx.x - 128;  // tensor-memory lane = d_v row within the tile
    const int q4 = warp & 3;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const int r_s = 16 * q4 + (lane & 15);  // S row held by this lane (M = 64 layout, lanes < 16)
    const bool own_rows = !PAIR || ((q4 >> 1) == rank);
    const int r_lo = PAIR ? 32 * rank : 0;
    const int prt = 1 - rank;
    uint32_t gph = 0;
    for (int k = 0; k < NC; ++k) {
      const int s = k & 1, par = k & 1;
      const size_t tok0 = (size_t)p * S + (size_t)k * kL;
      if (!mbar_wait(&sm.full[s], (k >> 1) & 1, err, 21, abort_ptr)) { set_abort(sm); break; }
      if (!mbar_wait(&sm.bar_S[s], (k >> 1) & 1, err, 22, abort_ptr)) { set_abort(sm); break; }
      if (t == 0) TRACE(3, k, 0);
      tc_fence_after();
      float srow[kL];
      {
        uint32_t u[4][16];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld16(tm + lane_base + kColS + 16 * c, u[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 16; ++i) srow[16 * c + i] = __uint_as_float(u[c][i]);
      }
      tc_fence_before();
      mbar_arrive(&sm.sfree);
      if (!mbar_wait(&sm.bar_nq[s], (k >> 1) & 1, err, 23, abort_ptr)) { set_abort(sm); break; }
      if (t == 0) TRACE(3, k, 1);
      if (PAIR && !own_rows) {
        // partial S rows and n.q of the partner's rows -> partner
        if (k >= 2 && !mbar_wait_cluster(&sm.sx_free[par], ((k >> 1) - 1) & 1, err, 24, abort_ptr)) {
          set_abort(sm);
          break;
        }
        if (lane < 16) {
          const int rr = r_s - 32 * prt;
          const uint32_t rbar = mapa_shared(smem_u32(&sm.sx_full[par]), prt);
          const uint32_t dst = mapa_shared(smem_u32(SX + (par * 32 + rr) * 64), prt);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            st_async_v4(dst + ((i ^ (rr & 7)) << 4), srow[4 * i], srow[4 * i + 1], srow[4 * i + 2], srow[4 * i + 3],
                        rbar);
          st_async_f32(mapa_shared(smem_u32(&sm.nqx[par][rr]), prt), sm.nq[s][r_s], rbar);
        }
      } else {
        if (PAIR) {
          if (lane == 0 && q4 == 2 * rank) mbar_arrive_expect_tx(&sm.sx_full[par], 32 * 64 * 4 + 32 * 4);
          if (!mbar_wait_cluster(&sm.sx_full[par], (k >> 1) & 1, err, 25, abort_ptr)) { set_abort(sm); break; }
          if (t == 0) TRACE(3, k, 2);
        }
        if (lane < 16) {
          const Gate &g = sm.g[s];
          float nqf = sm.nq[s][r_s];
          if (PAIR) {
            const int rr = r_s - 32 * rank;
            const float *src = SX + (par * 32 + rr) * 64;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float4 v4 = *reinterpret_cast<const float4 *>(src + 4 * (i ^ (rr & 7)));
              srow[4 * i] += v4.x;
              srow[4 * i + 1] += v4.y;
              srow[4 * i + 2] += v4.z;
              srow[4 * i + 3] += v4.w;
            }
            nqf += sm.nqx[par][rr];
          }
          const float mrr = g.mr[r_s];
          float den = 0.f;
          uint8_t *prow = sP + r_s * 128;
#pragma unroll
          for (int c8 = 0; c8 < kL / 8; ++c8) {
            float pv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int j = c8 * 8 + i;
              pv[i] = (j <= r_s) ? srow[j] * scale * __expf(g.xg[j] - mrr) : 0.f;
              den += pv[i];
            }
            uint4 w4;
            w4.x = pack_half2(pv[0], pv[1]);
            w4.y = pack_half2(pv[2], pv[3]);
            w4.z = pack_half2(pv[4], pv[5]);
            w4.w = pack_half2(pv[6], pv[7]);
            *reinterpret_cast<uint4 *>(prow + ((c8 ^ (r_s & 7)) << 4)) = w4;
          }
          den += g.beta[r_s] * nqf;
          sm.inv[par][r_s] = 1.f / fmaxf(fabsf(den), g.floor_[r_s]);
        }
        if (PAIR) {
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&sm.sx_free[par]), prt));
        }
      }
      fence_proxy_async_smem();
      if (t == 0) TRACE(3, k, 3);
      mbar_arrive(&sm.pready);
      // inv[] of this chunk visible to the whole warpgroup
      if (!group_sync(&sm.grp[0], gph, err, 29, abort_ptr)) { set_abort(sm); break; }
      // -------------------------------- epilogue: h rows of this CTA
      if (!mbar_wait(&sm.bar_H, k & 1, err, 26, abort_ptr)) { set_abort(sm); break; }
      if (t == 0) TRACE(3, k, 4);
      tc_fence_after();
      float hv[kL];
      {
        uint32_t u[4][16];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld16(tm + lane_base + kColH + 16 * c, u[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 16; ++i) hv[16 * c + i] = __uint_as_float(u[c][i]);
      }
      tc_fence_before();
      mbar_arrive(&sm.hfree);
      float own[NR];
      if (PAIR) {
        if (k >= 1 && !mbar_wait_cluster(&sm.hx_free, (k - 1) & 1, err, 27, abort_ptr)) { set_abort(sm); break; }
        const uint32_t rbar = mapa_shared(smem_u32(&sm.hx_full), prt);
        const uint32_t dst = mapa_shared(smem_u32(HX + t * 32), prt);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float e[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) e[j] = rank ? hv[4 * i + j] : hv[32 + 4 * i + j];
          st_async_v4(dst + ((i ^ (t & 7)) << 4), e[0], e[1], e[2], e[3], rbar);
        }
        if (t == 0) mbar_arrive_expect_tx(&sm.hx_full, 128 * 32 * 4);
        if (!mbar_wait_cluster(&sm.hx_full, k & 1, err, 28, abort_ptr)) { set_abort(sm); break; }
        if (t == 0) TRACE(3, k, 5);
        const float *src = HX + t * 32;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 v4 = *reinterpret_cast<const float4 *>(src + 4 * (i ^ (t & 7)));
          own[4 * i] = (rank ? hv[32 + 4 * i] : hv[4 * i]) + v4.x;
          own[4 * i + 1] = (rank ? hv[32 + 4 * i + 1] : hv[4 * i + 1]) + v4.y;
          own[4 * i + 2] = (rank ? hv[32 + 4 * i + 2] : hv[4 * i + 2]) + v4.z;
          own[4 * i + 3] = (rank ? hv[32 + 4 * i + 3] : hv[4 * i + 3]) + v4.w;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&sm.hx_free), prt));
      } else {
#pragma unroll
        for (int i = 0; i < NR; ++i) own[i] = hv[i];
      }
      TO *hp = h + (tok0 + r_lo) * DV + a0 + t;
#pragma unroll
      for (int i = 0; i < NR; ++i) hp[(size_t)i * DV] = from_f32<TO>(own[i] * sm.inv[par][r_lo + i]);
      if (t == 0) TRACE(3, k, 6);
    }
  } else if (warp >= 8 && warp < 12) {
    // ------------------------------------------------------------------ warpgroup 2: state copy
    const int t = threadIdx.x - 256;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    for (int c = 0; c < DH; c += 16) {
      uint32_t r[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        r[i] = __float_as_uint(C_init ? C_init[((size_t)p * DV + a0 + t) * D + c0 + c + i] : 0.f);
      tmem_st16(tm + lane_base + c, r);
    }
    tmem_wait_st();
    float sig_last = 0.f;
    bool ok = true;
    for (int k = 0; k < NC; ++k) {
      const int s = k & 1;
      if (!mbar_wait(&sm.full[s], (k >> 1) & 1, err, 31, abort_ptr)) { ok = false; break; }
      if (k >= 1 && !mbar_wait(&sm.bar_U, (k - 1) & 1, err, 32, abort_ptr)) { ok = false; break; }
      if (t == 0) TRACE(4, k, 0);
      tc_fence_after();
      const Gate &g = sm.g[s];
      const float fr_c = g.fr_c, fr_w = g.fr_w;
      const bool lazy = g.lazy != 0;
      sig_last = g.sig_next;
#pragma unroll 1
      for (int c = 0; c < DH; c += 32) {
        uint32_t u0[16], u1[16];
        tmem_ld16(tm + lane_base + c, u0);
        tmem_ld16(tm + lane_base + c + 16, u1);
        tmem_wait_ld();
        uint32_t hv[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          hv[i] = pack_half2(__uint_as_float(u0[2 * i]) * fr_c, __uint_as_float(u0[2 * i + 1]) * fr_c);
          hv[8 + i] = pack_half2(__uint_as_float(u1[2 * i]) * fr_c, __uint_as_float(u1[2 * i + 1]) * fr_c);
        }
        if (!lazy) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            u0[i] = __float_as_uint(__uint_as_float(u0[i]) * fr_w);
            u1[i] = __float_as_uint(__uint_as_float(u1[i]) * fr_w);
          }
          tmem_st16(tm + lane_base + c, u0);
          tmem_st16(tm + lane_base + c + 16, u1);
        }
        tmem_st16(tm + lane_base + kColC16 + c / 2, hv);
      }
      tmem_wait_st();
      tc_fence_before();
      if (t == 0) TRACE(4, k, 1);
      mbar_arrive(&sm.cready);
    }
    if (!ok) set_abort(sm);
    // final state C_last = exp(sigma) T, transposed through shared memory for coalesced stores
    if (ok && !mbar_wait(&sm.bar_U, (NC - 1) & 1, err, 33, abort_ptr)) ok = false;
    if (ok) {
      tc_fence_after();
      const float fr = __expf(sig_last);
      float *buf = reinterpret_cast<float *>(base + (((NC - 1) & 1) ^ 1) * STAGE);  // stage unused by chunk NC-1
      const int wq = warp & 3;
      uint32_t gph = 0;
#pragma unroll 1
      for (int c = 0; c < DH; c += 32) {
        uint32_t u0[16], u1[16];
        tmem_ld16(tm + lane_base + c, u0);
        tmem_ld16(tm + lane_base + c + 16, u1);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          buf[t * 33 + i] = __uint_as_float(u0[i]) * fr;
          buf[t * 33 + 16 + i] = __uint_as_float(u1[i]) * fr;
        }
        if (!group_sync(&sm.grp[1], gph, err, 34, abort_ptr)) break;
#pragma unroll 4
        for (int rr = 0; rr < 32; ++rr) {
          const int row = wq * 32 + rr;
          C_last[((size_t)p * DV + a0 + row) * D + c0 + c + lane] = buf[row * 33 + lane];
        }
        if (!group_sync(&sm.grp[1], gph, err, 35, abort_ptr)) break;
      }
    } else {
      set_abort(sm);
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------------ warpgroup 3: operands and n
    const int t = threadIdx.x - 384;
    constexpr int CPR = DH / 8;    // 16-byte chunks per row
    constexpr int RG = 128 / CPR;  // rows handled at once
    const int cc = t % CPR, rg = t / CPR;
    const int colb = (cc >> 3) * 8192, c8 = cc & 7;
    for (int c = t; c < DH; c += 128) sm.n[c] = n_init ? n_init[(size_t)p * D + c0 + c] : 0.f;
    uint32_t gph = 0;
    bool ok = group_sync(&sm.grp[2], gph, err, 50, abort_ptr);
    for (int k = 0; ok && k < NC; ++k) {
      const int s = k & 1;
      if (!mbar_wait(&sm.full[s], (k >> 1) & 1, err, 51, abort_ptr)) { ok = false; break; }
      if (!mbar_wait(&sm.bar_S[s], (k >> 1) & 1, err, 52, abort_ptr)) { ok = false; break; }
      if (t == 0) TRACE(5, k, 0);
      const Gate &g = sm.g[s];
      const float alpha = g.alpha;
      float nreg[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) nreg[e] = sm.n[cc * 8 + e];
      // q: n . q_r over this CTA's columns, and beta_r q_r in fp16 (in place)
#pragma unroll 2
      for (int i = 0; i < 64 / RG; ++i) {
        const int r = rg + RG * i;
        uint4 *ptr = reinterpret_cast<uint4 *>(STQ(s) + colb + r * 128 + ((c8 ^ (r & 7)) << 4));
        const uint4 raw = *ptr;
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
        float f[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          f[2 * e] = bf16_lo(w[e]);
          f[2 * e + 1] = bf16_hi(w[e]);
        }
        float part = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) part = fmaf(f[e], nreg[e], part);
#pragma unroll
        for (int o = CPR / 2; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (cc == 0) sm.nq[s][r] = part;
        const float bq = g.beta[r];
        uint4 o4;
        o4.x = pack_half2(f[0] * bq, f[1] * bq);
        o4.y = pack_half2(f[2] * bq, f[3] * bq);
        o4.z = pack_half2(f[4] * bq, f[5] * bq);
        o4.w = pack_half2(f[6] * bq, f[7] * bq);
        *ptr = o4;
      }
      if (t == 0) TRACE(5, k, 1);
      mbar_arrive(&sm.bar_nq[s]);
      // k: n-update partial sums, and w_j k_j (frame of T) in fp16 (in place)
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll 2
      for (int i = 0; i < 64 / RG; ++i) {
        const int j = rg + RG * i;
        uint4 *ptr = reinterpret_cast<uint4 *>(STK(s) + colb + j * 128 + ((c8 ^ (j & 7)) << 4));
        const uint4 raw = *ptr;
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
        float f[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          f[2 * e] = bf16_lo(w[e]);
          f[2 * e + 1] = bf16_hi(w[e]);
        }
        const float wt = g.wt[j], wkj = g.wk[j];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(wt, f[e], acc[e]);
        uint4 o4;
        o4.x = pack_half2(f[0] * wkj, f[1] * wkj);
        o4.y = pack_half2(f[2] * wkj, f[3] * wkj);
        o4.z = pack_half2(f[4] * wkj, f[5] * wkj);
        o4.w = pack_half2(f[6] * wkj, f[7] * wkj);
        *ptr = o4;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) sm.npart[rg * DH + cc * 8 + e] = acc[e];
      // v: bf16 -> fp16 (exact), in place
      uint4 *vp = reinterpret_cast<uint4 *>(STV(s));
#pragma unroll 2
      for (int i = t; i < 1024; i += 128) {
        const uint4 raw = vp[i];
        uint4 o4;
        o4.x = pack_half2(bf16_lo(raw.x), bf16_hi(raw.x));
        o4.y = pack_half2(bf16_lo(raw.y), bf16_hi(raw.y));
        o4.z = pack_half2(bf16_lo(raw.z), bf16_hi(raw.z));
        o4.w = pack_half2(bf16_lo(raw.w), bf16_hi(raw.w));
        vp[i] = o4;
      }
      fence_proxy_async_smem();
      if (t == 0) TRACE(5, k, 2);
      mbar_arrive(&sm.opready);
      // every partial of this chunk written
      if (!group_sync(&sm.grp[2], gph, err, 53, abort_ptr)) { ok = false; break; }
      for (int c = t; c < DH; c += 128) {
        float a = 0.f;
#pragma unroll
        for (int gi = 0; gi < RG; ++gi) a += sm.npart[gi * DH + c];
        sm.n[c] = alpha * sm.n[c] + a;
      }
      // n after chunk k visible before the next n . q
      if (!group_sync(&sm.grp[2], gph, err, 54, abort_ptr)) { ok = false; break; }
      if (t == 0) TRACE(5, k, 3);
    }
    if (!ok) set_abort(sm);
    if (ok && atile == 0) {
      for (int c = t; c < DH; c += 128) n_last[(size_t)p * D + c0 + c] = sm.n[c];
      if (rank == 0 && t == 0) m_last[p] = cm[(size_t)p * (NC + 1) + NC];
    }
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // no CTA leaves while its partner may still access its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tm, 512);
  }
#undef STQ
#undef STK
#undef STV
}

// Dynamic shared memory: two stages, P, the pair exchange buffers and alignment slack; never
// less than 120 KB, so that one CTA (which allocates all 512 tensor-memory columns) runs per SM.
template <int DH, bool PAIR>
size_t smem_bytes() {
  const size_t need = (size_t)2 * (2 * DH * 128 + 16384) + 8192 + (PAIR ? 32768 : 0) + 1024;
  return need > 120 * 1024 ? need : 120 * 1024;
}

template <int DH, bool PAIR, typename TO>
cudaError_t launch_one(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv, const float *gb,
                       const float *gx, const float *gu, const float *cm, int P, int S, int DV, float scale,
                       const float *C_init, const float *n_init, void *h, float *C_last, float *n_last,
                       float *m_last, int *err, cudaStream_t stream) {
  auto kern = fwd_tc_kernel<DH, PAIR, TO>;
  const size_t smem = smem_bytes<DH, PAIR>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((DV / kTile) * (PAIR ? 2 : 1), P, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, gb, gx, gu, cm, S, DV, scale, C_init, n_init,
                            static_cast<TO *>(h), C_last, n_last, m_last, err);
}

template <typename TO>
cudaError_t launch_dispatch(int DH, bool pair, const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                            const float *gb, const float *gx, const float *gu, const float *cm, int P, int S,
                            int DV, float scale, const float *C_init, const float *n_init, void *h, float *C_last,
                            float *n_last, float *m_last, int *err, cudaStream_t stream) {
#define MLSTM_TC_CASE(dh_, pr_)                                                                                  \
  if (DH == dh_ && pair == pr_)                                                                                  \
    return launch_one<dh_, pr_, TO>(mq, mk, mv, gb, gx, gu, cm, P, S, DV, scale, C_init, n_init, h, C_last,     \
                                    n_last, m_last, err, stream);
  MLSTM_TC_CASE(64, false)
  MLSTM_TC_CASE(128, false)
  MLSTM_TC_CASE(256, false)
  MLSTM_TC_CASE(64, true)
  MLSTM_TC_CASE(128, true)
  MLSTM_TC_CASE(256, true)
#undef MLSTM_TC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

bool fwd_tc_supported(int S, int L, int D, int DV, bool bf16) {
  return bf16 && L == kL && (D == 64 || D == 128 || D == 256 || D == 512) && DV % kTile == 0 && S > 0 &&
         S % kL == 0;
}

bool fwd_tc_pair(int P, int D, int DV) {
  // d_qk = 512 only fits split over a pair; smaller heads split when that fills more of the SMs.
  return D == 512 || (D >= 128 && (long long)P * (DV / kTile) < 148);
}

cudaError_t launch_fwd_tc(const void *q, const void *k, const void *v, bool out_bf16, const float *gb,
                          const float *gx, const float *gu, const float *cm, int P, int S, int D, int DV,
                          const float *C_init, const float *n_init, void *h, float *C_last, float *n_last,
                          float *m_last, int *err, cudaStream_t stream) {
  const bool pair = fwd_tc_pair(P, D, DV);
  const int DH = pair ? D / 2 : D;
  CUtensorMap mq, mk, mv;
  if (!make_tmap_2d_b16(&mq, q, true, (uint64_t)P * S, D, D, 64, kL)) return cudaErrorInvalidValue;
  if (!make_tmap_2d_b16(&mk, k, true, (uint64_t)P * S, D, D, 64, kL)) return cudaErrorInvalidValue;
  if (!make_tmap_2d_b16(&mv, v, true, (uint64_t)P * S, DV, DV, 64, kL)) return cudaErrorInvalidValue;
  const float scale = (float)(1.0 / __builtin_sqrt((double)D));
  if (out_bf16)
    return launch_dispatch<__nv_bfloat16>(DH, pair, mq, mk, mv, gb, gx, gu, cm, P, S, DV, scale, C_init, n_init, h,
                                          C_last, n_last, m_last, err, stream);
  return launch_dispatch<float>(DH, pair, mq, mk, mv, gb, gx, gu, cm, P, S, DV, scale, C_init, n_init, h, C_last,
                                n_last, m_last, err, stream);
}

}  // namespace mlstm
