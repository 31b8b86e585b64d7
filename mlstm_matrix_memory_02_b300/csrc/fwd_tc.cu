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
// q and k pass through two shared-memory stages.  A stage is read raw by the S product and then
// converted in place: q to beta q (B operand of the C q product), k to w k (B operand of the
// state update).  With two stages the operands of chunk k+1 are formed while chunk k's products
// run, so the serial chain of the recurrence is only: state copy to fp16, C q, state update.
//
// Warp roles (640 threads): warp 1 allocates tensor memory, issues the state chain's MMAs (C q,
// the update) and the TMA loads of q and k into the stage each update frees; warp 0 issues the S
// and P V products; warp 3 issues the TMA loads of v (two stages, L2 prefetch two chunks ahead
// for q, k and v); warp 2
// preprocesses the gates and computes the per-chunk factors; warpgroup 1 (warps 4-7) reads S,
// forms w k and the n-update partial sums, then P and the denominators; warpgroup 2 (warps 8-11)
// copies the state to fp16 (the serial chain) and stores the final state; warpgroup 3 (warps
// 12-15) keeps n and forms v and beta q in fp16 and n.q; warpgroup 4 (warps 16-19) reads H,
// completes it with the partner's columns and writes h.  Hand-offs use mbarriers; every wait is
// bounded in time and reports through an error word.
//
// Operand precision: q, k, v arrive as bf16 and convert to fp16 exactly; the computed operands
// (P, beta q, w k and the state copy) are rounded to fp16 (11 significant bits); sums are fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.cuh"
#include "sm100.cuh"
#include "tmap.cuh"


namespace mlstm {
namespace {

using namespace sm100;

constexpr int kL = 64;        // chunk length
constexpr int kTile = 128;    // d_v rows per CTA (MMA M)
constexpr int kThreads = 640;
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
  uint64_t qk_full[2], qk_empty[2], v_full[2], v_empty[2], g_full[2], bar_nq[2];
  uint64_t bar_S[2], xready[2], kready[2];  // by chunk parity: the producers may run a chunk ahead
  uint64_t sfree, bar_X, bar_U, bar_H, hfree, cready, npart_free, pready, fin;
  uint64_t sx_full[2], sx_free[2], hx_full, hx_free, nqx_full[2], nqx_free[2];
  uint64_t inv_ready[2], inv_free[2];  // 1/den of a chunk: written by warpgroup 1, read by warpgroup 4
  uint64_t grp[3];  // bounded group barriers of warpgroups 1, 2 and 3
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) Gate g[2];
  alignas(16) float n[2][256];    // normaliser entering chunk k in n[k & 1], this CTA's d_qk columns
  alignas(16) float npart[1024];  // n-update partial sums of a chunk (warpgroup 1 -> warpgroup 3)
  float nq[2][kL];       // n . q_r over this CTA's columns
  float nqx[2][32];      // partner's n . q_r for the rows finalised here (written remotely)
  float inv[2][kL];      // 1 / max(|den_r|, exp(-m_r))
  float m_fin;           // stabiliser after the last chunk
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

// Packed pairs of fp32 (Blackwell f32x2 arithmetic: one instruction for two lanes of data).
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// bf16 pair -> fp32 pair
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) { return f2pack(bf16_lo(w), bf16_hi(w)); }
// fp32 pair -> fp16 pair (round to nearest)
__device__ __forceinline__ uint32_t f2_to_h2(uint64_t x) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
  return pack_half2(lo, hi);
}
__device__ __forceinline__ float f2sum(uint64_t x) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
  return lo + hi;
}

template <int DH, bool PAIR, typename TO>
__global__ void __launch_bounds__(kThreads, 1) fwd_tc_kernel(
    const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
    const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapC,
    const float *__restrict__ gb, const float *__restrict__ gx, const float *__restrict__ gu,
    const float *__restrict__ cm, const float *__restrict__ igp, const float *__restrict__ fgp,
    const float *__restrict__ m_init, int S, int DV, float scale, const float *__restrict__ C_init,
    const float *__restrict__ n_init, TO *__restrict__ h, float *__restrict__ n_last, float *__restrict__ m_last,
    int *__restrict__ err, int exp_fg) {
  constexpr int D = PAIR ? 2 * DH : DH;  // d_qk
  constexpr int QB = DH * 128;           // bytes of a [64 x DH] 2-byte tile (DH / 64 swizzled blocks)
  constexpr uint32_t kColC16 = DH;
  constexpr int NR = PAIR ? 32 : 64;     // output rows finalised per CTA
  static_assert(DH == 64 || DH == 128 || DH == 256, "DH");
  // dynamic shared memory map (every region 1024-byte aligned)
  constexpr int OFF_V = 4 * QB;  // [0, 4 QB): two stages of (q, k)
  constexpr int OFF_P = OFF_V + 2 * 16384, OFF_SO = OFF_P + 8192, OFF_SX = OFF_SO + NR * 256;
  constexpr int OFF_HX = OFF_SX + 16384;

  extern __shared__ uint8_t smem_dyn[];
  __shared__ Smem sm;
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t *const sP = base + OFF_P;    // P, fp16 [64 x 64], K-major
  float *const SO = reinterpret_cast<float *>(base + OFF_SO);  // this CTA's partial S rows [NR][64]
  float *const SX = reinterpret_cast<float *>(base + OFF_SX);  // [2][32][64] partner's partial S rows
  float *const HX = reinterpret_cast<float *>(base + OFF_HX);  // [128][32] partner's H^T columns
// stage s of q (raw bf16 from TMA with 128-byte swizzle, then beta q in fp16) and of k (raw,
// then w k in fp16); v stage s (bf16, then fp16)
#define STQ(s_) (base + (2 * (s_)) * QB)
#define STK(s_) (base + (2 * (s_) + 1) * QB)
#define STV(s_) (base + OFF_V + (s_) * 16384)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = PAIR ? (int)cluster_ctarank() : 0;
  const int atile = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int a0 = atile * kTile, c0 = rank * DH, p = blockIdx.y;
  const int NC = S / kL;
  const int r_lo = PAIR ? 32 * rank : 0;  // first output row finalised here
  const int prt = 1 - rank;
  const int *abort_ptr = &sm.abort_flag;

  // The wait-error word starts at zero for this launch (a wait only gives up after about a
  // second, long after the first CTA has started).
  if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) *(volatile int *)err = 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.qk_full[i], 1);
      mbar_init(&sm.qk_empty[i], 1);  // committed after the state update that last reads the stage
      mbar_init(&sm.v_full[i], 1);
      mbar_init(&sm.v_empty[i], 2);  // the state update (warp 1) and P V (warp 0) of the chunk
      mbar_init(&sm.g_full[i], 1);
      mbar_init(&sm.bar_nq[i], 128);
      mbar_init(&sm.sx_full[i], 1);
      mbar_init(&sm.sx_free[i], 4);
      mbar_init(&sm.nqx_full[i], 1);
      mbar_init(&sm.nqx_free[i], 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.bar_S[i], 1);
      mbar_init(&sm.xready[i], 128);  // warpgroup 3: beta q and v in fp16
      mbar_init(&sm.kready[i], 128);  // warpgroup 1: w k in fp16 and the n-update partial sums
    }
    mbar_init(&sm.sfree, 128);
    mbar_init(&sm.bar_X, 1);
    mbar_init(&sm.bar_U, 1);
    mbar_init(&sm.bar_H, 1);
    mbar_init(&sm.hfree, 128);
    mbar_init(&sm.cready, 128);
    mbar_init(&sm.npart_free, 128);  // warpgroup 3 has read the partial sums
    mbar_init(&sm.pready, 128);
    mbar_init(&sm.fin, 2);  // both MMA issuers
    mbar_init(&sm.hx_full, 1);
    mbar_init(&sm.hx_free, 4);
    for (int i = 0; i < 3; ++i) mbar_init(&sm.grp[i], 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.inv_ready[i], 128);
      mbar_init(&sm.inv_free[i], 128);
    }
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
    // ------------------------------------------------------------------ MMA issuer: S and P V
    if (lane == 0) {
      const uint32_t id_S = idesc_f16(64, kL, /*bf16*/ 1, 0, 0);
      const uint32_t id_P = idesc_f16(kTile, NR, 0, 1, 0);
      const uint64_t dp_own = smem_desc(smem_u32(sP) + r_lo * 128, 16, 1024, kSwizzle128B);
      // per step k: S_k = Q K^T (raw bf16 inputs) once its stage has landed and the S columns are
      // free, then H^T[own rows] += V^T P^T of chunk k-1 once P is formed and X_{k-1} is done
      int k = 0;
      for (; k <= NC; ++k) {
        if (k < NC) {
          const int s = k & 1;
          if (!mbar_wait(&sm.qk_full[s], (k >> 1) & 1, err, 12, abort_ptr)) break;
          if (k >= 1 && !mbar_wait(&sm.sfree, (k - 1) & 1, err, 13, abort_ptr)) break;
          tc_fence_after();
          const uint64_t dq_raw = smem_desc(smem_u32(STQ(s)), 16, 1024, kSwizzle128B);
          const uint64_t dk_raw = smem_desc(smem_u32(STK(s)), 16, 1024, kSwizzle128B);
#pragma unroll 1
          for (int c = 0; c < DH / 16; ++c) {
            const uint64_t off = (uint64_t)(((c >> 2) * 8192 + (c & 3) * 32) >> 4);
            mma_f16_ss(tm + kColS, dq_raw + off, dk_raw + off, id_S, c > 0);
          }
          mma_commit(&sm.bar_S[s]);
        }
        if (k >= 1) {
          const int kp = k - 1;
          if (!mbar_wait(&sm.pready, kp & 1, err, 17, abort_ptr)) break;
          if (!mbar_wait(&sm.bar_X, kp & 1, err, 9, abort_ptr)) break;
          tc_fence_after();
          const uint64_t dv = smem_desc(smem_u32(STV(kp & 1)), 8192, 1024, kSwizzle128B);
#pragma unroll 1
          for (int kk = 0; kk < kL / 16; ++kk)
            mma_f16_ss(tm + kColH + r_lo, dv + (uint64_t)(kk * 2048 >> 4), dp_own + (uint64_t)(kk * 32 >> 4), id_P, 1);
          mma_commit(&sm.bar_H);
          mma_commit(&sm.v_empty[kp & 1]);
        }
      }
      if (k <= NC) set_abort(sm);
      mma_commit(&sm.fin);
      mbar_wait(&sm.fin, 0, err, 8);
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------------ TMA: v (two stages)
    if (lane == 0) {
      prefetch_tensormap(&mapV);
      int issued = 0;
      for (int k = 0; k < NC; ++k) {
        const int s = k & 1;
        if (k >= 2 && !mbar_wait(&sm.v_empty[s], ((k >> 1) - 1) & 1, err, 61, abort_ptr)) { set_abort(sm); break; }
        if (aborted(sm)) break;
        mbar_arrive_expect_tx(&sm.v_full[s], 16384u);
        const int row = p * S + k * kL;
        tma_load_2d(STV(s), &mapV, a0, row, &sm.v_full[s]);
        tma_load_2d(STV(s) + 8192, &mapV, a0 + 64, row, &sm.v_full[s]);
        if (k + 2 < NC) {
          tma_prefetch_2d(&mapV, a0, row + 2 * kL);
          tma_prefetch_2d(&mapV, a0 + 64, row + 2 * kL);
        }
        issued = k + 1;
      }
      for (int k = issued >= 2 ? issued - 2 : 0; k < issued; ++k)
        mbar_wait(&sm.v_full[k & 1], (k >> 1) & 1, err, 69);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_X = idesc_f16(kTile, kL, 0, 0, 0);
      const uint32_t id_U = idesc_f16(kTile, DH, 0, /*a MN-major*/ 1, /*b MN-major*/ 1);
      // The state chain: X_k (H^T = C16 (beta q)^T) and U_k (T += V^T (w k)), and the q/k loads
      // of chunk k+2 into the stage that U_k frees.  S and P V are issued by warp 0, so that
      // neither chain waits behind the other.  Descriptors are advanced by adding (byte offset >> 4)
      // to the start-address field; the loops stay rolled.
      prefetch_tensormap(&mapQ);
      prefetch_tensormap(&mapK);
      auto load_qk = [&](int kk) {
        const int s = kk & 1, row = p * S + kk * kL;
        mbar_arrive_expect_tx(&sm.qk_full[s], (uint32_t)(2 * QB));
#pragma unroll 1
        for (int kb = 0; kb < DH / 64; ++kb) {
          tma_load_2d(STQ(s) + kb * 8192, &mapQ, c0 + kb * 64, row, &sm.qk_full[s]);
          tma_load_2d(STK(s) + kb * 8192, &mapK, c0 + kb * 64, row, &sm.qk_full[s]);
          if (kk + 2 < NC) {
            tma_prefetch_2d(&mapQ, c0 + kb * 64, row + 2 * kL);
            tma_prefetch_2d(&mapK, c0 + kb * 64, row + 2 * kL);
          }
        }
      };
      for (int kk = 0; kk < 2 && kk < NC; ++kk) load_qk(kk);
      int k = 0;
      for (; k < NC; ++k) {
        const int s = k & 1;
        if (!mbar_wait(&sm.cready, k & 1, err, 14, abort_ptr)) break;
        if (!mbar_wait(&sm.xready[s], (k >> 1) & 1, err, 15, abort_ptr)) break;
        if (k >= 1 && !mbar_wait(&sm.hfree, (k - 1) & 1, err, 16, abort_ptr)) break;
        tc_fence_after();
        const uint64_t dq_b = smem_desc(smem_u32(STQ(s)), 16, 1024, kSwizzle128B);
#pragma unroll 1
        for (int kk = 0; kk < DH / 16; ++kk)
          mma_f16_ts(tm + kColH, tm + kColC16 + kk * 8, dq_b + (uint64_t)(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4),
                     id_X, kk > 0);
        mma_commit(&sm.bar_X);
        if (!mbar_wait(&sm.kready[s], (k >> 1) & 1, err, 10, abort_ptr)) break;
        tc_fence_after();
        const uint64_t dv = smem_desc(smem_u32(STV(s)), 8192, 1024, kSwizzle128B);
        const uint64_t dk_w = smem_desc(smem_u32(STK(s)), 8192, 1024, kSwizzle128B);
#pragma unroll 1
        for (int kk = 0; kk < kL / 16; ++kk)
          mma_f16_ss(tm, dv + (uint64_t)(kk * 2048 >> 4), dk_w + (uint64_t)(kk * 2048 >> 4), id_U, 1);
        mma_commit(&sm.bar_U);
        mma_commit(&sm.qk_empty[s]);
        mma_commit(&sm.v_empty[s]);  // with warp 0's commit after P V
        // stage s is free once X_k and U_k (the last readers of beta q and w k) are done
        if (k + 2 < NC) {
          if (!mbar_wait(&sm.qk_empty[s], (k >> 1) & 1, err, 11, abort_ptr)) break;
          load_qk(k + 2);
        }
      }
      if (k < NC) set_abort(sm);
      mma_commit(&sm.fin);  // completes once every MMA issued above has finished
      mbar_wait(&sm.fin, 0, err, 18);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------------ gate factors
    float sigma = 0.f;  // frame of T entering the chunk: C = exp(sigma) T
    float m_chain = m_init ? m_init[p] : 0.f;  // stabiliser entering the chunk (raw-gate mode)
    // raw pre-activations of the next chunk, loaded one chunk ahead
    float2 f2n = make_float2(0.f, 0.f), i2n = f2n;
    if (igp != nullptr && NC > 0) {
      f2n = *reinterpret_cast<const float2 *>(fgp + (size_t)p * S + 2 * lane);
      i2n = *reinterpret_cast<const float2 *>(igp + (size_t)p * S + 2 * lane);
    }
    for (int k = 0; k < NC; ++k) {
      const int s = k & 1;
      // the factors of chunk k share the lifetime of v stage s (free once PV of chunk k-2 is done)
      if (k >= 2 && !mbar_wait(&sm.v_empty[s], ((k >> 1) - 1) & 1, err, 41, abort_ptr)) { set_abort(sm); break; }
      if (aborted(sm)) break;
      const size_t tok0 = (size_t)p * S + (size_t)k * kL;
      // b, x = i~ - b and the running max u for rows 2 lane and 2 lane + 1, and the chunk's
      // stabiliser chain m_out = b_L + max(m_in, u_L)
      float bb[2], xx[2], uu[2], m_in, m_out;
      if (igp != nullptr) {
        // from the raw pre-activations (the same operations, in the same order, as the gate kernel)
        const float2 f2 = f2n, i2 = i2n;
        if (k + 1 < NC) {
          f2n = *reinterpret_cast<const float2 *>(fgp + tok0 + kL + 2 * lane);
          i2n = *reinterpret_cast<const float2 *>(igp + tok0 + kL + 2 * lane);
        }
        float lf0 = log_forget(f2.x, exp_fg), lf1 = log_forget(f2.y, exp_fg);
        float bsum = lf0;
        bsum += lf1;
        lf1 = bsum;
        float incl = bsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const float excl = incl - bsum;
        bb[0] = lf0 + excl;
        bb[1] = lf1 + excl;
        xx[0] = i2.x - bb[0];
        xx[1] = i2.y - bb[1];
        float imax = fmaxf(fmaxf(-INFINITY, xx[0]), xx[1]);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, imax, o);
          if (lane >= o) imax = fmaxf(imax, y);
        }
        float run = __shfl_up_sync(0xffffffffu, imax, 1);
        if (lane == 0) run = -INFINITY;
        run = fmaxf(run, xx[0]);
        uu[0] = run;
        run = fmaxf(run, xx[1]);
        uu[1] = run;
        m_in = m_chain;
        m_out = __shfl_sync(0xffffffffu, bb[1], 31) + fmaxf(m_in, __shfl_sync(0xffffffffu, uu[1], 31));
        m_chain = m_out;
      } else {
        m_in = cm[(size_t)p * (NC + 1) + k];
        m_out = cm[(size_t)p * (NC + 1) + k + 1];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          bb[i] = gb[tok0 + 2 * lane + i];
          xx[i] = gx[tok0 + 2 * lane + i];
          uu[i] = gu[tok0 + 2 * lane + i];
        }
      }
      const float bl = __shfl_sync(0xffffffffu, bb[1], 31);
      const float log_alpha = bl + m_in - m_out;  // <= 0
      const bool lazy = -(sigma + log_alpha) <= kRescaleLog;
      const float sig_next = lazy ? sigma + log_alpha : 0.f;
      Gate &g = sm.g[s];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = 2 * lane + i;
        const float mr = fmaxf(m_in, uu[i]);
        g.mr[r] = mr;
        g.floor_[r] = __expf(-(bb[i] + mr));
        g.beta[r] = __expf(m_in - mr);
        g.xg[r] = xx[i];
        g.wk[r] = __expf(bl + xx[i] - m_out - sig_next) * scale;
        g.wt[r] = __expf(bl + xx[i] - m_out) * scale;
      }
      if (lane == 0) {
        if (k == NC - 1) sm.m_fin = m_out;
        g.alpha = __expf(log_alpha);
        g.fr_c = __expf(sigma);
        g.fr_w = __expf(sigma + log_alpha);
        g.sig_next = sig_next;
        g.lazy = lazy ? 1 : 0;
      }
      sigma = sig_next;
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.g_full[s]);
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------------ warpgroup 1: S, w k and P
    // Per chunk: the S rows (own rows kept, the partner's sent), then w k and the n-update partial
    // sums while the partner's S rows are in flight, then P and the denominators.
    const int t = threadIdx.x - 128;  // tensor-memory lane = d_v row within the tile
    const int q4 = warp & 3;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const int r_s = 16 * q4 + (lane & 15);  // S row held by this lane (M = 64 layout, lanes < 16)
    const bool own_rows = !PAIR || ((q4 >> 1) == rank);
    constexpr int TPR = 128 / NR;  // P formation: threads per row (4 with a pair, 2 without)
    constexpr int SEG = kL / TPR;  // columns per thread (16 or 32)
    const int pi = t / TPR, pseg = t % TPR;
    const int pr = r_lo + pi;  // the row this thread forms
    constexpr int KCPR = DH / 8;     // w k pass: 16-byte chunks per row of k
    constexpr int KRG = 128 / KCPR;  // rows handled at once (column layout)
    const int kcc = t % KCPR, krg = t / KCPR;
    const int kcolb = (kcc >> 3) * 8192, kc8 = kcc & 7;
    uint32_t gph = 0;

    // S rows of chunk kk: own rows -> SO, the partner's rows -> partner's SX
    auto s_read = [&](int kk) -> bool {
      const int s = kk & 1, par = kk & 1;
      if (!mbar_wait(&sm.g_full[s], (kk >> 1) & 1, err, 21, abort_ptr)) return false;
      if (!mbar_wait(&sm.bar_S[kk & 1], (kk >> 1) & 1, err, 22, abort_ptr)) return false;
      tc_fence_after();
      uint32_t u[2][32];
      tmem_ld32(tm + lane_base + kColS, u[0]);
      tmem_ld32(tm + lane_base + kColS + 32, u[1]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&sm.sfree);
      // S of the next chunk can complete before every thread is done with the previous P rows:
      // SO is rewritten only after the whole group has left the previous p_form
      if (kk >= 1 && !group_sync(&sm.grp[0], gph, err, 38, abort_ptr)) return false;
      if (own_rows) {
        if (lane < 16) {
          const int i = r_s - r_lo;
          float *dst = SO + i * 64;
#pragma unroll
          for (int c = 0; c < 16; ++c)
            *reinterpret_cast<float4 *>(dst + 4 * (c ^ (i & 7))) =
                make_float4(__uint_as_float(u[c >> 3][(4 * c) & 31]), __uint_as_float(u[c >> 3][(4 * c + 1) & 31]),
                            __uint_as_float(u[c >> 3][(4 * c + 2) & 31]), __uint_as_float(u[c >> 3][(4 * c + 3) & 31]));
        }
      } else if (PAIR) {
        if (kk >= 2 && !mbar_wait_cluster(&sm.sx_free[par], ((kk >> 1) - 1) & 1, err, 24, abort_ptr)) return false;
        if (lane < 16) {
          const int rr = r_s - 32 * prt;
          const uint32_t rbar = mapa_shared(smem_u32(&sm.sx_full[par]), prt);
          const uint32_t dst = mapa_shared(smem_u32(SX + (par * 32 + rr) * 64), prt);
#pragma unroll
          for (int c = 0; c < 16; ++c)
            st_async_v4(dst + ((c ^ (rr & 7)) << 4), __uint_as_float(u[c >> 3][(4 * c) & 31]),
                        __uint_as_float(u[c >> 3][(4 * c + 1) & 31]), __uint_as_float(u[c >> 3][(4 * c + 2) & 31]),
                        __uint_as_float(u[c >> 3][(4 * c + 3) & 31]), rbar);
        }
      }
      return true;
    };

    // w_j k_j (frame of T) in fp16, in place over the raw k of the stage, and the n-update partial
    // sums sum_j w_j k_j / sqrt(d) (column layout), once the S product of the chunk has read raw k
    auto k_pass = [&](int kk) -> bool {
      const int s = kk & 1;
      if (!mbar_wait(&sm.qk_full[s], (kk >> 1) & 1, err, 36, abort_ptr)) return false;
      if (kk >= 1 && !mbar_wait(&sm.npart_free, (kk - 1) & 1, err, 37, abort_ptr)) return false;
      const Gate &g = sm.g[s];
      uint8_t *const kb = STK(s);
      // rows in batches of four: every load of a batch is issued before its stores
      uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll 1
      for (int i0 = 0; i0 < 64 / KRG; i0 += 4) {
        uint4 raw[4];
        int off[4];
        float wt[4], wk[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int j = krg + KRG * (i0 + b);
          off[b] = kcolb + j * 128 + ((kc8 ^ (j & 7)) << 4);
          raw[b] = *reinterpret_cast<const uint4 *>(kb + off[b]);
          wt[b] = g.wt[j];
          wk[b] = g.wk[j];
        }
        uint4 o4[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const uint64_t wt2 = f2pack(wt[b], wt[b]), wk2 = f2pack(wk[b], wk[b]);
          const uint64_t x0 = bf2_to_f2(raw[b].x), x1 = bf2_to_f2(raw[b].y), x2 = bf2_to_f2(raw[b].z),
                         x3 = bf2_to_f2(raw[b].w);
          acc[0] = f2fma(wt2, x0, acc[0]);
          acc[1] = f2fma(wt2, x1, acc[1]);
          acc[2] = f2fma(wt2, x2, acc[2]);
          acc[3] = f2fma(wt2, x3, acc[3]);
          o4[b].x = f2_to_h2(f2mul(x0, wk2));
          o4[b].y = f2_to_h2(f2mul(x1, wk2));
          o4[b].z = f2_to_h2(f2mul(x2, wk2));
          o4[b].w = f2_to_h2(f2mul(x3, wk2));
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) *reinterpret_cast<uint4 *>(kb + off[b]) = o4[b];
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) *reinterpret_cast<uint64_t *>(&sm.npart[krg * DH + kcc * 8 + 2 * e]) = acc[e];
      fence_proxy_async_smem();
      mbar_arrive(&sm.kready[kk & 1]);
      return true;
    };

    // P rows of chunk kk (needs SO of every warp: call after a group barrier) and their 1/den
    auto p_form = [&](int kk) -> bool {
      const int s = kk & 1, par = kk & 1;
      if (PAIR) {
        if (t == 0) {
          mbar_arrive_expect_tx(&sm.sx_full[par], 32 * 64 * 4);
          mbar_arrive_expect_tx(&sm.nqx_full[par], 32 * 4);
        }
        if (!mbar_wait_cluster(&sm.sx_full[par], (kk >> 1) & 1, err, 25, abort_ptr)) return false;
        if (!mbar_wait_cluster(&sm.nqx_full[par], (kk >> 1) & 1, err, 30, abort_ptr)) return false;
      }
      if (!mbar_wait(&sm.bar_nq[par], (kk >> 1) & 1, err, 23, abort_ptr)) return false;
      // P of the previous chunk has been read by its P V product (which may run after S of this chunk)
      if (kk >= 1 && !mbar_wait(&sm.bar_H, (kk - 1) & 1, err, 39, abort_ptr)) return false;
      const Gate &g = sm.g[s];
      const float mrr = g.mr[pr];
      const float *so = SO + pi * 64;
      const float *sx = SX + (par * 32 + pi) * 64;
      float den = 0.f;
#pragma unroll
      for (int h16 = 0; h16 < SEG / 16; ++h16) {
        const int j0 = SEG * pseg + 16 * h16;  // first column of this block
        float sv[16], xv[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int c4 = j0 / 4 + q;
          float4 a = *reinterpret_cast<const float4 *>(so + 4 * (c4 ^ (pi & 7)));
          if (PAIR) {
            const float4 b = *reinterpret_cast<const float4 *>(sx + 4 * (c4 ^ (pi & 7)));
            a.x += b.x;
            a.y += b.y;
            a.z += b.z;
            a.w += b.w;
          }
          const float4 xq = *reinterpret_cast<const float4 *>(&g.xg[j0 + 4 * q]);
          sv[4 * q] = a.x;
          sv[4 * q + 1] = a.y;
          sv[4 * q + 2] = a.z;
          sv[4 * q + 3] = a.w;
          xv[4 * q] = xq.x;
          xv[4 * q + 1] = xq.y;
          xv[4 * q + 2] = xq.z;
          xv[4 * q + 3] = xq.w;
        }
        float pv[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float pe = sv[e] * scale * __expf(xv[e] - mrr);
          pv[e] = (j0 + e <= pr) ? pe : 0.f;
        }
        float d8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) d8[e] = pv[e] + pv[e + 8];
        den += ((d8[0] + d8[4]) + (d8[1] + d8[5])) + ((d8[2] + d8[6]) + (d8[3] + d8[7]));
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int cb = j0 / 8 + hh;  // 16-byte chunk of the P row (8 fp16 columns)
          uint4 w4;
          w4.x = pack_half2(pv[8 * hh], pv[8 * hh + 1]);
          w4.y = pack_half2(pv[8 * hh + 2], pv[8 * hh + 3]);
          w4.z = pack_half2(pv[8 * hh + 4], pv[8 * hh + 5]);
          w4.w = pack_half2(pv[8 * hh + 6], pv[8 * hh + 7]);
          *reinterpret_cast<uint4 *>(sP + pr * 128 + ((cb ^ (pr & 7)) << 4)) = w4;
        }
      }
#pragma unroll
      for (int o = 1; o < TPR; o <<= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
      // warpgroup 4 has read this slot's 1/den for chunk kk-2
      if (kk >= 2 && !mbar_wait(&sm.inv_free[par], ((kk >> 1) - 1) & 1, err, 31, abort_ptr)) return false;
      if (pseg == 0) {
        // denominator of row pr: intra-chunk part + beta_r n.q_r (both halves of d_qk with a pair)
        float nqf = sm.nq[par][pr];
        if (PAIR) nqf += sm.nqx[par][pi];
        const float dn = den + g.beta[pr] * nqf;
        sm.inv[par][pr] = 1.f / fmaxf(fabsf(dn), g.floor_[pr]);
      }
      if (PAIR) {
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_remote(mapa_shared(smem_u32(&sm.sx_free[par]), prt));
          mbar_arrive_remote(mapa_shared(smem_u32(&sm.nqx_free[par]), prt));
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&sm.pready);
      mbar_arrive(&sm.inv_ready[par]);
      return true;
    };

    bool ok = true;
    for (int k = 0; ok && k < NC; ++k) {
      if (!s_read(k) || !k_pass(k) || !group_sync(&sm.grp[0], gph, err, 20, abort_ptr) || !p_form(k)) ok = false;
    }
    if (!ok) set_abort(sm);
  } else if (warp >= 16) {
    // ------------------------------------------------------------------ warpgroup 4: h
    const int t = threadIdx.x - 512;  // tensor-memory lane = d_v row within the tile
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    bool ok = true;
    for (int k = 0; k < NC; ++k) {
      const int par = k & 1;
      const size_t tok0 = (size_t)p * S + (size_t)k * kL;
      // H^T of chunk k: send the partner's columns, keep this CTA's rows, free the accumulator
      if (!mbar_wait(&sm.bar_H, k & 1, err, 26, abort_ptr)) { ok = false; break; }
      tc_fence_after();
      float own[NR];
      if (PAIR) {
        if (k >= 1 && !mbar_wait_cluster(&sm.hx_free, (k - 1) & 1, err, 27, abort_ptr)) { ok = false; break; }
        {
          uint32_t u[32];
          tmem_ld32(tm + lane_base + kColH + 32 * prt, u);  // the partner's 32 rows
          tmem_wait_ld();
          const uint32_t rbar = mapa_shared(smem_u32(&sm.hx_full), prt);
          const uint32_t dst = mapa_shared(smem_u32(HX + t * 32), prt);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            st_async_v4(dst + ((i ^ (t & 7)) << 4), __uint_as_float(u[4 * i]), __uint_as_float(u[4 * i + 1]),
                        __uint_as_float(u[4 * i + 2]), __uint_as_float(u[4 * i + 3]), rbar);
        }
        {
          uint32_t u[32];
          tmem_ld32(tm + lane_base + kColH + 32 * rank, u);  // this CTA's rows
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) own[i] = __uint_as_float(u[i]);
        }
      } else {
        uint32_t u[32];
        tmem_ld32(tm + lane_base + kColH, u);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) own[i] = __uint_as_float(u[i]);
        tmem_ld32(tm + lane_base + kColH + 32, u);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) own[32 + i] = __uint_as_float(u[i]);
      }
      tc_fence_before();
      mbar_arrive(&sm.hfree);
      if (PAIR) {
        if (t == 0) mbar_arrive_expect_tx(&sm.hx_full, 128 * 32 * 4);
        if (!mbar_wait_cluster(&sm.hx_full, k & 1, err, 28, abort_ptr)) { ok = false; break; }
        const float *src = HX + t * 32;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 v4 = *reinterpret_cast<const float4 *>(src + 4 * (i ^ (t & 7)));
          own[4 * i] += v4.x;
          own[4 * i + 1] += v4.y;
          own[4 * i + 2] += v4.z;
          own[4 * i + 3] += v4.w;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&sm.hx_free), prt));
      }
      // 1/den of every row of chunk k (warpgroup 1)
      if (!mbar_wait(&sm.inv_ready[par], (k >> 1) & 1, err, 29, abort_ptr)) { ok = false; break; }
      TO *hp = h + (tok0 + r_lo) * DV + a0 + t;
#pragma unroll
      for (int i = 0; i < NR; ++i) hp[(size_t)i * DV] = from_f32<TO>(own[i] * sm.inv[par][r_lo + i]);
      mbar_arrive(&sm.inv_free[par]);
    }
    if (!ok) set_abort(sm);
  } else if (warp >= 8 && warp < 12) {
    // ------------------------------------------------------------------ warpgroup 2: state copy
    const int t = threadIdx.x - 256;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    uint32_t gph2 = 0;
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
      if (!mbar_wait(&sm.g_full[s], (k >> 1) & 1, err, 40, abort_ptr)) { ok = false; break; }
      if (k >= 1 && !mbar_wait(&sm.bar_U, (k - 1) & 1, err, 32, abort_ptr)) { ok = false; break; }
      tc_fence_after();
      const Gate &g = sm.g[s];
      const float fr_c = g.fr_c, fr_w = g.fr_w;
      const bool lazy = g.lazy != 0;
      sig_last = g.sig_next;
      if (lazy) {
        // C16 = fp16(exp(sigma) T): the next 32 columns load while the current ones convert
        uint32_t ua[32], ub[32];
        tmem_ld32(tm + lane_base, ua);
        tmem_wait_ld();
#pragma unroll 1
        for (int c = 0; c < DH; c += 64) {
          tmem_ld32(tm + lane_base + c + 32, ub);
          {
            uint32_t hv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              hv[i] = pack_half2(__uint_as_float(ua[2 * i]) * fr_c, __uint_as_float(ua[2 * i + 1]) * fr_c);
            tmem_st16(tm + lane_base + kColC16 + c / 2, hv);
          }
          tmem_wait_ld();
          if (c + 64 < DH) tmem_ld32(tm + lane_base + c + 64, ua);
          {
            uint32_t hv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              hv[i] = pack_half2(__uint_as_float(ub[2 * i]) * fr_c, __uint_as_float(ub[2 * i + 1]) * fr_c);
            tmem_st16(tm + lane_base + kColC16 + c / 2 + 16, hv);
          }
          tmem_wait_ld();
        }
      } else {
        // eager: also write the decayed state back to frame 0
#pragma unroll 1
        for (int c = 0; c < DH; c += 32) {
          uint32_t u[32];
          tmem_ld32(tm + lane_base + c, u);
          tmem_wait_ld();
          uint32_t hv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            hv[i] = pack_half2(__uint_as_float(u[2 * i]) * fr_c, __uint_as_float(u[2 * i + 1]) * fr_c);
          tmem_st16(tm + lane_base + kColC16 + c / 2, hv);
          uint32_t w0[16], w1[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            w0[i] = __float_as_uint(__uint_as_float(u[i]) * fr_w);
            w1[i] = __float_as_uint(__uint_as_float(u[16 + i]) * fr_w);
          }
          tmem_st16(tm + lane_base + c, w0);
          tmem_st16(tm + lane_base + c + 16, w1);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&sm.cready);
    }
    if (ok && atile == 0 && rank == 0 && t == 0) m_last[p] = sm.m_fin;
    if (!ok) set_abort(sm);
    // final state C_last = exp(sigma) T, transposed through shared memory for coalesced stores
    if (ok && !mbar_wait(&sm.bar_U, (NC - 1) & 1, err, 33, abort_ptr)) ok = false;
    if (ok) {
      // C_last = exp(sigma) T, 32 columns at a time through two swizzled staging tiles
      // [128 rows x 128 bytes] in the (now unused) q/k stages, stored by TMA
      tc_fence_after();
      const float fr = __expf(sig_last);
#pragma unroll 1
      for (int c = 0, slab = 0; c < DH; c += 32, ++slab) {
        uint8_t *tile = base + (slab & 1) * 16384;
        if (slab >= 2) {
          if (t == 0) bulk_wait_read<1>();  // the store that used this tile has read it
          if (!group_sync(&sm.grp[1], gph2, err, 34, abort_ptr)) break;
        }
        uint32_t u[32];
        tmem_ld32(tm + lane_base + c, u);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<float4 *>(tile + t * 128 + ((i ^ (t & 7)) << 4)) =
              make_float4(__uint_as_float(u[4 * i]) * fr, __uint_as_float(u[4 * i + 1]) * fr,
                          __uint_as_float(u[4 * i + 2]) * fr, __uint_as_float(u[4 * i + 3]) * fr);
        fence_proxy_async_smem();
        if (!group_sync(&sm.grp[1], gph2, err, 35, abort_ptr)) break;
        if (t == 0) {
          tma_store_2d(&mapC, c0 + c, p * DV + a0, tile);
          bulk_commit();
        }
      }
      if (t == 0) bulk_wait_all();
    } else {
      set_abort(sm);
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------------ warpgroup 3: n, v and beta q
    const int t = threadIdx.x - 384;
    constexpr int CPR = DH / 8;      // 16-byte chunks per row
    constexpr int KRG = 128 / CPR;   // row groups of warpgroup 1's n-update partial sums
    // row layout for q: two threads per row, each half of the row's chunks
    const int qr = t >> 1, qh = t & 1;
    for (int c = t; c < DH; c += 128) sm.n[0][c] = n_init ? n_init[(size_t)p * D + c0 + c] : 0.f;
    uint32_t gph = 0;
    float alpha_prev = 1.f;  // decay of the previous chunk
    // n after chunk kk (into n[(kk + 1) & 1]): alpha n + the partial sums of the w k pass; each
    // thread updates columns t and t + 128
    auto n_update = [&](int kk) -> bool {
      if (!mbar_wait(&sm.kready[kk & 1], (kk >> 1) & 1, err, 58, abort_ptr)) return false;
      const float *src = sm.n[kk & 1];
      float *dst = sm.n[(kk + 1) & 1];
      for (int c = t; c < DH; c += 128) {
        float a = 0.f;
#pragma unroll
        for (int gi = 0; gi < KRG; ++gi) a += sm.npart[gi * DH + c];
        dst[c] = alpha_prev * src[c] + a;
      }
      mbar_arrive(&sm.npart_free);
      return true;
    };
    bool ok = group_sync(&sm.grp[2], gph, err, 50, abort_ptr);
    for (int k = 0; ok && k < NC; ++k) {
      const int s = k & 1, par = k & 1;
      // n entering chunk k (every thread's columns in before any row reads them)
      if (k >= 1 && (!n_update(k - 1) || !group_sync(&sm.grp[2], gph, err, 59, abort_ptr))) { ok = false; break; }
      if (!mbar_wait(&sm.g_full[s], (k >> 1) & 1, err, 51, abort_ptr)) { ok = false; break; }
      if (!mbar_wait(&sm.v_full[s], (k >> 1) & 1, err, 55, abort_ptr)) { ok = false; break; }
      // v: bf16 -> fp16 (exact), in place
      {
        uint4 *vp = reinterpret_cast<uint4 *>(STV(s));
#pragma unroll 1
        for (int i0 = t; i0 < 1024; i0 += 4 * 128) {
          uint4 raw[4];
#pragma unroll
          for (int b = 0; b < 4; ++b) raw[b] = vp[i0 + 128 * b];
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            uint4 o4;
            o4.x = pack_half2(bf16_lo(raw[b].x), bf16_hi(raw[b].x));
            o4.y = pack_half2(bf16_lo(raw[b].y), bf16_hi(raw[b].y));
            o4.z = pack_half2(bf16_lo(raw[b].z), bf16_hi(raw[b].z));
            o4.w = pack_half2(bf16_lo(raw[b].w), bf16_hi(raw[b].w));
            vp[i0 + 128 * b] = o4;
          }
        }
      }
      // raw q of the stage has landed and the S product has read it
      if (!mbar_wait(&sm.qk_full[s], (k >> 1) & 1, err, 52, abort_ptr)) { ok = false; break; }
      if (!mbar_wait(&sm.bar_S[k & 1], (k >> 1) & 1, err, 56, abort_ptr)) { ok = false; break; }
      const Gate &g = sm.g[s];
      alpha_prev = g.alpha;
      uint8_t *const qb = STQ(s);
      const float *nk = sm.n[k & 1];
      // q: n . q_r over this CTA's columns and beta_r q_r in fp16 in place (row layout)
      {
        const float bq = g.beta[qr];
        const uint64_t bq2 = f2pack(bq, bq);
        uint64_t part2 = 0;
#pragma unroll 1
        for (int i0 = 0; i0 < CPR / 2; i0 += 4) {
          // chunks in batches of four: every load of a batch is issued before its stores
          uint4 raw[4], na[4], nb[4];
          int off[4];
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const int ch = qh * (CPR / 2) + i0 + b;  // chunk of the row
            off[b] = (ch >> 3) * 8192 + qr * 128 + (((ch & 7) ^ (qr & 7)) << 4);
            raw[b] = *reinterpret_cast<const uint4 *>(qb + off[b]);
            na[b] = *reinterpret_cast<const uint4 *>(&nk[ch * 8]);
            nb[b] = *reinterpret_cast<const uint4 *>(&nk[ch * 8 + 4]);
          }
          uint4 o4[4];
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const uint64_t x0 = bf2_to_f2(raw[b].x), x1 = bf2_to_f2(raw[b].y), x2 = bf2_to_f2(raw[b].z),
                           x3 = bf2_to_f2(raw[b].w);
            part2 = f2fma(x0, (uint64_t)na[b].x | ((uint64_t)na[b].y << 32), part2);
            part2 = f2fma(x1, (uint64_t)na[b].z | ((uint64_t)na[b].w << 32), part2);
            part2 = f2fma(x2, (uint64_t)nb[b].x | ((uint64_t)nb[b].y << 32), part2);
            part2 = f2fma(x3, (uint64_t)nb[b].z | ((uint64_t)nb[b].w << 32), part2);
            o4[b].x = f2_to_h2(f2mul(x0, bq2));
            o4[b].y = f2_to_h2(f2mul(x1, bq2));
            o4[b].z = f2_to_h2(f2mul(x2, bq2));
            o4[b].w = f2_to_h2(f2mul(x3, bq2));
          }
#pragma unroll
          for (int b = 0; b < 4; ++b) *reinterpret_cast<uint4 *>(qb + off[b]) = o4[b];
        }
        float part = f2sum(part2);
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        if (PAIR && (qr >> 5) == prt) {
          // n . q of the partner's rows -> partner (after it has used the previous one in this slot)
          if (k >= 2 && !mbar_wait_cluster(&sm.nqx_free[par], ((k >> 1) - 1) & 1, err, 57, abort_ptr)) {
            ok = false;
            break;
          }
          if (qh == 0)
            st_async_f32(mapa_shared(smem_u32(&sm.nqx[par][qr & 31]), prt), part,
                         mapa_shared(smem_u32(&sm.nqx_full[par]), prt));
        } else if (qh == 0) {
          sm.nq[par][qr] = part;
        }
      }
      mbar_arrive(&sm.bar_nq[par]);
      fence_proxy_async_smem();
      mbar_arrive(&sm.xready[k & 1]);
    }
    // n after the last chunk
    if (ok && NC > 0) ok = n_update(NC - 1);
    if (ok && atile == 0)
      for (int c = t; c < DH; c += 128) n_last[(size_t)p * D + c0 + c] = sm.n[NC & 1][c];
    if (!ok) set_abort(sm);
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // no CTA leaves while its partner may still access its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tm, 512);
  }
#undef STV
}

// Dynamic shared memory: raw and converted q/k tiles, two v stages, P, this CTA's partial S rows,
// the pair exchange buffers and alignment slack; never less than 120 KB, so that one CTA (which
// allocates all 512 tensor-memory columns) runs per SM.
template <int DH, bool PAIR>
size_t smem_bytes() {
  const size_t NR = PAIR ? 32 : 64;
  const size_t need = (size_t)4 * DH * 128 + 2 * 16384 + 8192 + NR * 256 + (PAIR ? 32768 : 0) + 1024;
  return need > 120 * 1024 ? need : 120 * 1024;
}

template <int DH, bool PAIR, typename TO>
cudaError_t launch_one(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mc,
                       const float *gb, const float *gx, const float *gu, const float *cm, const float *ig,
                       const float *fg, const float *m_init, int P, int S, int DV, float scale,
                       const float *C_init, const float *n_init, void *h, float *n_last, float *m_last, int *err,
                       int exp_fg, cudaStream_t stream) {
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
  return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mc, gb, gx, gu, cm, ig, fg, m_init, S, DV, scale, C_init, n_init,
                            static_cast<TO *>(h), n_last, m_last, err, exp_fg);
}

template <typename TO>
cudaError_t launch_dispatch(int DH, bool pair, const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                            const CUtensorMap &mc, const float *gb, const float *gx, const float *gu,
                            const float *cm, const float *ig, const float *fg, const float *m_init, int P, int S,
                            int DV, float scale, const float *C_init, const float *n_init, void *h, float *n_last,
                            float *m_last, int *err, int exp_fg, cudaStream_t stream) {
#define MLSTM_TC_CASE(dh_, pr_)                                                                                  \
  if (DH == dh_ && pair == pr_)                                                                                  \
    return launch_one<dh_, pr_, TO>(mq, mk, mv, mc, gb, gx, gu, cm, ig, fg, m_init, P, S, DV, scale, C_init,    \
                                    n_init, h, n_last, m_last, err, exp_fg, stream);
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
                          const float *gx, const float *gu, const float *cm, const float *ig, const float *fg,
                          const float *m_init, int P, int S, int D, int DV, const float *C_init,
                          const float *n_init, void *h, float *C_last, float *n_last, float *m_last, int *err,
                          cudaStream_t stream, bool exp_fg) {
  const bool pair = fwd_tc_pair(P, D, DV);
  const int DH = pair ? D / 2 : D;
  CUtensorMap mq, mk, mv, mc;
  if (!make_tmap_2d_b16(&mq, q, true, (uint64_t)P * S, D, D, 64, kL)) return cudaErrorInvalidValue;
  if (!make_tmap_2d_b16(&mk, k, true, (uint64_t)P * S, D, D, 64, kL)) return cudaErrorInvalidValue;
  if (!make_tmap_2d_b16(&mv, v, true, (uint64_t)P * S, DV, DV, 64, kL)) return cudaErrorInvalidValue;
  if (!make_tmap_2d_f32(&mc, C_last, (uint64_t)P * DV, D, kTile)) return cudaErrorInvalidValue;
  const float scale = (float)(1.0 / __builtin_sqrt((double)D));
  if (out_bf16)
    return launch_dispatch<__nv_bfloat16>(DH, pair, mq, mk, mv, mc, gb, gx, gu, cm, ig, fg, m_init, P, S, DV, scale,
                                          C_init, n_init, h, n_last, m_last, err, exp_fg ? 1 : 0, stream);
  return launch_dispatch<float>(DH, pair, mq, mk, mv, mc, gb, gx, gu, cm, ig, fg, m_init, P, S, DV, scale, C_init,
                                n_init, h, n_last, m_last, err, exp_fg ? 1 : 0, stream);
}

}  // namespace mlstm
