// fwd_tc.cu -- tensor-core chunkwise forward of the mLSTM cell: the inter-chunk recurrence and the
// intra-chunk output in one pass per (head, 128-row d_v tile[, d_qk half]), the matrix state
// resident in tensor memory for the whole sequence.
//
// Page "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural Networks"
// (llms.blog): section 3 "The Parallel Dual Form" (H = ((Q K^T) o D) V inside a chunk, the state
// unrolled across chunks), section 3 "Associative Matrix Cell State" (C and n updates, the
// retrieval h = C q / max(|n^T q|, .), k scaled by 1/sqrt(d)), section 2 (the max stabiliser).
// Per chunk k, entering state (C, n, m_in), and the per-token b (in-chunk prefix sum of log f),
// x = i~ - b and running max u (so the row stabiliser is m_r = b_r + mr_r, mr_r = max(m_in, u_r)):
//   S   = Q K^T                                   bf16 inputs, fp32 accumulate
//   P   = S / sqrt(d) * exp(x_j - mr_r), j <= r   fp32, rounded to fp16 for the next product
//   H^T = C (beta q)^T + V^T P^T,  beta_r = exp(m_in - mr_r)
//   h_r = H_r / max(|sum_j P_rj + beta_r n.q_r|, exp(-m_r))
//   C  <- alpha C + V^T diag(w) K / sqrt(d),  n <- alpha n + K^T w / sqrt(d)
//
// Work split.  A CTA owns 128 rows of d_v (MMA M) and DH columns of d_qk.  With PAIR, two CTAs of
// a cluster split d_qk in halves (DH = d_qk / 2): each holds its half of the state, computes
// partial Q K^T, n.q and C q sums over its half and exchanges them through distributed shared
// memory; CTA rank rho finalises output rows r in [32 rho, 32 rho + 32).
//
// Tensor memory (512 columns): [0, DH) fp32 state T, [DH, 3 DH / 2) its fp16 copy C16 (A operand
// of the C q product), [384, 448) S (M = 64 layout), [448, 512) H^T.  The state is kept in a
// lazily rescaled frame C = exp(sigma) T: the chunk decay is folded into sigma and into the scale
// of the update's k operand, and T is multiplied back only when exp(-sigma) would exceed 2^8.
//
// The tensor pipe serialises MMAs that accumulate into the same tensor-memory accumulator (about
// 96 cycles each for these shapes) but overlaps independent ones, and a commit covers every MMA
// its thread issued before it.  So the products of a chunk come from three issuers: warp 0 issues
// S, warp 1 the state update U and the C q product X, and the epilogue's first thread P V (whose
// commit then covers P V alone).  U and X are issued block by block as the conversion passes
// publish their operands (w k per 16 tokens, beta q per 64 columns of d_qk).  The loops that bound
// a chunk are
//   H:      X_k -> P V_k -> the epilogue loads H -> X_{k+1}
//   state:  U_k, X_k -> copy T -> C16 -> X_{k+1}
//   stage:  X_k frees its q/k stage -> TMA of chunk k+2 -> S_{k+2} -> conversions -> X_{k+2}
// and the CUDA-core passes are spread over four warpgroups so that each can finish inside them.
//
// Warp roles (640 threads, every hand-off an mbarrier, every wait bounded in time):
//   warp 0       MMA issuer: S_k, as soon as the raw q/k stage lands and S has been read
//   warp 1       tensor-memory allocation; MMA issuer: U_k and X_k, block by block
//   warp 2       TMA loads of v (two stages) and the gate preprocessing (prefix scans,
//                stabiliser chain, factors) two chunks ahead, into four gate slots
//   warp 3       TMA loads of q and k (two stages, L2 prefetch two chunks ahead)
//   warps 4-7    state copy T -> fp16 C16 (and the eager rescale); P and the denominators; the
//                final state
//   warps 8-11   P V (first thread); the epilogue: H from tensor memory, the partner's columns,
//                1/den, the h stores
//   warps 12-15  q -> beta q (fp16, in place) and the partial n.q; v of the next chunk -> fp16
//   warps 16-19  k -> w k (fp16, in place) and the n-update partial sums; S from tensor memory
//                (own rows kept, the partner's sent); the normaliser n
//
// Operand precision: q, k, v arrive as bf16 and convert to fp16 exactly; the computed operands
// (P, beta q, w k and the state copy) are rounded to fp16 (11 significant bits); sums are fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "f2math.cuh"
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
  uint64_t qk_full[2], qk_empty[2], v_full[2], v_empty[2], g_full[4];
  uint64_t bar_S[2], xready[2], vready[2], nready[2];
  uint64_t xblk[2][4];  // beta q of d_qk block b (64 columns) in fp16: warpgroup 3 -> X
  uint64_t kblk[2][4];  // w k of token block b (16 rows) in fp16: warpgroup 4 -> U
  uint64_t sfree, soready, sofree, bar_X, bar_H, hfree, cready, pready, fin;
  uint64_t sx_full[2], sx_free[2], hx_full, hx_free, nqx_full[2], nqx_free[2];
  uint64_t inv_ready[2], inv_free[2];  // 1/den of a chunk: warpgroup 1 -> warpgroup 2
  uint64_t grp[3];  // bounded group barriers of warpgroups 1, 2 and 4
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) Gate g[4];           // gate factors of chunk k in g[k & 3]
  alignas(16) float n[2][256];    // normaliser entering chunk k in n[k & 1], this CTA's d_qk columns
  alignas(16) float npart[1024];  // n-update partial sums of a chunk: [row group][column]
  alignas(16) float nq[2][kL];    // n . q_r over this CTA's columns (rows finalised here)
  alignas(16) float nqx[2][32];   // partner's n . q_r for the rows finalised here (written remotely)
  alignas(16) float inv[2][kL];   // 1 / max(|den_r|, exp(-m_r))
  float m_fin;                    // stabiliser after the last chunk
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

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.qk_full[i], 1);
      mbar_init(&sm.qk_empty[i], 1);  // committed after X_k, the last reader of the stage
      mbar_init(&sm.v_full[i], 1);
      mbar_init(&sm.v_empty[i], 2);   // U (warp 1) and P V (warp 0) of the chunk
      mbar_init(&sm.bar_S[i], 1);
      mbar_init(&sm.xready[i], 128);  // warpgroup 3: beta q and n . q
      for (int b = 0; b < 4; ++b) {
        mbar_init(&sm.xblk[i][b], 128);
        mbar_init(&sm.kblk[i][b], 128);
      }
      mbar_init(&sm.vready[i], 128);  // warpgroup 2: v in fp16
      mbar_init(&sm.sx_full[i], 1);
      mbar_init(&sm.sx_free[i], 4);
      mbar_init(&sm.nqx_full[i], 1);
      mbar_init(&sm.nqx_free[i], 4);
      mbar_init(&sm.nready[i], 128);  // warpgroup 4: n entering the chunk of this parity
      mbar_init(&sm.inv_ready[i], 128);
      mbar_init(&sm.inv_free[i], 128);
    }
    for (int i = 0; i < 4; ++i) mbar_init(&sm.g_full[i], 1);
    mbar_init(&sm.sfree, 128);    // warpgroup 4 has read S
    mbar_init(&sm.soready, 128);  // warpgroup 4 has written (or sent) its S rows
    mbar_init(&sm.sofree, 128);   // warpgroup 2 has formed P from them
    mbar_init(&sm.bar_X, 1);
    mbar_init(&sm.bar_H, 1);
    mbar_init(&sm.hfree, 128);
    mbar_init(&sm.cready, 128);
    mbar_init(&sm.pready, 128);
    mbar_init(&sm.fin, 3);  // the three MMA issuers (warps 0, 1 and 8)
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
    // ------------------------------------------------------------------ MMA issuer: S
    if (lane == 0) {
      const uint32_t id_S = idesc_f16(64, kL, /*bf16*/ 1, 0, 0);
      // S_k = Q K^T (raw bf16 inputs) once its stage has landed and the S columns are free.  P V is
      // issued by the epilogue's warpgroup, so that the commit it waits on covers no S product
      int k = 0;
      for (; k < NC; ++k) {
        {
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
      }
      if (k < NC) set_abort(sm);
      mma_commit(&sm.fin);
      mbar_wait(&sm.fin, 0, err, 8);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer: U and X
    if (lane == 0) {
      const uint32_t id_X = idesc_f16(kTile, kL, 0, 0, 0);
      const uint32_t id_U = idesc_f16(kTile, DH, 0, /*a MN-major*/ 1, /*b MN-major*/ 1);
      constexpr int NXB = DH / 64;  // d_qk blocks of X (four K = 16 steps each)
      // Per chunk k, once the copy of the state is done: U_k (T += V^T (w k), one K = 16 step per
      // token block of 16) and X_k (H^T = C16 (beta q)^T, four K = 16 steps per d_qk block of 64)
      // are issued block by block, whichever block's operands are ready first (X also needs the
      // epilogue of chunk k-1 to have read H), so that neither stream waits behind the other or
      // behind a whole conversion pass.  One commit after both covers them (the copy of chunk
      // k+1 waits for it).  Descriptors are advanced by adding (byte offset >> 4) to the
      // start-address field.
      int k = 0;
      for (; k < NC; ++k) {
        const int s = k & 1;
        const uint32_t par = (k >> 1) & 1;
        if (!mbar_wait(&sm.cready, k & 1, err, 14, abort_ptr)) break;
        if (!mbar_wait(&sm.vready[s], par, err, 19, abort_ptr)) break;
        const uint64_t dv = smem_desc(smem_u32(STV(s)), 8192, 1024, kSwizzle128B);
        const uint64_t dk_w = smem_desc(smem_u32(STK(s)), 8192, 1024, kSwizzle128B);
        const uint64_t dq_b = smem_desc(smem_u32(STQ(s)), 16, 1024, kSwizzle128B);
        bool hfree_ok = k == 0;
        int ub = 0, xb = 0;
        const long long t0 = clock64();
        bool ok = true;
        while (ub < 4 || xb < NXB) {
          bool progress = false;
          if (ub < 4 && mbar_test(&sm.kblk[s][ub], par)) {
            tc_fence_after();
            mma_f16_ss(tm, dv + (uint64_t)(ub * 2048 >> 4), dk_w + (uint64_t)(ub * 2048 >> 4), id_U, 1);
            ++ub;
            progress = true;
          }
          if (xb < NXB) {
            if (!hfree_ok) hfree_ok = mbar_test(&sm.hfree, (k - 1) & 1);
            if (hfree_ok && mbar_test(&sm.xblk[s][xb], par)) {
              tc_fence_after();
#pragma unroll
              for (int kk = 4 * xb; kk < 4 * xb + 4; ++kk)
                mma_f16_ts(tm + kColH, tm + kColC16 + kk * 8,
                           dq_b + (uint64_t)(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4), id_X, kk > 0);
              ++xb;
              progress = true;
            }
          }
          if (!progress) {
            if (aborted(sm) || clock64() - t0 > kWaitCycles) {
              atomicCAS(err, 0, 10);
              ok = false;
              break;
            }
            __nanosleep(32);
          }
        }
        if (!ok) break;
        mma_commit(&sm.bar_X);
        mma_commit(&sm.qk_empty[s]);
        mma_commit(&sm.v_empty[s]);  // with warp 0's commit after P V
      }
      if (k < NC) set_abort(sm);
      mma_commit(&sm.fin);  // completes once every MMA issued above has finished
      mbar_wait(&sm.fin, 0, err, 18);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------------ v loads and gate factors
    // v stage s and the gate slot s are free once chunk k-2 is done (its U and P V, which come
    // after every other reader of the chunk's gate factors)
    if (lane == 0) prefetch_tensormap(&mapV);
    float sigma = 0.f;  // frame of T entering the chunk: C = exp(sigma) T
    float m_chain = m_init ? m_init[p] : 0.f;  // stabiliser entering the chunk (raw-gate mode)
    // raw pre-activations of the next chunk, loaded one chunk ahead
    float2 f2n = make_float2(0.f, 0.f), i2n = f2n;
    if (igp != nullptr && NC > 0) {
      f2n = *reinterpret_cast<const float2 *>(fgp + (size_t)p * S + 2 * lane);
      i2n = *reinterpret_cast<const float2 *>(igp + (size_t)p * S + 2 * lane);
    }
    // gate factors of chunk kk into slot kk & 3 (chunks in order: the stabiliser chain is serial)
    auto gates = [&](int kk) {
        const size_t tok0 = (size_t)p * S + (size_t)kk * kL;
        // b, x = i~ - b and the running max u for rows 2 lane and 2 lane + 1, and the chunk's
        // stabiliser chain m_out = b_L + max(m_in, u_L)
        float bb[2], xx[2], uu[2], m_in, m_out;
        if (igp != nullptr) {
          // from the raw pre-activations (the same operations, in the same order, as the gate kernel)
          const float2 f2 = f2n, i2 = i2n;
          if (kk + 1 < NC) {
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
          m_in = cm[(size_t)p * (NC + 1) + kk];
          m_out = cm[(size_t)p * (NC + 1) + kk + 1];
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
        Gate &g = sm.g[kk & 3];
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
          if (kk == NC - 1) sm.m_fin = m_out;
          g.alpha = __expf(log_alpha);
          g.fr_c = __expf(sigma);
          g.fr_w = __expf(sigma + log_alpha);
          g.sig_next = sig_next;
          g.lazy = lazy ? 1 : 0;
        }
        sigma = sig_next;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.g_full[kk & 3]);
    };
    // The factors run two chunks ahead of the v loads: slot (k + 2) & 3 held chunk k-2, whose
    // readers are all done once its U and P V are (v_empty of chunk k-2).
    for (int kk = 0; kk < 2 && kk < NC; ++kk) gates(kk);
    int issued = 0;
    for (int k = 0; k < NC; ++k) {
      const int s = k & 1;
      int ok = 1;
      if (lane == 0) {
        if (k >= 2 && !mbar_wait(&sm.v_empty[s], ((k >> 1) - 1) & 1, err, 62, abort_ptr)) ok = 0;
        if (ok && !aborted(sm)) {
          const int row = p * S + k * kL;
          mbar_arrive_expect_tx(&sm.v_full[s], 16384u);
          tma_load_2d(STV(s), &mapV, a0, row, &sm.v_full[s]);
          tma_load_2d(STV(s) + 8192, &mapV, a0 + 64, row, &sm.v_full[s]);
          issued = k + 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok || aborted(sm)) {
        set_abort(sm);
        break;
      }
      if (k + 2 < NC) gates(k + 2);
    }
    if (lane == 0) {
      // nothing may leave while loads it issued are still landing
      for (int k = issued >= 2 ? issued - 2 : 0; k < issued; ++k) mbar_wait(&sm.v_full[k & 1], (k >> 1) & 1, err, 69);
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------------ q and k loads
    // stage s is free once X_{k-2} (and U_{k-2}), its last readers, are done
    if (lane == 0) {
      prefetch_tensormap(&mapQ);
      prefetch_tensormap(&mapK);
      int issued = 0;
      for (int k = 0; k < NC; ++k) {
        const int s = k & 1;
        if (k >= 2 && !mbar_wait(&sm.qk_empty[s], ((k >> 1) - 1) & 1, err, 61, abort_ptr)) {
          set_abort(sm);
          break;
        }
        if (aborted(sm)) break;
        const int row = p * S + k * kL;
        mbar_arrive_expect_tx(&sm.qk_full[s], (uint32_t)(2 * QB));
#pragma unroll 1
        for (int kb = 0; kb < DH / 64; ++kb) {
          tma_load_2d(STQ(s) + kb * 8192, &mapQ, c0 + kb * 64, row, &sm.qk_full[s]);
          tma_load_2d(STK(s) + kb * 8192, &mapK, c0 + kb * 64, row, &sm.qk_full[s]);
        }
        issued = k + 1;
        if (k + 2 < NC) {
#pragma unroll 1
          for (int kb = 0; kb < DH / 64; ++kb) {
            tma_prefetch_2d(&mapQ, c0 + kb * 64, row + 2 * kL);
            tma_prefetch_2d(&mapK, c0 + kb * 64, row + 2 * kL);
          }
        }
      }
      for (int k = issued >= 2 ? issued - 2 : 0; k < issued; ++k) mbar_wait(&sm.qk_full[k & 1], (k >> 1) & 1, err, 69);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------------ warpgroup 1: state copy, P
    const int t = threadIdx.x - 128;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    uint32_t gph = 0;
    for (int c = 0; c < DH; c += 16) {
      uint32_t r[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        r[i] = __float_as_uint(C_init ? C_init[((size_t)p * DV + a0 + t) * D + c0 + c + i] : 0.f);
      tmem_st16(tm + lane_base + c, r);
    }
    tmem_wait_st();
    constexpr int TPR = 128 / NR;  // P formation: threads per row (4 with a pair, 2 without)
    constexpr int SEG = kL / TPR;  // columns per thread (16 or 32)
    const int pi = t / TPR, pseg = t % TPR;
    const int pr = r_lo + pi;  // the row this thread forms
    // P rows of chunk kk and their 1/den: needs this CTA's S rows (warpgroup 4), the partner's
    // (distributed shared memory), n . q of both halves and P V_{kk-1} done with the P buffer
    auto p_form = [&](int kk) -> bool {
      const int s = kk & 1, par = kk & 1;
      if (!mbar_wait(&sm.soready, kk & 1, err, 20, abort_ptr)) return false;
      if (!mbar_wait(&sm.xready[s], (kk >> 1) & 1, err, 23, abort_ptr)) return false;
      if (kk >= 1 && !mbar_wait(&sm.bar_H, (kk - 1) & 1, err, 31, abort_ptr)) return false;
      if (PAIR) {
        if (t == 0) {
          mbar_arrive_expect_tx(&sm.sx_full[par], 32 * 64 * 4);
          mbar_arrive_expect_tx(&sm.nqx_full[par], 32 * 4);
        }
        if (!mbar_wait_cluster(&sm.sx_full[par], (kk >> 1) & 1, err, 25, abort_ptr)) return false;
        if (!mbar_wait_cluster(&sm.nqx_full[par], (kk >> 1) & 1, err, 30, abort_ptr)) return false;
      }
      const Gate &g = sm.g[kk & 3];
      const float mrr = g.mr[pr];
      const float *so = SO + pi * 64;
      const float *sx = SX + (par * 32 + pi) * 64;
      float den = 0.f;
#pragma unroll
      for (int h16 = 0; h16 < SEG / 16; ++h16) {
        const int j0 = SEG * pseg + 16 * h16;  // first column of this block
        float pv[16];
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
          pv[4 * q] = a.x * scale * __expf(xq.x - mrr);
          pv[4 * q + 1] = a.y * scale * __expf(xq.y - mrr);
          pv[4 * q + 2] = a.z * scale * __expf(xq.z - mrr);
          pv[4 * q + 3] = a.w * scale * __expf(xq.w - mrr);
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) pv[e] = (j0 + e <= pr) ? pv[e] : 0.f;
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
      // the epilogue of chunk kk-2 has read this slot of 1/den
      if (kk >= 2 && !mbar_wait(&sm.inv_free[par], ((kk >> 1) - 1) & 1, err, 41, abort_ptr)) return false;
      if (pseg == 0) {
        // denominator of row pr: intra-chunk part + beta_r n.q_r (both halves of d_qk with a pair)
        float nqf = sm.nq[par][pr];
        if (PAIR) nqf += sm.nqx[par][pi];
        const float dn = den + g.beta[pr] * nqf;
        sm.inv[par][pr] = 1.f / fmaxf(fabsf(dn), g.floor_[pr]);
      }
      fence_proxy_async_smem();
      mbar_arrive(&sm.sofree);
      mbar_arrive(&sm.pready);
      mbar_arrive(&sm.inv_ready[par]);
      if (PAIR) {
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_remote(mapa_shared(smem_u32(&sm.sx_free[par]), prt));
          mbar_arrive_remote(mapa_shared(smem_u32(&sm.nqx_free[par]), prt));
        }
      }
      return true;
    };

    float sig_last = 0.f;
    bool ok = true;
    for (int k = 0; k < NC; ++k) {
      if (!mbar_wait(&sm.g_full[k & 3], (k >> 2) & 1, err, 40, abort_ptr)) { ok = false; break; }
      // U_{k-1} and X_{k-1} (which reads C16) are done
      if (k >= 1 && !mbar_wait(&sm.bar_X, (k - 1) & 1, err, 32, abort_ptr)) { ok = false; break; }
      tc_fence_after();
      const Gate &g = sm.g[k & 3];
      const float fr_c = g.fr_c, fr_w = g.fr_w;
      const bool lazy = g.lazy != 0;
      sig_last = g.sig_next;
      const uint64_t frc2 = f2pack(fr_c, fr_c), frw2 = f2pack(fr_w, fr_w);
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
              hv[i] = f2_to_h2(f2mul(f2pack(__uint_as_float(ua[2 * i]), __uint_as_float(ua[2 * i + 1])), frc2));
            tmem_st16(tm + lane_base + kColC16 + c / 2, hv);
          }
          tmem_wait_ld();
          if (c + 64 < DH) tmem_ld32(tm + lane_base + c + 64, ua);
          {
            uint32_t hv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              hv[i] = f2_to_h2(f2mul(f2pack(__uint_as_float(ub[2 * i]), __uint_as_float(ub[2 * i + 1])), frc2));
            tmem_st16(tm + lane_base + kColC16 + c / 2 + 16, hv);
          }
          if (c + 64 < DH) tmem_wait_ld();
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
          for (int i = 0; i < 16; ++i) {
            const uint64_t x = f2pack(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1]));
            hv[i] = f2_to_h2(f2mul(x, frc2));
            float lo, hi;
            f2unpack(f2mul(x, frw2), lo, hi);
            u[2 * i] = __float_as_uint(lo);
            u[2 * i + 1] = __float_as_uint(hi);
          }
          tmem_st16(tm + lane_base + kColC16 + c / 2, hv);
          tmem_st16(tm + lane_base + c, *reinterpret_cast<const uint32_t(*)[16]>(&u[0]));
          tmem_st16(tm + lane_base + c + 16, *reinterpret_cast<const uint32_t(*)[16]>(&u[16]));
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&sm.cready);
      if (!p_form(k)) { ok = false; break; }
    }
    if (ok && atile == 0 && rank == 0 && t == 0) m_last[p] = sm.m_fin;
    // final state C_last = exp(sigma) T, transposed through shared memory for coalesced stores;
    // once the last X is done (and so the last U), every q/k stage is free for the staging
    if (ok && NC > 0 && !mbar_wait(&sm.bar_X, (NC - 1) & 1, err, 33, abort_ptr)) ok = false;
    if (ok) {
      tc_fence_after();
      const float fr = __expf(sig_last);
      // 32 columns at a time through two swizzled staging tiles [128 rows x 128 bytes]
#pragma unroll 1
      for (int c = 0, slab = 0; c < DH; c += 32, ++slab) {
        uint8_t *tile = base + (slab & 1) * 16384;
        if (slab >= 2) {
          if (t == 0) bulk_wait_read<1>();  // the store that used this tile has read it
          if (!group_sync(&sm.grp[0], gph, err, 34, abort_ptr)) { ok = false; break; }
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
        if (!group_sync(&sm.grp[0], gph, err, 35, abort_ptr)) { ok = false; break; }
        if (t == 0) {
          tma_store_2d(&mapC, c0 + c, p * DV + a0, tile);
          bulk_commit();
        }
      }
      if (t == 0) bulk_wait_all();
    }
    if (!ok) set_abort(sm);
  } else if (warp < 12) {
    // ------------------------------------------------------------------ warpgroup 2: P V, epilogue
    const int t = threadIdx.x - 256;  // tensor-memory lane = d_v row within the tile
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t id_P = idesc_f16(kTile, NR, 0, 1, 0);
    const uint64_t dp_own = smem_desc(smem_u32(sP) + r_lo * 128, 16, 1024, kSwizzle128B);

    // H^T of chunk kk: read it (and free the accumulator at once), exchange the partner's columns,
    // scale by 1/den and store h
    auto epilogue = [&](int kk) -> bool {
      const int par = kk & 1;
      const size_t tok0 = (size_t)p * S + (size_t)kk * kL;
      if (t == 0) {
        // H^T[own rows] += V^T P^T once P is formed (so v of the chunk is in fp16 too) and X_kk
        // (which wrote H) is done; this thread's commit then covers P V alone
        if (!mbar_wait(&sm.pready, kk & 1, err, 17, abort_ptr) || !mbar_wait(&sm.bar_X, kk & 1, err, 9, abort_ptr)) {
          set_abort(sm);
          return false;
        }
        tc_fence_after();
        const uint64_t dv = smem_desc(smem_u32(STV(kk & 1)), 8192, 1024, kSwizzle128B);
#pragma unroll 1
        for (int j = 0; j < kL / 16; ++j)
          mma_f16_ss(tm + kColH + r_lo, dv + (uint64_t)(j * 2048 >> 4), dp_own + (uint64_t)(j * 32 >> 4), id_P, 1);
        mma_commit(&sm.bar_H);
        mma_commit(&sm.v_empty[kk & 1]);
      }
      if (!mbar_wait(&sm.bar_H, kk & 1, err, 26, abort_ptr)) return false;
      tc_fence_after();
      uint32_t u[2][32];
      tmem_ld32(tm + lane_base + kColH + 32 * rank, u[0]);       // rows finalised here
      tmem_ld32(tm + lane_base + kColH + 32 * (PAIR ? prt : 1), u[1]);  // the partner's / the rest
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&sm.hfree);
      if (PAIR) {
        if (kk >= 1 && !mbar_wait_cluster(&sm.hx_free, (kk - 1) & 1, err, 27, abort_ptr)) return false;
        const uint32_t rbar = mapa_shared(smem_u32(&sm.hx_full), prt);
        const uint32_t dst = mapa_shared(smem_u32(HX + t * 32), prt);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          st_async_v4(dst + ((i ^ (t & 7)) << 4), __uint_as_float(u[1][4 * i]), __uint_as_float(u[1][4 * i + 1]),
                      __uint_as_float(u[1][4 * i + 2]), __uint_as_float(u[1][4 * i + 3]), rbar);
        if (t == 0) mbar_arrive_expect_tx(&sm.hx_full, 128 * 32 * 4);
        if (!mbar_wait_cluster(&sm.hx_full, kk & 1, err, 28, abort_ptr)) return false;
        const float *src = HX + t * 32;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 v4 = *reinterpret_cast<const float4 *>(src + 4 * (i ^ (t & 7)));
          u[0][4 * i] = __float_as_uint(__uint_as_float(u[0][4 * i]) + v4.x);
          u[0][4 * i + 1] = __float_as_uint(__uint_as_float(u[0][4 * i + 1]) + v4.y);
          u[0][4 * i + 2] = __float_as_uint(__uint_as_float(u[0][4 * i + 2]) + v4.z);
          u[0][4 * i + 3] = __float_as_uint(__uint_as_float(u[0][4 * i + 3]) + v4.w);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&sm.hx_free), prt));
      }
      // 1/den of the rows of chunk kk (warpgroup 1)
      if (!mbar_wait(&sm.inv_ready[par], (kk >> 1) & 1, err, 29, abort_ptr)) return false;
      TO *hp = h + (tok0 + r_lo) * DV + a0 + t;
      const float *iv = sm.inv[par] + r_lo;
#pragma unroll
      for (int i = 0; i < NR; i += 4) {
        const float4 i4 = *reinterpret_cast<const float4 *>(iv + i);
        const uint32_t *src = u[i >> 5] + (i & 31);
        hp[(size_t)i * DV] = from_f32<TO>(__uint_as_float(src[0]) * i4.x);
        hp[(size_t)(i + 1) * DV] = from_f32<TO>(__uint_as_float(src[1]) * i4.y);
        hp[(size_t)(i + 2) * DV] = from_f32<TO>(__uint_as_float(src[2]) * i4.z);
        hp[(size_t)(i + 3) * DV] = from_f32<TO>(__uint_as_float(src[3]) * i4.w);
      }
      mbar_arrive(&sm.inv_free[par]);
      return true;
    };

    bool ok = true;
    for (int k = 0; ok && k < NC; ++k) ok = epilogue(k);
    if (!ok) set_abort(sm);
    if (t == 0) {
      mma_commit(&sm.fin);  // completes once every MMA issued by warps 0, 1 and this thread is done
      mbar_wait(&sm.fin, 0, err, 7);
    }
  } else if (warp < 16) {
    // ------------------------------------------------------------------ warpgroup 3: beta q, n . q, v
    const int t = threadIdx.x - 384;
    constexpr int CPR = DH / 8;  // 16-byte chunks per row
    // row layout: two threads per row, each half of every block's chunks
    const int qr = t >> 1, qh = t & 1;
    // v of chunk kk: bf16 -> fp16 (exact), in place
    auto v_pass = [&](int kk) -> bool {
      const int s = kk & 1;
      if (!mbar_wait(&sm.v_full[s], (kk >> 1) & 1, err, 55, abort_ptr)) return false;
      uint4 *vp = reinterpret_cast<uint4 *>(STV(s));
      uint4 raw[8];
#pragma unroll
      for (int b = 0; b < 8; ++b) raw[b] = vp[t + 128 * b];
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        uint4 o4;
        o4.x = bf2_to_h2(raw[b].x);
        o4.y = bf2_to_h2(raw[b].y);
        o4.z = bf2_to_h2(raw[b].z);
        o4.w = bf2_to_h2(raw[b].w);
        vp[t + 128 * b] = o4;
      }
      fence_proxy_async_smem();
      mbar_arrive(&sm.vready[s]);
      return true;
    };

    bool ok = NC == 0 || v_pass(0);
    for (int k = 0; ok && k < NC; ++k) {
      const int s = k & 1, par = k & 1;
      if (!mbar_wait(&sm.g_full[k & 3], (k >> 2) & 1, err, 51, abort_ptr) ||
          !mbar_wait(&sm.nready[s], (k >> 1) & 1, err, 53, abort_ptr) ||
          !mbar_wait(&sm.bar_S[s], (k >> 1) & 1, err, 56, abort_ptr)) {  // S_k has read raw q
        ok = false;
        break;
      }
      const Gate &g = sm.g[k & 3];
      uint8_t *const qb = STQ(s);
      const float *nk = sm.n[k & 1];
      const float bq = g.beta[qr];
      const uint64_t bq2 = f2pack(bq, bq);
      uint64_t part2 = 0;
      // d_qk block by block (64 columns, 8 chunks of 16 bytes per row), so that X can start on
      // block b as soon as it is converted; each thread takes four chunks of its row per block
#pragma unroll 1
      for (int blk = 0; blk < CPR / 8; ++blk) {
        uint4 raw[4], na[4], nb[4];
        int off[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int ch = blk * 8 + qh * 4 + b;  // chunk of the row
          off[b] = blk * 8192 + qr * 128 + (((ch & 7) ^ (qr & 7)) << 4);
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
        fence_proxy_async_smem();
        mbar_arrive(&sm.xblk[s][blk]);
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
      fence_proxy_async_smem();
      mbar_arrive(&sm.xready[s]);
      // v of the next chunk (U of that chunk waits for it)
      if (k + 1 < NC && !v_pass(k + 1)) ok = false;
    }
    if (!ok) set_abort(sm);
  } else {
    // ------------------------------------------------------------------ warpgroup 4: w k, S, n
    const int t = threadIdx.x - 512;
    const int q4 = warp & 3;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const int r_s = 16 * q4 + (lane & 15);  // S row held by this lane (M = 64 layout, lanes < 16)
    const bool own_rows = !PAIR || ((q4 >> 1) == rank);
    constexpr int KCPR = DH / 8;     // w k pass: 16-byte chunks per row of k
    constexpr int KRG = 128 / KCPR;  // rows handled at once (column layout)
    const int kcc = t % KCPR, krg = t / KCPR;
    const int kcolb = (kcc >> 3) * 8192, kc8 = kcc & 7;
    uint32_t gph = 0;
    float al_k = 1.f;  // chunk decay of the chunk being processed
    // n entering chunk k lives in n[k & 1]
    for (int c = t; c < DH; c += 128) sm.n[0][c] = n_init ? n_init[(size_t)p * D + c0 + c] : 0.f;
    mbar_arrive(&sm.nready[0]);
    bool ok = true;
    for (int k = 0; ok && k < NC; ++k) {
      const int s = k & 1, par = k & 1;
      if (!mbar_wait(&sm.g_full[k & 3], (k >> 2) & 1, err, 21, abort_ptr) ||
          !mbar_wait(&sm.bar_S[s], (k >> 1) & 1, err, 22, abort_ptr)) {
        ok = false;
        break;
      }
      // w_j k_j (frame of T) in fp16, in place over the raw k of the stage, and the n-update
      // partial sums sum_j w_j k_j / sqrt(d) per row group (column layout)
      {
        const Gate &g = sm.g[k & 3];
        al_k = g.alpha;  // read now: the slot is rewritten once this chunk's U and P V are done
        uint8_t *const kb = STK(s);
        uint64_t acc[4] = {0, 0, 0, 0};
        // token block by token block (16 rows), so that U can start on block b as soon as it is
        // converted; each thread takes RPB rows of its column chunk per block
        constexpr int RPB = 16 / KRG;
#pragma unroll 1
        for (int rb = 0; rb < 4; ++rb) {
          uint4 raw[RPB];
          int off[RPB];
          float wt[RPB], wk[RPB];
#pragma unroll
          for (int b = 0; b < RPB; ++b) {
            const int j = 16 * rb + krg + KRG * b;
            off[b] = kcolb + j * 128 + ((kc8 ^ (j & 7)) << 4);
            raw[b] = *reinterpret_cast<const uint4 *>(kb + off[b]);
            wt[b] = g.wt[j];
            wk[b] = g.wk[j];
          }
          uint4 o4[RPB];
#pragma unroll
          for (int b = 0; b < RPB; ++b) {
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
          for (int b = 0; b < RPB; ++b) *reinterpret_cast<uint4 *>(kb + off[b]) = o4[b];
          fence_proxy_async_smem();
          mbar_arrive(&sm.kblk[s][rb]);
        }
        float *np = &sm.npart[krg * DH + kcc * 8];
#pragma unroll
        for (int e = 0; e < 4; ++e) *reinterpret_cast<uint64_t *>(np + 2 * e) = acc[e];
      }
      // S rows of chunk k: own rows -> SO, the partner's rows -> partner's SX
      {
        tc_fence_after();
        uint32_t u[2][32];
        tmem_ld32(tm + lane_base + kColS, u[0]);
        tmem_ld32(tm + lane_base + kColS + 32, u[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&sm.sfree);
        // SO is rewritten (and soready re-armed) only after P of the previous chunk was formed
        if (k >= 1 && !mbar_wait(&sm.sofree, (k - 1) & 1, err, 38, abort_ptr)) { ok = false; break; }
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
          if (k >= 2 && !mbar_wait_cluster(&sm.sx_free[par], ((k >> 1) - 1) & 1, err, 37, abort_ptr)) {
            ok = false;
            break;
          }
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
        mbar_arrive(&sm.soready);
      }
      // n entering chunk k+1 = alpha_k n_k + the partial sums; it overwrites n[(k + 1) & 1], which
      // the q pass of chunk k-1 read (done once xready of chunk k-1 has completed)
      if (!group_sync(&sm.grp[2], gph, err, 58, abort_ptr) ||
          (k >= 1 && !mbar_wait(&sm.xready[(k - 1) & 1], ((k - 1) >> 1) & 1, err, 59, abort_ptr))) {
        ok = false;
        break;
      }
      {
        for (int c = t; c < DH; c += 128) {
          float a = al_k * sm.n[k & 1][c];
#pragma unroll
          for (int gi = 0; gi < KRG; ++gi) a += sm.npart[gi * DH + c];
          sm.n[(k + 1) & 1][c] = a;
        }
      }
      mbar_arrive(&sm.nready[(k + 1) & 1]);
      // every thread has read the partial sums before the next chunk's k pass rewrites them
      if (!group_sync(&sm.grp[2], gph, err, 39, abort_ptr)) { ok = false; break; }
    }
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
#undef STQ
#undef STK
#undef STV
}

// Dynamic shared memory: two (q, k) stages, two v stages, P, this CTA's partial S rows, the pair
// exchange buffers and alignment slack; never less than 120 KB, so that one CTA (which allocates
// all 512 tensor-memory columns) runs per SM.
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

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      n > 0)
    return n;
  cudaGetLastError();
  return 148;
}

bool fwd_tc_supported(int S, int L, int D, int DV, bool bf16) {
  return bf16 && L == kL && (D == 64 || D == 128 || D == 256 || D == 512) && DV % kTile == 0 && S > 0 &&
         S % kL == 0;
}

bool fwd_tc_pair(int P, int D, int DV) {
  // d_qk = 512 only fits split over a pair; smaller heads split when that fills more of the SMs.
  return D == 512 || (D >= 128 && (long long)P * (DV / kTile) < sm_count());
}

int fwd_tc_segments(int P, int S, int D, int DV) {
  // Sequence segments that run in parallel: the largest power of two G with G times the CTAs of
  // the plain launch still within the SMs, segments of at least four chunks, S divisible by G
  // chunks.  Long sequences over few heads (B * NH small) are what this is for.
  const long long ctas = (long long)P * (DV / kTile) * (fwd_tc_pair(P, D, DV) ? 2 : 1);
  const int sms = sm_count();
  int G = 1;
  while (ctas * (2 * G) <= sms && S % (kL * 2 * G) == 0 && S / (2 * G) >= 4 * kL) G *= 2;
  return G;
}

cudaError_t launch_fwd_tc(const void *q, const void *k, const void *v, bool out_bf16, const float *gb,
                          const float *gx, const float *gu, const float *cm, const float *ig, const float *fg,
                          const float *m_init, int P, int S, int D, int DV, const float *C_init,
                          const float *n_init, void *h, float *C_last, float *n_last, float *m_last, int *err,
                          cudaStream_t stream, bool exp_fg, int pair_heads) {
  // the CTA-pair decision is that of the caller's head count (the segmented passes keep it)
  const bool pair = fwd_tc_pair(pair_heads > 0 ? pair_heads : P, D, DV);
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
