// fused_tc.cu -- tensor-core chunkwise forward: inter-chunk recurrence and intra-chunk output
// in one persistent pass per (head, 128-row d_v tile), the state resident in tensor memory.
//
// Page "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural Networks"
// (llms.blog): section 3 "The Parallel Dual Form" (H = ((Q K^T) o S) V inside a chunk, the
// unrolled C_T across chunks), section 3 "Associative Matrix Cell State" (C, n updates, the
// retrieval h = C q / max(|n^T q|, .), k scaled by 1/sqrt(d)), section 2 (max stabiliser).
// Per chunk k with entering state (C, n, m_in) and the gate kernel's b, x, u:
//   S = Q K^T / sqrt(d)                              (tensor cores, bf16 inputs, fp32 accumulate)
//   P_rj = S_rj exp(x_j - max(m_in, u_r)), j <= r   (fp32), den_r = sum_j P_rj + beta_r n.q_r
//   H^T = V^T P^T + C (beta q)^T                     (tensor cores, fp16 operands)
//   h_r = H_r / max(|den_r|, exp(-m_r))
//   C <- alpha C + V^T diag(w) K / sqrt(d)           (tensor cores into the resident state)
//   n <- alpha n + K^T w / sqrt(d)                   (CUDA cores, fp32)
//
// The state tile T (128 rows of d_v x d_qk, fp32) lives in TMEM for the whole sequence and is
// the accumulator of the update MMA.  It is kept in a lazily rescaled frame C = exp(sigma) T:
// the decay alpha is folded into sigma (and into the scale of the next update's operand), and
// T is multiplied back to sigma = 0 only when exp(-sigma) would exceed 2^8.  Its fp16 copy
// (written TMEM -> registers -> TMEM each chunk) is the A operand of the C q term.
//
// Roles (384 threads):  warp 0 lane 0 issues TMA loads of the bf16 q/k chunks (two stages);
// warp 1 lane 0 allocates tensor memory and issues every MMA; warpgroup 1 (warps 4-7) loads
// v into tensor memory, forms P and writes h; warpgroup 2 (warps 8-11) copies the state,
// rescales it, prepares the scaled fp16 q and k operands and keeps n.  Hand-offs use
// mbarriers; every wait is bounded and reports through an error word.
//
// Operand precision: q, k, v arrive as bf16 and convert to fp16 exactly; the computed
// operands (P, C, w k) are rounded to fp16 (11 significant bits); all sums are fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.cuh"
#include "sm100.cuh"
#include "tmap.cuh"

namespace mlstm {
namespace {

using namespace sm100;

constexpr int kL = 64;         // chunk length handled by this kernel
constexpr int kTile = 128;     // d_v rows per CTA (MMA M)
constexpr int kThreads = 384;
constexpr float kRescaleLog = 5.545177444479562f;  // ln(2^8): largest lazy frame factor

// tensor-memory column map (512 columns allocated)
constexpr uint32_t kColState = 0;    // [0, D)        fp32 state T
constexpr uint32_t kColC16 = 256;    // [256, 256+D/2) fp16 copy of T (A operand)
constexpr uint32_t kColSH = 384;     // [384, 448)    S (M=64 layout), then H^T (M=128, N=64)
constexpr uint32_t kColV16 = 448;    // [448, 480)    fp16 V^T (A operand, K = 64 tokens)

struct Smem {
  // barriers
  uint64_t full[2], empty[2];
  uint64_t bar_S, bar_H, bar_U, bar_ready, bar_hfree;
  uint32_t tmem_base;
  int abort_flag;
  // per-chunk scalars, double-buffered by chunk parity
  float beta[2][kL];     // exp(m_in - max(m_in, u_r)) * exp(sigma_k)   (scale of q in the C q term)
  float mr[2][kL];       // max(m_in, u_r)
  float floor_[2][kL];   // exp(-m_r)
  float den_x[2][kL];    // beta_r * n . q_r   (true beta, not the frame-scaled one)
  float den_i[2][kL];    // sum_j P_rj
  float xg[kL];          // x_j of the chunk
  float wk[kL];          // w_j * exp(-sigma_{k+1}) / sqrt(d)   (scale of k in the update)
  float w_true[kL];      // w_j / sqrt(d)                          (for n)
  float n[256];          // normaliser of the entering state (fp32)
  float nq_part[2][kL];  // partial n . q sums (two threads per row)
};

__device__ __forceinline__ bool aborted(const Smem &sm) { return *(volatile const int *)&sm.abort_flag != 0; }
__device__ __forceinline__ void set_abort(Smem &sm) { *(volatile int *)&sm.abort_flag = 1; }

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

template <typename TO>
__global__ void __launch_bounds__(kThreads, 1) fused_tc_kernel(
    const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
    const __nv_bfloat16 *__restrict__ vin, const float *__restrict__ gb, const float *__restrict__ gx,
    const float *__restrict__ gu, const float *__restrict__ cm, int S, int D, int DV,
    const float *__restrict__ C_init, const float *__restrict__ n_init, TO *__restrict__ h,
    float *__restrict__ C_last, float *__restrict__ n_last, float *__restrict__ m_last, int *__restrict__ err) {
  extern __shared__ uint8_t smem_dyn[];
  __shared__ Smem sm;
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const int blk = D * kL * 2;             // bytes of one [64 x D] 2-byte matrix
  // stage s holds q at base + 2 s blk and k at base + (2 s + 1) blk
#define SQ(s_) (base + (2 * (s_)) * blk)
#define SK(s_) (base + (2 * (s_) + 1) * blk)
  uint8_t *sQb = base + 4 * blk;          // fp16 beta-scaled q  (K-major, B of the C q term)
  uint8_t *sKw = base + 5 * blk;          // fp16 w-scaled k     (MN-major, B of the update)
  uint8_t *sP = base + 6 * blk;           // fp16 P [64 x 64]    (K-major, B of V^T P^T)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a0 = blockIdx.x * kTile, p = blockIdx.y;
  const int NC = S / kL;
  const float scale = rsqrtf((float)D);
  const int nkb = D / 64;  // 64-column blocks of q / k

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) { mbar_init(&sm.full[i], 1); mbar_init(&sm.empty[i], 1); }
    mbar_init(&sm.bar_S, 1);
    mbar_init(&sm.bar_H, 1);
    mbar_init(&sm.bar_U, 1);
    mbar_init(&sm.bar_ready, 256);
    mbar_init(&sm.bar_hfree, 128);
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
  const uint32_t tm = sm.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&mapQ);
      prefetch_tensormap(&mapK);
      for (int k = 0; k < NC; ++k) {
        const int s = k & 1;
        if (k >= 2 && !mbar_wait(&sm.empty[s], ((k >> 1) - 1) & 1, err, 11)) { set_abort(sm); break; }
        if (aborted(sm)) break;
        mbar_arrive_expect_tx(&sm.full[s], (uint32_t)(2 * blk));
        const int row = p * S + k * kL;
        for (int kb = 0; kb < nkb; ++kb) {
          tma_load_2d(SQ(s) + kb * kL * 128, &mapQ, kb * 64, row, &sm.full[s]);
          tma_load_2d(SK(s) + kb * kL * 128, &mapK, kb * 64, row, &sm.full[s]);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_S = idesc_f16(64, kL, /*bf16*/ 1, 0, 0);
      const uint32_t id_H = idesc_f16(kTile, kL, 0, 0, 0);
      const uint32_t id_U = idesc_f16(kTile, D, 0, 0, /*b MN-major*/ 1);
      for (int k = 0; k < NC; ++k) {
        const int s = k & 1;
        if (!mbar_wait(&sm.full[s], (k >> 1) & 1, err, 12)) { set_abort(sm); break; }
        // S and H share tensor-memory columns: S_k waits for the h epilogue of chunk k-1
        if (k >= 1 && !mbar_wait(&sm.bar_hfree, (k - 1) & 1, err, 13)) { set_abort(sm); break; }
        tc_fence_after();
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kL * 128 + (kk & 3) * 32;
          mma_f16_ss(tm + kColSH, smem_desc(smem_u32(SQ(s)) + off, 16, 1024, kSwizzle128B),
                     smem_desc(smem_u32(SK(s)) + off, 16, 1024, kSwizzle128B), id_S, kk > 0);
        }
        mma_commit(&sm.bar_S);
        if (!mbar_wait(&sm.bar_ready, k & 1, err, 14)) { set_abort(sm); break; }
        tc_fence_after();
        // H^T[a, r] = V^T P^T  (+)  C16 (beta q)^T
        for (int kk = 0; kk < kL / 16; ++kk) {
          const uint64_t bd = smem_desc(smem_u32(sP) + kk * 32, 16, 1024, kSwizzle128B);
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tm + kColSH),
              "r"(tm + kColV16 + kk * 8), "l"(bd), "r"(id_H), "r"(kk > 0 ? 1u : 0u)
              : "memory");
        }
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kL * 128 + (kk & 3) * 32;
          const uint64_t bd = smem_desc(smem_u32(sQb) + off, 16, 1024, kSwizzle128B);
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tm + kColSH),
              "r"(tm + kColC16 + kk * 8), "l"(bd), "r"(id_H), "r"(1u)
              : "memory");
        }
        mma_commit(&sm.bar_H);
        // T += V^T (w k)   (B = w k, MN-major: rows are tokens, 64-column blocks LBO apart)
        for (int kk = 0; kk < kL / 16; ++kk) {
          const uint64_t bd = smem_desc(smem_u32(sKw) + kk * 2048, kL * 128, 1024, kSwizzle128B);
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tm + kColState),
              "r"(tm + kColV16 + kk * 8), "l"(bd), "r"(id_U), "r"(1u)
              : "memory");
        }
        mma_commit(&sm.bar_U);
        mma_commit(&sm.empty[s]);
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ warpgroup 1: V, P, h
    const int t = threadIdx.x - 128;              // 0..127 == tensor-memory lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int q4 = warp & 3;
    for (int k = 0; k < NC; ++k) {
      const int par = k & 1;
      const size_t tok0 = (size_t)p * S + (size_t)k * kL;
      // V^T of this chunk into tensor memory (row a = lane t), after update k-1 read the old one
      float vcol[kL];
#pragma unroll
      for (int j = 0; j < kL; ++j) vcol[j] = __bfloat162float(vin[(tok0 + j) * DV + a0 + t]);
      if (k >= 1 && !mbar_wait(&sm.bar_U, (k - 1) & 1, err, 21)) { set_abort(sm); }
      if (aborted(sm)) break;
      tc_fence_after();
#pragma unroll
      for (int j0 = 0; j0 < kL / 2; j0 += 16) {
        uint32_t r[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = pack_half2(vcol[2 * (j0 + i)], vcol[2 * (j0 + i) + 1]);
        tmem_st16(tm + lane_base + kColV16 + j0, r);
      }
      tmem_wait_st();
      // P from S (M=64 layout: row r = 16 q4 + l in lanes 32 q4 + l, l < 16)
      named_barrier_sync(3, 256);  // chunk scalars (mr, x) written by warpgroup 2
      if (!mbar_wait(&sm.bar_S, par, err, 22)) { set_abort(sm); break; }
      tc_fence_after();
      {
        const int r = 16 * q4 + (lane & 15);
        float srow[kL];
#pragma unroll
        for (int c0 = 0; c0 < kL; c0 += 16) {
          uint32_t u[16];
          tmem_ld16(tm + lane_base + kColSH + c0, u);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) srow[c0 + i] = __uint_as_float(u[i]);
        }
        if (lane < 16) {
          const float mrr = sm.mr[par][r];
          float den = 0.f;
          uint8_t *prow = sP + r * 128;
#pragma unroll
          for (int c8 = 0; c8 < kL / 8; ++c8) {
            float pv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int j = c8 * 8 + i;
              pv[i] = (j <= r) ? srow[j] * scale * __expf(sm.xg[j] - mrr) : 0.f;
              den += pv[i];
            }
            uint4 w4;
            w4.x = pack_half2(pv[0], pv[1]);
            w4.y = pack_half2(pv[2], pv[3]);
            w4.z = pack_half2(pv[4], pv[5]);
            w4.w = pack_half2(pv[6], pv[7]);
            *reinterpret_cast<uint4 *>(prow + ((c8 ^ (r & 7)) << 4)) = w4;
          }
          sm.den_i[par][r] = den;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&sm.bar_ready);
      // h epilogue: H^T[a = t][r]
      if (!mbar_wait(&sm.bar_H, par, err, 23)) { set_abort(sm); break; }
      tc_fence_after();
      named_barrier_sync(1, 256);  // den_x of this chunk written by warpgroup 2
#pragma unroll
      for (int c0 = 0; c0 < kL; c0 += 16) {
        uint32_t u[16];
        tmem_ld16(tm + lane_base + kColSH + c0, u);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = c0 + i;
          const float den = sm.den_i[par][r] + sm.den_x[par][r];
          const float out = __uint_as_float(u[i]) / fmaxf(fabsf(den), sm.floor_[par][r]);
          h[(tok0 + r) * DV + a0 + t] = from_f32<TO>(out);
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.bar_hfree);
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ warpgroup 2: state, q/k, n
    const int t = threadIdx.x - 256;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const bool n_owner = true;
    float sigma = 0.f;  // C = exp(sigma) T
    // initial state into tensor memory
    for (int c = t; c < D; c += 128) sm.n[c] = n_init ? n_init[(size_t)p * D + c] : 0.f;
    for (int c0 = 0; c0 < D; c0 += 16) {
      uint32_t r[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        r[i] = __float_as_uint(C_init ? C_init[((size_t)p * DV + a0 + t) * D + c0 + i] : 0.f);
      tmem_st16(tm + lane_base + kColState + c0, r);
    }
    tmem_wait_st();
    named_barrier_sync(2, 128);
    (void)n_owner;
    for (int k = 0; k < NC; ++k) {
      const int par = k & 1, s = k & 1;
      const size_t tok0 = (size_t)p * S + (size_t)k * kL;
      const float m_in = cm[(size_t)p * (NC + 1) + k], m_out = cm[(size_t)p * (NC + 1) + k + 1];
      const float bl = gb[tok0 + kL - 1];
      const float log_alpha = bl + m_in - m_out;  // <= 0
      // scalars of this chunk
      if (t < kL) {
        const float u = gu[tok0 + t], x = gx[tok0 + t];
        const float mrr = fmaxf(m_in, u);
        sm.mr[par][t] = mrr;
        sm.floor_[par][t] = __expf(-(gb[tok0 + t] + mrr));
        sm.xg[t] = x;
        sm.w_true[t] = __expf(bl + x - m_out) * scale;
      }
      // previous update must be complete before the state is read or q/k buffers reused
      if (k >= 1 && !mbar_wait(&sm.bar_U, (k - 1) & 1, err, 31)) { set_abort(sm); }
      if (aborted(sm)) break;
      tc_fence_after();
      // Frame of the resident state: C = exp(sigma) T.  Lazy: keep T, fold alpha into the frame
      // (sigma_next = sigma + log alpha) as long as exp(-sigma_next) <= 2^8.  Otherwise eager:
      // write back T exp(sigma) alpha (the decayed state) and restart the frame at 0.
      const bool lazy = -(sigma + log_alpha) <= kRescaleLog;
      const float sig_k = lazy ? sigma : 0.f;                  // frame of the fp16 copy of C^(k)
      const float fr_c = lazy ? 1.f : __expf(sigma);           // T -> fp16 copy
      const float fr_w = __expf(sigma + log_alpha);            // eager write-back factor
      const float sig_next = lazy ? sigma + log_alpha : 0.f;   // frame after the update
      if (t < kL) {
        const float beta = __expf(m_in - fmaxf(m_in, gu[tok0 + t]));
        sm.beta[par][t] = beta * __expf(sig_k);
        sm.wk[t] = __expf(bl + gx[tok0 + t] - m_out - sig_next) * scale;
        sm.den_x[par][t] = beta;  // multiplied by n.q below
      }
      // fp16 copy of the state into the A-operand columns (and the eager write-back)
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t u0[16], u1[16];
        tmem_ld16(tm + lane_base + kColState + c0, u0);
        tmem_ld16(tm + lane_base + kColState + c0 + 16, u1);
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
          tmem_st16(tm + lane_base + kColState + c0, u0);
          tmem_st16(tm + lane_base + kColState + c0 + 16, u1);
        }
        tmem_st16(tm + lane_base + kColC16 + c0 / 2, hv);
      }
      tmem_wait_st();
      sigma = sig_next;
      named_barrier_sync(2, 128);    // chunk scalars visible inside warpgroup 2
      named_barrier_arrive(3, 256);  // ... and to warpgroup 1 (P needs mr and x)
      // q and k of this chunk in shared memory
      if (!mbar_wait(&sm.full[s], (k >> 1) & 1, err, 32)) { set_abort(sm); break; }
      // scaled fp16 copies (same swizzled positions: a 16-byte chunk holds 8 elements of one row)
      const int nchunks = blk / 16;
      for (int i = t; i < nchunks; i += 128) {
        const int row = (i >> 3) & (kL - 1);
        const uint4 q4v = reinterpret_cast<const uint4 *>(SQ(s))[i];
        const uint4 k4v = reinterpret_cast<const uint4 *>(SK(s))[i];
        const float bq = sm.beta[par][row], wkr = sm.wk[row];
        const __nv_bfloat162 *qb = reinterpret_cast<const __nv_bfloat162 *>(&q4v);
        const __nv_bfloat162 *kb = reinterpret_cast<const __nv_bfloat162 *>(&k4v);
        uint4 qo, ko;
        uint32_t *qo32 = reinterpret_cast<uint32_t *>(&qo), *ko32 = reinterpret_cast<uint32_t *>(&ko);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 qf = __bfloat1622float2(qb[e]);
          const float2 kf = __bfloat1622float2(kb[e]);
          qo32[e] = pack_half2(qf.x * bq, qf.y * bq);
          ko32[e] = pack_half2(kf.x * wkr, kf.y * wkr);
        }
        reinterpret_cast<uint4 *>(sQb)[i] = qo;
        reinterpret_cast<uint4 *>(sKw)[i] = ko;
      }
      // n . q_r with the entering n (two threads per row, halves of d_qk)
      {
        const int r = t >> 1, half = t & 1;
        float acc = 0.f;
        for (int c8 = half * (D / 16); c8 < (half + 1) * (D / 16); ++c8) {
          const int kb = c8 >> 3, cc = c8 & 7;
          const uint4 q4v = *reinterpret_cast<const uint4 *>(SQ(s) + kb * kL * 128 + r * 128 + ((cc ^ (r & 7)) << 4));
          const __nv_bfloat162 *qb = reinterpret_cast<const __nv_bfloat162 *>(&q4v);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 qf = __bfloat1622float2(qb[e]);
            acc = fmaf(qf.x, sm.n[c8 * 8 + 2 * e], acc);
            acc = fmaf(qf.y, sm.n[c8 * 8 + 2 * e + 1], acc);
          }
        }
        sm.nq_part[half][r] = acc;
      }
      named_barrier_sync(2, 128);
      if (t < kL) sm.den_x[par][t] *= sm.nq_part[0][t] + sm.nq_part[1][t];
      // n <- alpha n + sum_j w_j k_j / sqrt(d)
      {
        const float alpha = __expf(log_alpha);
        for (int c = t; c < D; c += 128) {
          const int kb = c >> 6, cc = (c & 63) >> 3, e = c & 7;
          float acc = 0.f;
          for (int j = 0; j < kL; ++j) {
            const __nv_bfloat16 kv =
                *reinterpret_cast<const __nv_bfloat16 *>(SK(s) + kb * kL * 128 + j * 128 + ((cc ^ (j & 7)) << 4) + e * 2);
            acc = fmaf(sm.w_true[j], __bfloat162float(kv), acc);
          }
          sm.n[c] = alpha * sm.n[c] + acc;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&sm.bar_ready);
      named_barrier_sync(1, 256);  // den_x visible to warpgroup 1's h epilogue
    }
    // final state: C_last = exp(sigma) T
    if (!aborted(sm) && NC > 0 && !mbar_wait(&sm.bar_U, (NC - 1) & 1, err, 33)) set_abort(sm);
    if (!aborted(sm)) {
      tc_fence_after();
      const float fr = __expf(sigma);
      for (int c0 = 0; c0 < D; c0 += 16) {
        uint32_t u[16];
        tmem_ld16(tm + lane_base + kColState + c0, u);
        tmem_wait_ld();
        float *dst = C_last + ((size_t)p * DV + a0 + t) * D + c0;
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          *reinterpret_cast<float4 *>(dst + i) =
              make_float4(__uint_as_float(u[i]) * fr, __uint_as_float(u[i + 1]) * fr,
                          __uint_as_float(u[i + 2]) * fr, __uint_as_float(u[i + 3]) * fr);
      }
      named_barrier_sync(2, 128);
      if (blockIdx.x == 0) {
        for (int c = t; c < D; c += 128) n_last[(size_t)p * D + c] = sm.n[c];
        if (t == 0) m_last[p] = cm[(size_t)p * (NC + 1) + NC];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tm, 512);
  }
}

#undef SQ
#undef SK

}  // namespace

bool fused_tc_supported(int S, int L, int D, int DV, bool bf16) {
  return bf16 && L == kL && (D == 64 || D == 128 || D == 256) && DV % kTile == 0 && S > 0 && S % kL == 0;
}

size_t fused_tc_smem_bytes(int D) { return (size_t)6 * D * kL * 2 + (size_t)kL * kL * 2 + 1024; }

cudaError_t launch_fused_tc(const void *q, const void *k, const void *v, bool out_bf16, const float *gb,
                            const float *gx, const float *gu, const float *cm, int P, int S, int D, int DV,
                            const float *C_init, const float *n_init, void *h, float *C_last, float *n_last,
                            float *m_last, int *err, cudaStream_t stream) {
  CUtensorMap mq, mk;
  if (!make_tmap_2d_b16(&mq, q, true, (uint64_t)P * S, D, D, 64, kL)) return cudaErrorInvalidValue;
  if (!make_tmap_2d_b16(&mk, k, true, (uint64_t)P * S, D, D, 64, kL)) return cudaErrorInvalidValue;
  const size_t smem = fused_tc_smem_bytes(D);
  dim3 grid(DV / kTile, P);
  if (out_bf16) {
    auto kern = fused_tc_kernel<__nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, stream>>>(mq, mk, (const __nv_bfloat16 *)v, gb, gx, gu, cm, S, D, DV, C_init,
                                           n_init, (__nv_bfloat16 *)h, C_last, n_last, m_last, err);
  } else {
    auto kern = fused_tc_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, stream>>>(mq, mk, (const __nv_bfloat16 *)v, gb, gx, gu, cm, S, D, DV, C_init,
                                           n_init, (float *)h, C_last, n_last, m_last, err);
  }
  return cudaGetLastError();
}

}  // namespace mlstm
