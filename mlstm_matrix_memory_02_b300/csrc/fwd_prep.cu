// fwd_prep.cu -- the parts of the tensor-core forward that do not depend on the matrix state,
// done once per (head, chunk) ahead of the state walk.
//
// Page "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural Networks"
// (llms.blog): section 3 "The Parallel Dual Form" (inside a chunk H = ((Q K^T) o D) V with the
// decay matrix D), section 3 "Associative Matrix Cell State" (the normaliser n and the
// denominator max(|n^T q|, .), k scaled by 1/sqrt(d)), section 2 (the max stabiliser) and the
// chunked form's prefix sums (section 5).  Per chunk k of a head, with b, x = i~ - b and the
// running max u of the chunk (as in the gate kernel), the entering stabiliser m_in and
// mr_r = max(m_in, u_r):
//   P_rj  = (q_r . k_j) / sqrt(d) * exp(x_j - mr_r)   for j <= r (0 above the diagonal)
//   den_r = sum_j P_rj                                 (the in-chunk part of the denominator)
//   beta_r q_r with beta_r = exp(m_in - mr_r)          (the query of the state product)
//   w_j k_j  with the update weight of token j in the frame of the state walk
//   dn_k  = sum_j w_j k_j / sqrt(d)                    (the chunk's increment of n)
// Every one of these is the same for all d_v tiles of a head, so it is computed here once
// instead of in each tile of the state walk (fwd_state.cu).  Four kernels, in stream order:
//   gate chain  per head: the gate prefix sums of every chunk, the stabiliser chain and the
//               frame of the state walk over the chunks, every token's factors
//   pre-pass    per (chunk, head), four CTAs to an SM (the whole grid of the 1.3B layer resident
//               at once): q and k arrive by TMA in four parts of d_qk; for each part one thread
//               issues its share of Q K^T on the tensor cores (M = 64, N = 64, bf16 in, fp32
//               accumulated in tensor memory) while every thread converts the part into the fp16
//               operands beta q and w k and sums the n increment; warps 0-3 then read S from
//               tensor memory and write P (fp16) and its row sums
//   n chain     per head: n_{k+1} = alpha_k n_k + dn_k over the chunks (n entering each chunk)
//   denominator per (chunk, head): 1 / max(|den_r + beta_r n_k . q_r|, exp(-m_r)) per token
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

constexpr int kLp = 64;                  // chunk length
constexpr int kPrepThreads = 256;
constexpr int kPrepParts = 4;            // d_qk in four parts: 42 KB of shared memory, four CTAs per SM
constexpr int kPrepMaxChunks = 64;       // chunks per head this path takes (S <= 4096)
constexpr float kFrameLog = 5.545177444479562f;  // ln(2^8): largest lazy frame factor of the state walk

struct PrepSmem {
  uint64_t full, done;
  uint32_t tmem_base;
  float x[kLp], mr[kLp], beta[kLp], wk[kLp], wt[kLp];
};

// b, x and u of the 64 tokens of one chunk (lane owns tokens 2 lane, 2 lane + 1), in the
// operations and order of the gate kernel: in-chunk inclusive prefix of log f, x = i~ - b and
// the running max of x.
__device__ __forceinline__ void chunk_scan(const float *__restrict__ ig, const float *__restrict__ fg, size_t tok0,
                                           int lane, int exp_fg, float (&bb)[2], float (&xx)[2], float (&uu)[2]) {
  const float2 f2 = *reinterpret_cast<const float2 *>(fg + tok0 + 2 * lane);
  const float2 i2 = *reinterpret_cast<const float2 *>(ig + tok0 + 2 * lane);
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
}

// Per head: the gate prefix sums of every chunk (one warp per chunk), the stabiliser chain
// m_out = b_L + max(m_in, u_L) and the frame of the state walk over the chunks (one thread, in
// chunk order: the same operations as the fused kernel's gate warp), then every token's factors.
// tok4 = (x, mr, beta, w in the walk's frame / sqrt(d)), tok2 = (w / sqrt(d), exp(-m)); per chunk
// cdat = (m_in, m_out, alpha, frame after), (exp(frame), exp(frame) alpha, lazy, 0).
__global__ void __launch_bounds__(1024) fwd_gchain_kernel(const float *__restrict__ ig, const float *__restrict__ fg,
                                                          const float *__restrict__ m_init, int S, float scale,
                                                          int exp_fg, float4 *__restrict__ tok4,
                                                          float2 *__restrict__ tok2, float4 *__restrict__ cdat) {
  __shared__ float endb[kPrepMaxChunks], endu[kPrepMaxChunks];
  __shared__ float c_min[kPrepMaxChunks], c_mout[kPrepMaxChunks], c_sig[kPrepMaxChunks];
  pdl_trigger();
  const int p = blockIdx.x, NC = S / kLp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  constexpr int kPer = kPrepMaxChunks / 32;  // chunks a warp holds (blockDim.x = 1024)
  float kb[kPer][2], kx[kPer][2], ku[kPer][2];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int c = warp + nw * j;
    if (c < NC) {
      chunk_scan(ig, fg, (size_t)p * S + (size_t)c * kLp, lane, exp_fg, kb[j], kx[j], ku[j]);
      if (lane == 31) {
        endb[c] = kb[j][1];
        endu[c] = ku[j][1];
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = m_init ? m_init[p] : 0.f, sigma = 0.f;
    for (int c = 0; c < NC; ++c) {
      const float m_in = m, bl = endb[c];
      const float m_out = bl + fmaxf(m_in, endu[c]);
      const float log_alpha = bl + m_in - m_out;  // <= 0
      const bool lazy = -(sigma + log_alpha) <= kFrameLog;
      const float sig_next = lazy ? sigma + log_alpha : 0.f;
      c_min[c] = m_in;
      c_mout[c] = m_out;
      c_sig[c] = sig_next;
      cdat[2 * ((size_t)p * NC + c)] = make_float4(m_in, m_out, __expf(log_alpha), sig_next);
      cdat[2 * ((size_t)p * NC + c) + 1] =
          make_float4(__expf(sigma), __expf(sigma + log_alpha), lazy ? 1.f : 0.f, 0.f);
      sigma = sig_next;
      m = m_out;
    }
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int c = warp + nw * j;
    if (c < NC) {
      const float m_in = c_min[c], m_out = c_mout[c], bl = endb[c], sig_next = c_sig[c];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const size_t t = (size_t)p * S + (size_t)c * kLp + 2 * lane + i;
        const float mr = fmaxf(m_in, ku[j][i]);
        tok4[t] = make_float4(kx[j][i], mr, __expf(m_in - mr), __expf(bl + kx[j][i] - m_out - sig_next) * scale);
        tok2[t] = make_float2(__expf(bl + kx[j][i] - m_out) * scale, __expf(-(kb[j][i] + mr)));
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kPrepThreads, 4) fwd_prep_kernel(
    const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
    const float4 *__restrict__ tok4, const float2 *__restrict__ tok2, int S, float scale, __half *__restrict__ qb,
    __half *__restrict__ kw, __half *__restrict__ pm, float *__restrict__ den, float *__restrict__ dn,
    int *__restrict__ err) {
  constexpr int NP = kPrepParts;           // q and k arrive in NP parts of d_qk
  constexpr int DH = D / NP;               // columns per part
  constexpr int HBYTES = DH * 128;         // a [64 x DH] 2-byte tile: DH / 64 swizzled blocks of 8 KB
  constexpr int CPR = DH / 8;              // 16-byte chunks per row of a part
  constexpr int RG = kPrepThreads / CPR;   // rows converted at once
  static_assert(DH % 64 == 0 && D <= 512 && kPrepThreads % CPR == 0, "D");
  extern __shared__ uint8_t prep_dyn[];
  __shared__ PrepSmem sm;
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(prep_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t *const sq = base, *const sk = base + HBYTES;
  float *const spart = reinterpret_cast<float *>(base + 2 * HBYTES);  // [RG][DH] partial sums of w k

  const int k = blockIdx.x, p = blockIdx.y, NC = S / kLp;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t tok0 = (size_t)p * S + (size_t)k * kLp;
  pdl_trigger();

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
  // q and k columns [hf DH, hf DH + DH) of the chunk into the (single) stage
  auto load_half = [&](int hf) {
    mbar_arrive_expect_tx(&sm.full, 2u * HBYTES);
#pragma unroll 1
    for (int b = 0; b < DH / 64; ++b) {
      tma_load_2d(sq + b * 8192, &mapQ, hf * DH + b * 64, (int)tok0, &sm.full);
      tma_load_2d(sk + b * 8192, &mapK, hf * DH + b * 64, (int)tok0, &sm.full);
    }
  };
  if (tid == 0) {
    prefetch_tensormap(&mapQ);
    prefetch_tensormap(&mapK);
    load_half(0);
  }

  pdl_wait();  // the gate factors come from the previous kernel
  if (tid < kLp) {
    const float4 a4 = tok4[tok0 + tid];
    sm.x[tid] = a4.x;
    sm.mr[tid] = a4.y;
    sm.beta[tid] = a4.z;
    sm.wk[tid] = a4.w;
    sm.wt[tid] = tok2[tok0 + tid].x;
  }
  __syncthreads();

  bool ok = true;
#pragma unroll 1
  for (int hf = 0; hf < NP; ++hf) {
    ok = __syncthreads_and(mbar_wait(&sm.full, hf & 1, err, 101)) != 0;
    if (!ok) break;
    if (tid == 32) {
      // S += Q K^T over this part's columns (M = 64, N = 64, K = DH)
      tc_fence_after();
      const uint32_t id_S = idesc_f16(64, kLp, /*bf16*/ 1, 0, 0);
      const uint64_t dq = smem_desc(smem_u32(sq), 16, 1024, kSwizzle128B);
      const uint64_t dk = smem_desc(smem_u32(sk), 16, 1024, kSwizzle128B);
#pragma unroll 1
      for (int c = 0; c < DH / 16; ++c) {
        const uint64_t off = (uint64_t)(((c >> 2) * 8192 + (c & 3) * 32) >> 4);
        mma_f16_ss(tm, dq + off, dk + off, id_S, (hf | c) != 0);
      }
      mma_commit(&sm.done);
    }
    // beta q and w k of this part into the 16-bit operands (global, row-major), and the partial
    // sums of the n increment per row group: thread = (16-byte column chunk, row group)
    {
      const int ch = tid % CPR, rg = tid / CPR;
      const int cb = (ch >> 3) * 8192, c8 = ch & 7;
      const size_t gcol = (size_t)hf * DH + ch * 8;
      uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll 4
      for (int r = rg; r < kLp; r += RG) {
        const int off = cb + r * 128 + ((c8 ^ (r & 7)) << 4);
        const uint4 rq = *reinterpret_cast<const uint4 *>(sq + off);
        const uint4 rk = *reinterpret_cast<const uint4 *>(sk + off);
        const uint64_t bq2 = f2pack(sm.beta[r], sm.beta[r]);
        const uint64_t wk2 = f2pack(sm.wk[r], sm.wk[r]), wt2 = f2pack(sm.wt[r], sm.wt[r]);
        uint4 oq, ok4;
        oq.x = f2_to_h2(f2mul(bf2_to_f2(rq.x), bq2));
        oq.y = f2_to_h2(f2mul(bf2_to_f2(rq.y), bq2));
        oq.z = f2_to_h2(f2mul(bf2_to_f2(rq.z), bq2));
        oq.w = f2_to_h2(f2mul(bf2_to_f2(rq.w), bq2));
        const uint64_t x0 = bf2_to_f2(rk.x), x1 = bf2_to_f2(rk.y), x2 = bf2_to_f2(rk.z), x3 = bf2_to_f2(rk.w);
        acc[0] = f2fma(wt2, x0, acc[0]);
        acc[1] = f2fma(wt2, x1, acc[1]);
        acc[2] = f2fma(wt2, x2, acc[2]);
        acc[3] = f2fma(wt2, x3, acc[3]);
        ok4.x = f2_to_h2(f2mul(x0, wk2));
        ok4.y = f2_to_h2(f2mul(x1, wk2));
        ok4.z = f2_to_h2(f2mul(x2, wk2));
        ok4.w = f2_to_h2(f2mul(x3, wk2));
        *reinterpret_cast<uint4 *>(qb + (tok0 + r) * D + gcol) = oq;
        *reinterpret_cast<uint4 *>(kw + (tok0 + r) * D + gcol) = ok4;
      }
      float *sp = spart + rg * DH + ch * 8;
#pragma unroll
      for (int e = 0; e < 4; ++e) *reinterpret_cast<uint64_t *>(sp + 2 * e) = acc[e];
    }
    __syncthreads();
    for (int c = tid; c < DH; c += kPrepThreads) {
      float a = 0.f;
#pragma unroll
      for (int g = 0; g < RG; ++g) a += spart[g * DH + c];
      dn[((size_t)p * NC + k) * D + hf * DH + c] = a;
    }
    if (hf + 1 < NP) {
      // the stage is reloaded once this part's products have read it (every thread has passed
      // the conversion above, which read it last)
      if (tid == 0) {
        ok = mbar_wait(&sm.done, hf & 1, err, 104);
        if (ok) load_half(hf + 1);
      }
      ok = __syncthreads_and(ok) != 0;
      if (!ok) break;
    }
  }
  // P and its row sums from S (M = 64 layout: row 16 w + l in lane l < 16 of warp w's quarter)
  if (ok && warp < 4) {
    const bool got = __all_sync(0xffffffffu, mbar_wait(&sm.done, (NP - 1) & 1, err, 102));
    if (got) {
      tc_fence_after();
      const uint32_t lb = (uint32_t)(warp * 32) << 16;
      const int r = 16 * warp + (lane & 15);
      const float mrr = sm.mr[r];
      float d = 0.f;
      uint4 *prow = reinterpret_cast<uint4 *>(pm + (((size_t)p * NC + k) * kLp + r) * kLp);
      // 16 columns of S at a time (the loads are warp-wide; lanes 16-31 hold no row)
#pragma unroll 1
      for (int c16 = 0; c16 < kLp / 16; ++c16) {
        uint32_t u[16];
        tmem_ld16(tm + lb + 16 * c16, u);
        tmem_wait_ld();
        if (lane < 16) {
#pragma unroll
          for (int h8 = 0; h8 < 2; ++h8) {
            float pv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int j = 16 * c16 + 8 * h8 + e;
              pv[e] = j <= r ? __uint_as_float(u[8 * h8 + e]) * scale * __expf(sm.x[j] - mrr) : 0.f;
              d += pv[e];
            }
            uint4 w4;
            w4.x = pack_half2(pv[0], pv[1]);
            w4.y = pack_half2(pv[2], pv[3]);
            w4.z = pack_half2(pv[4], pv[5]);
            w4.w = pack_half2(pv[6], pv[7]);
            prow[2 * c16 + h8] = w4;
          }
        }
      }
      if (lane < 16) den[tok0 + r] = d;
    }
  }
  if (!ok && tid == 0) {
    // nothing may leave while its loads or products are still in flight
    mbar_wait(&sm.full, 0, err, 103);
    mbar_wait(&sm.done, 0, err, 105);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tm, 64);
  }
}

// Per head and block of 256 columns: n entering every chunk, n_{k+1} = alpha_k n_k + dn_k from
// n_init in chunk order, written over dn in place (each dn_k is read before n_k replaces it), and
// n_last; the loads of a batch of chunks go out before their products.
__global__ void __launch_bounds__(256) fwd_nchain_kernel(float *__restrict__ dn, const float4 *__restrict__ cdat,
                                                         const float *__restrict__ n_init, int S, int D,
                                                         float *__restrict__ n_last) {
  const int p = blockIdx.y, c = blockIdx.x * 256 + threadIdx.x, NC = S / kLp;
  pdl_trigger();
  pdl_wait();  // the n increments come from the previous kernel
  if (c >= D) return;
  float *dp = dn + (size_t)p * NC * D + c;
  const float4 *cp = cdat + 2 * (size_t)p * NC;
  float n = n_init ? n_init[(size_t)p * D + c] : 0.f;
#pragma unroll 1
  for (int k0 = 0; k0 < NC; k0 += 16) {
    float a[16], d[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int kk = k0 + e < NC ? k0 + e : NC - 1;
      a[e] = cp[2 * kk].z;
      d[e] = dp[(size_t)kk * D];
    }
#pragma unroll
    for (int e = 0; e < 16; ++e)
      if (k0 + e < NC) {
        dp[(size_t)(k0 + e) * D] = n;
        n = a[e] * n + d[e];
      }
  }
  n_last[(size_t)p * D + c] = n;
}

// The reciprocal denominator of each token: inv_r = 1 / max(|den_r + beta_r n_k . q_r|, exp(-m_r)),
// n . q from the bf16 q in fp32 (the fp16 beta q operand would put its rounding into rows whose
// denominator cancels).  One CTA per (chunk, head), eight rows per warp, every row requested
// before any is reduced.
template <int D>
__global__ void __launch_bounds__(256, 4) fwd_ninv_kernel(const __nv_bfloat16 *__restrict__ q,
                                                          const float *__restrict__ nk,
                                                          const float4 *__restrict__ cdat,
                                                          const float *__restrict__ den,
                                                          const float4 *__restrict__ tok4,
                                                          const float2 *__restrict__ tok2, int S,
                                                          float *__restrict__ inv, float *__restrict__ m_last) {
  constexpr int PER = D / 32;  // elements of a row per lane
  constexpr int RB = 4;        // rows of a warp requested at once (64 registers: four CTAs per SM)
  const int k = blockIdx.x, p = blockIdx.y, NC = S / kLp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t tok0 = (size_t)p * S + (size_t)k * kLp;
  uint4 qv[RB][PER / 8];
  auto load_rows = [&](int half) {
#pragma unroll
    for (int rr = 0; rr < RB; ++rr) {
      const uint4 *qr = reinterpret_cast<const uint4 *>(q + (tok0 + warp + 8 * (RB * half + rr)) * D + lane * PER);
#pragma unroll
      for (int v8 = 0; v8 < PER / 8; ++v8) qv[rr][v8] = qr[v8];
    }
  };
  load_rows(0);
  pdl_trigger();
  pdl_wait();  // n, den and the gate factors come from the previous kernels
  float nv[PER];
  const float4 *np = reinterpret_cast<const float4 *>(nk + ((size_t)p * NC + k) * D + lane * PER);
#pragma unroll
  for (int e = 0; e < PER / 4; ++e) {
    const float4 f = np[e];
    nv[4 * e] = f.x;
    nv[4 * e + 1] = f.y;
    nv[4 * e + 2] = f.z;
    nv[4 * e + 3] = f.w;
  }
  // written here, after every CTA of the gate kernel has read m_init (which m_last may alias)
  if (k == NC - 1 && threadIdx.x == 0) m_last[p] = cdat[2 * ((size_t)p * NC + k)].y;
#pragma unroll 1
  for (int half = 0; half < 8 / RB; ++half) {
    if (half > 0) load_rows(half);
    float dots[RB];
#pragma unroll
    for (int rr = 0; rr < RB; ++rr) {
      float a = 0.f;
#pragma unroll
      for (int v8 = 0; v8 < PER / 8; ++v8) {
        const uint4 w = qv[rr][v8];
        a += bf16_lo(w.x) * nv[8 * v8] + bf16_hi(w.x) * nv[8 * v8 + 1];
        a += bf16_lo(w.y) * nv[8 * v8 + 2] + bf16_hi(w.y) * nv[8 * v8 + 3];
        a += bf16_lo(w.z) * nv[8 * v8 + 4] + bf16_hi(w.z) * nv[8 * v8 + 5];
        a += bf16_lo(w.w) * nv[8 * v8 + 6] + bf16_hi(w.w) * nv[8 * v8 + 7];
      }
      dots[rr] = a;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int rr = 0; rr < RB; ++rr) dots[rr] += __shfl_xor_sync(0xffffffffu, dots[rr], o);
    if (lane < RB) {
      float a = dots[0];
#pragma unroll
      for (int rr = 1; rr < RB; ++rr) a = lane == rr ? dots[rr] : a;
      const size_t t = tok0 + warp + 8 * (RB * half + lane);
      inv[t] = 1.f / fmaxf(fabsf(den[t] + tok4[t].z * a), tok2[t].y);
    }
  }
}

// A launch that may start while the previous kernel in the stream finishes (the kernel waits
// for it with pdl_wait before reading its results).
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Params>(args)...);
}

template <int D>
cudaError_t launch_prep_d(const void *q, const void *k, const float *ig, const float *fg, const float *m_init,
                          int P, int S, bool exp_fg, const PrepBuffers &b, const float *n_init, float *n_last,
                          float *m_last, int *err, cudaStream_t stream) {
  CUtensorMap mq, mk;
  if (!make_tmap_2d_b16(&mq, q, true, (uint64_t)P * S, D, D, 64, kLp)) return cudaErrorInvalidValue;
  if (!make_tmap_2d_b16(&mk, k, true, (uint64_t)P * S, D, D, 64, kLp)) return cudaErrorInvalidValue;
  const float scale = (float)(1.0 / __builtin_sqrt((double)D));
  fwd_gchain_kernel<<<P, 1024, 0, stream>>>(ig, fg, m_init, S, scale, exp_fg ? 1 : 0, b.tok4, b.tok2, b.cdat);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // one stage of q and k (a part of d_qk), the row-group partial sums of a part, alignment slack
  constexpr int DP = D / kPrepParts;
  const size_t smem = (size_t)2 * DP * 128 + (size_t)(kPrepThreads / (DP / 8)) * DP * 4 + 1024;
  auto kern = fwd_prep_kernel<D>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  const dim3 grid(S / kLp, P);
  e = launch_pdl(kern, grid, dim3(kPrepThreads), smem, stream, mq, mk, b.tok4, b.tok2, S, scale, b.qb, b.kw, b.pm,
                 b.den, b.dn, err);
  if (e != cudaSuccess) return e;
  e = launch_pdl(fwd_nchain_kernel, dim3((D + 255) / 256, P), dim3(256), 0, stream, b.dn, b.cdat, n_init, S, D,
                 n_last);
  if (e != cudaSuccess) return e;
  return launch_pdl(fwd_ninv_kernel<D>, grid, dim3(256), 0, stream, static_cast<const __nv_bfloat16 *>(q), b.dn,
                    b.cdat, b.den, b.tok4, b.tok2, S, b.inv, m_last);
}

}  // namespace

// d_qk = 512 only: at d_qk = 256 (two d_v tiles share the work) the five kernels measured within
// 1 % of the single fused kernel, so that size keeps the fused kernel.
bool fwd_prep_supported(int S, int D) {
  return D == 512 && S >= kLp && S % kLp == 0 && S / kLp <= kPrepMaxChunks;
}

cudaError_t launch_fwd_prep(const void *q, const void *k, const float *ig, const float *fg, const float *m_init,
                            int P, int S, int D, bool exp_fg, const PrepBuffers &b, const float *n_init,
                            float *n_last, float *m_last, int *err, cudaStream_t stream) {
  if (P == 0 || S == 0) return cudaSuccess;
  if (!fwd_prep_supported(S, D)) return cudaErrorInvalidValue;
  return launch_prep_d<512>(q, k, ig, fg, m_init, P, S, exp_fg, b, n_init, n_last, m_last, err, stream);
}

}  // namespace mlstm
