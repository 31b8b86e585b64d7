// bwd_simt.cu -- backward of the chunkwise mLSTM cell forward on CUDA cores, fp32 arithmetic.
//
// Page "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural Networks"
// (llms.blog): section 3 "The Parallel Dual Form" (the cell as a masked, decay-weighted
// attention, trained in parallel), "Associative Matrix Cell State" (C_t = f_t C_{t-1} +
// i_t v_t khat_t^T, n_t likewise, h~_t = C_t q_t / max(|n_t^T q_t|, 1)) and section 2 (the
// stabiliser m_t, which rescales C and n by exp(-m_t) and changes no value of h).
//
// The gradients are those of the unstabilised cell, carried in the stabilised frame so that every
// factor is one the forward already forms (all <= 1).  With D_t = max(|n_t . q_t|, exp(-m_t)),
// s_t = sign(n_t . q_t) where |n_t . q_t| > exp(-m_t) (else 0: the floor depends on neither q nor
// n), g_t = dh_t / D_t and c_t = -(dh_t . h_t) s_t / D_t, and the decay weight of a pair (u, t),
// t <= u, E_ut = exp(i~_t + sum_{tau=t+1..u} log f_tau - m_u):
//   dq_u  = sum_{t<=u} E_ut (g_u . v_t + c_u) khat_t   (+ the entering state's part)
//   dk_t  = sum_{u>=t} E_ut (g_u . v_t + c_u) q_u / sqrt(d)
//   dv_t  = sum_{u>=t} E_ut (q_u . khat_t) g_u
//   di~_t = k_t . dk_t,   df~_t = (1 - f_t) sum_{tau>=t} (q_tau . dq_tau - k_tau . dk_tau)
// (each pair's term depends on the forget gates strictly between its ends, so d/d log f_t sums
// the pairs that straddle t: those ending at or after t minus those starting at or after t).
// Chunked with chunk L: inside a chunk the pairs form L x L matrices (the forward's decay
// matrix); across chunks they pass through the forward's boundary states C^(k), n^(k) (for dq)
// and through the adjoint states entering each boundary from the right,
//   G^(k) = alpha_k G^(k+1) + sum_{u in chunk k} beta_u g_u q_u^T,   N^(k) likewise with c_u q_u,
// (alpha_k the forward's chunk decay, beta_u = exp(m^(k) - max(m^(k), u_u)) its entering-state
// factor) for dk and dv, weighted by the forward's state-update weights w_t.  With an initial
// state, dC0 = G^(0), dn0 = N^(0) and dm0 = <G^(0), C0> + N^(0) . n0.
#include "common.cuh"
#include "kernels.cuh"

namespace mlstm {

namespace {
constexpr int kCols = 32;    // output columns per CTA (of d_qk for dq/dk, of d_v for dv)
constexpr int kSlab = 32;    // reduction columns staged in shared memory at a time
constexpr int kRows = 16;    // adjoint-state rows per CTA
constexpr int kTok = 16;     // tokens staged at a time by the adjoint-state kernel
constexpr int kMaxCols = 8;  // d_qk <= 512 = 64 threads x 8
}  // namespace

// ---------------------------------------------------------------- per-token 1 / D_t and c_t
template <typename T>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const T *__restrict__ dh, const float *__restrict__ h32,
                                                       const float *__restrict__ den, const float *__restrict__ gb,
                                                       const float *__restrict__ gu, const float *__restrict__ cm,
                                                       int S, int L, int DV, long long tokens,
                                                       float *__restrict__ invD, float *__restrict__ cc) {
  const long long tok = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (tok >= tokens) return;
  const int lane = threadIdx.x & 31;
  const int p = (int)(tok / S), t = (int)(tok % S), NC = S / L;
  float dot = 0.f;
  for (int a = lane; a < DV; a += 32) dot = fmaf(to_f32(dh[(size_t)tok * DV + a]), h32[(size_t)tok * DV + a], dot);
  dot = warp_sum(dot);
  if (lane == 0) {
    const float m_in = cm[(size_t)p * (NC + 1) + t / L];
    const float floor_ = expf(-(gb[tok] + fmaxf(m_in, gu[tok])));
    const float a = den[tok];
    const float D = fmaxf(fabsf(a), floor_);
    const float s = fabsf(a) > floor_ ? (a > 0.f ? 1.f : -1.f) : 0.f;
    invD[tok] = 1.f / D;
    cc[tok] = -dot * s / D;
  }
}

// ---------------------------------------------------------------- adjoint states, right to left
// CTA (16 rows of G, head): each thread keeps 4 rows x ceil(DQK / 64) columns in registers
// through all chunks, walking them from the last to the first; Gs/Ns [P, NC+1, ...] receive the
// state entering every boundary (G^(NC) = 0).
template <typename T>
__global__ void __launch_bounds__(256) bwd_states_kernel(
    const T *__restrict__ qin, const T *__restrict__ dh, const float *__restrict__ invD,
    const float *__restrict__ cc, const float *__restrict__ gb, const float *__restrict__ gu,
    const float *__restrict__ cm, int S, int L, int DQK, int DV, float *__restrict__ Gs, float *__restrict__ Ns) {
  __shared__ float sK[kTok][512];
  __shared__ float sV[kTok][kRows];
  __shared__ float sB[kTok], sC[kTok];
  const int p = blockIdx.y, a0 = blockIdx.x * kRows;
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;
  const int NC = S / L;
  const int ncol = (DQK + 63) / 64;
  const bool do_n = blockIdx.x == 0 && ty == 0;
  float acc[4][kMaxCols], nacc[kMaxCols];
#pragma unroll
  for (int j = 0; j < kMaxCols; ++j) {
    nacc[j] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i][j] = 0.f;
  }
  auto store_state = [&](int kb) {
    float *G = Gs + ((size_t)p * (NC + 1) + kb) * (size_t)DV * DQK;
    float *N = Ns + ((size_t)p * (NC + 1) + kb) * (size_t)DQK;
#pragma unroll
    for (int j = 0; j < kMaxCols; ++j) {
      const int c = tx + 64 * j;
      if (j < ncol && c < DQK) {
#pragma unroll
        for (int i = 0; i < 4; ++i) G[(size_t)(a0 + ty * 4 + i) * DQK + c] = acc[i][j];
        if (do_n) N[c] = nacc[j];
      }
    }
  };
  store_state(NC);
  for (int kc = NC - 1; kc >= 0; --kc) {
    const size_t tbase = (size_t)p * S + (size_t)kc * L;
    const float m_in = cm[(size_t)p * (NC + 1) + kc];
    const float m_out = cm[(size_t)p * (NC + 1) + kc + 1];
    const float alpha = expf(gb[tbase + L - 1] + m_in - m_out);
#pragma unroll
    for (int j = 0; j < kMaxCols; ++j) {
      nacc[j] *= alpha;
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i][j] *= alpha;
    }
    for (int r0 = 0; r0 < L; r0 += kTok) {
      __syncthreads();
      if (threadIdx.x < kTok) {
        const size_t u = tbase + r0 + threadIdx.x;
        sB[threadIdx.x] = expf(m_in - fmaxf(m_in, gu[u]));
        sC[threadIdx.x] = cc[u];
      }
      __syncthreads();
      for (int e = threadIdx.x; e < kTok * DQK; e += blockDim.x) {
        const int r = e / DQK, c = e - r * DQK;
        sK[r][c] = to_f32(qin[(tbase + r0 + r) * DQK + c]) * sB[r];
      }
      for (int e = threadIdx.x; e < kTok * kRows; e += blockDim.x) {
        const int r = e / kRows, a = e - r * kRows;
        sV[r][a] = to_f32(dh[(tbase + r0 + r) * DV + a0 + a]) * invD[tbase + r0 + r];
      }
      __syncthreads();
#pragma unroll 4
      for (int r = 0; r < kTok; ++r) {
        float vv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) vv[i] = sV[r][ty * 4 + i];
        const float cr = sC[r];
#pragma unroll
        for (int j = 0; j < kMaxCols; ++j) {
          if (j < ncol) {
            const int c = tx + 64 * j;
            const float kk = c < DQK ? sK[r][c] : 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i][j] = fmaf(vv[i], kk, acc[i][j]);
            if (do_n) nacc[j] = fmaf(cr, kk, nacc[j]);
          }
        }
      }
    }
    store_state(kc);
  }
}

// ---------------------------------------------------------------- dq and dk
// CTA (chunk, 32 columns of d_qk, head), 256 threads.  M1_ut = E_ut (g_u . v_t + c_u) for t <= u
// (an L x L matrix over d_v), then for the CTA's columns
//   dq = M1 khat + beta (g C^(k) + c n^(k)),   dk = (M1^T q + w (v G^(k+1) + N^(k+1))) / sqrt(d)
// and each row's partial sums of q . dq and k . dk over the columns.
template <typename T, int L>
__global__ void __launch_bounds__(256) bwd_dqdk_kernel(
    const T *__restrict__ qin, const T *__restrict__ kin, const T *__restrict__ vin, const T *__restrict__ dh,
    const float *__restrict__ invD, const float *__restrict__ cc, const float *__restrict__ gb,
    const float *__restrict__ gx, const float *__restrict__ gu, const float *__restrict__ cm,
    const float *__restrict__ Cs, const float *__restrict__ ns, const float *__restrict__ Gs,
    const float *__restrict__ Ns, int S, int DQK, int DV, T *__restrict__ dq, T *__restrict__ dk,
    float *__restrict__ part_q, float *__restrict__ part_k, const float *__restrict__ yq,
    const float *__restrict__ yk, const float *__restrict__ m1) {
  constexpr int RB = L / 16;  // L x L tile entries per thread (16 x 16 thread grid)
  constexpr int RR = L / 8;   // output rows per thread (8 x 32 thread grid)
  constexpr int KR = L > kSlab ? L : kSlab;
  extern __shared__ float smem[];
  float *sM = smem;                  // [L][L+1]  M1
  float *sA = sM + L * (L + 1);      // [L][kSlab+1]
  float *sB = sA + L * (kSlab + 1);  // [KR][kSlab+1]
  float *sInv = sB + KR * (kSlab + 1);
  float *sC = sInv + L, *sMx = sC + L, *sGx = sMx + L, *sBeta = sGx + L, *sW = sBeta + L;

  const int kc = blockIdx.x, c0 = blockIdx.y * kCols, p = blockIdx.z;
  const int NC = S / L, ntiles = DQK / kCols;
  const int tid = threadIdx.x;
  const size_t tbase = (size_t)p * S + (size_t)kc * L;
  const float scale = rsqrtf((float)DQK);
  const float m_in = cm[(size_t)p * (NC + 1) + kc], m_out = cm[(size_t)p * (NC + 1) + kc + 1];
  const float bl = gb[tbase + L - 1];
  if (tid < L) {
    const size_t u = tbase + tid;
    const float mx = fmaxf(m_in, gu[u]);
    sInv[tid] = invD[u];
    sC[tid] = cc[u];
    sMx[tid] = mx;
    sGx[tid] = gx[u];
    sBeta[tid] = expf(m_in - mx);
    sW[tid] = expf(bl + gx[u] - m_out);
  }

  // ---- A = g V^T over d_v; thread (ty, tx) owns rows ty + 16 i, columns tx + 16 j
  const int ty = tid >> 4, tx = tid & 15;
  float s[RB][RB];
#pragma unroll
  for (int i = 0; i < RB; ++i)
#pragma unroll
    for (int j = 0; j < RB; ++j) s[i][j] = 0.f;
  for (int a0 = 0; a0 < DV && m1 == nullptr; a0 += kSlab) {
    __syncthreads();
    for (int e = tid; e < L * kSlab; e += blockDim.x) {
      const int r = e / kSlab, a = e - r * kSlab;
      sA[r * (kSlab + 1) + a] = to_f32(dh[(tbase + r) * DV + a0 + a]) * sInv[r];
      sB[r * (kSlab + 1) + a] = to_f32(vin[(tbase + r) * DV + a0 + a]);
    }
    __syncthreads();
#pragma unroll 4
    for (int a = 0; a < kSlab; ++a) {
      float ga[RB], vb[RB];
#pragma unroll
      for (int i = 0; i < RB; ++i) ga[i] = sA[(ty + 16 * i) * (kSlab + 1) + a];
#pragma unroll
      for (int j = 0; j < RB; ++j) vb[j] = sB[(tx + 16 * j) * (kSlab + 1) + a];
#pragma unroll
      for (int i = 0; i < RB; ++i)
#pragma unroll
        for (int j = 0; j < RB; ++j) s[i][j] = fmaf(ga[i], vb[j], s[i][j]);
    }
  }
  if (m1 != nullptr) {  // the chunk's M1, formed once
    __syncthreads();
    const float *mc = m1 + ((size_t)p * NC + kc) * L * L;
    for (int e = tid; e < L * L; e += blockDim.x) sM[(e / L) * (L + 1) + e % L] = mc[e];
  } else {
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      const int u = ty + 16 * i;
#pragma unroll
      for (int j = 0; j < RB; ++j) {
        const int t = tx + 16 * j;
        sM[u * (L + 1) + t] = t <= u ? (s[i][j] + sC[u]) * expf(sGx[t] - sMx[u]) : 0.f;
      }
    }
  }

  // ---- intra-chunk parts for the CTA's 32 columns; thread (ry, cx) owns rows ry + 8 i
  const int ry = tid >> 5, cx = tid & 31;
  float dq_in[RR], dk_in[RR], dq_x[RR], dk_x[RR];
#pragma unroll
  for (int i = 0; i < RR; ++i) dq_in[i] = dk_in[i] = dq_x[i] = dk_x[i] = 0.f;
  __syncthreads();
  for (int e = tid; e < L * kCols; e += blockDim.x) {
    const int r = e / kCols, c = e - r * kCols;
    sA[r * (kSlab + 1) + c] = to_f32(qin[(tbase + r) * DQK + c0 + c]);
    sB[r * (kSlab + 1) + c] = to_f32(kin[(tbase + r) * DQK + c0 + c]) * scale;
  }
  __syncthreads();
  {
    // register tiles of L/16 rows x 2 columns (thread (rq, cq): rows RQ rq + i, columns 2 cq + j),
    // so that each shared-memory read feeds two or more products
    constexpr int RQ = L / 16;
    const int cq = tid & 15, rq = tid >> 4;
    float aq[RQ][2], ak[RQ][2];
#pragma unroll
    for (int i = 0; i < RQ; ++i) aq[i][0] = aq[i][1] = ak[i][0] = ak[i][1] = 0.f;
#pragma unroll 4
    for (int t = 0; t < L; ++t) {
      const float k0 = sB[t * (kSlab + 1) + 2 * cq], k1 = sB[t * (kSlab + 1) + 2 * cq + 1];
      const float q0 = sA[t * (kSlab + 1) + 2 * cq], q1 = sA[t * (kSlab + 1) + 2 * cq + 1];
#pragma unroll
      for (int i = 0; i < RQ; ++i) {
        const float mr = sM[(RQ * rq + i) * (L + 1) + t];  // M1[u][t]: sum_t M1[u][t] khat_t
        const float mc = sM[t * (L + 1) + RQ * rq + i];    // M1[t][u]: sum_t M1[t][u] q_t
        aq[i][0] = fmaf(mr, k0, aq[i][0]);
        aq[i][1] = fmaf(mr, k1, aq[i][1]);
        ak[i][0] = fmaf(mc, q0, ak[i][0]);
        ak[i][1] = fmaf(mc, q1, ak[i][1]);
      }
    }
    // back to the row-per-thread layout of the rest of the kernel, through shared memory
    __syncthreads();
#pragma unroll
    for (int i = 0; i < RQ; ++i)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        sA[(RQ * rq + i) * (kSlab + 1) + 2 * cq + j] = aq[i][j];
        sB[(RQ * rq + i) * (kSlab + 1) + 2 * cq + j] = ak[i][j];
      }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < RR; ++i) {
      dq_in[i] = sA[(ry + 8 * i) * (kSlab + 1) + cx];
      dk_in[i] = sB[(ry + 8 * i) * (kSlab + 1) + cx];
    }
  }

  // ---- inter-chunk parts: g C^(k) (entering state) and v G^(k+1) (adjoint from the right)
  const float *Ck = Cs + ((size_t)p * (NC + 1) + kc) * (size_t)DV * DQK;
  const float *Gk = Gs + ((size_t)p * (NC + 1) + kc + 1) * (size_t)DV * DQK;
  for (int pass = 0; pass < 2 && yq == nullptr; ++pass) {
    const float *St = pass == 0 ? Ck : Gk;
    for (int a0 = 0; a0 < DV; a0 += kSlab) {
      __syncthreads();
      for (int e = tid; e < L * kSlab; e += blockDim.x) {
        const int r = e / kSlab, a = e - r * kSlab;
        sA[r * (kSlab + 1) + a] = pass == 0 ? to_f32(dh[(tbase + r) * DV + a0 + a]) * sInv[r]
                                            : to_f32(vin[(tbase + r) * DV + a0 + a]);
      }
      for (int e = tid; e < kSlab * kCols; e += blockDim.x) {
        const int a = e / kCols, c = e - a * kCols;
        sB[a * (kSlab + 1) + c] = St[(size_t)(a0 + a) * DQK + c0 + c];
      }
      __syncthreads();
#pragma unroll 4
      for (int a = 0; a < kSlab; ++a) {
        const float sv = sB[a * (kSlab + 1) + cx];
#pragma unroll
        for (int i = 0; i < RR; ++i) {
          const float x = sA[(ry + 8 * i) * (kSlab + 1) + a] * sv;
          if (pass == 0) dq_x[i] += x;
          else dk_x[i] += x;
        }
      }
    }
  }
  const float nk = ns[((size_t)p * (NC + 1) + kc) * DQK + c0 + cx];
  const float Nk = Ns[((size_t)p * (NC + 1) + kc + 1) * DQK + c0 + cx];
#pragma unroll
  for (int i = 0; i < RR; ++i) {
    const int u = ry + 8 * i;
    const size_t at = (tbase + u) * DQK + c0 + cx;
    if (yq != nullptr) {
      dq_x[i] = yq[at];
      dk_x[i] = yk[at];
    }
    const float dqv = dq_in[i] + sBeta[u] * (dq_x[i] + sC[u] * nk);
    const float dkv = scale * (dk_in[i] + sW[u] * (dk_x[i] + Nk));
    dq[at] = from_f32<T>(dqv);
    dk[at] = from_f32<T>(dkv);
    const float pq = warp_sum(to_f32(qin[at]) * dqv);
    const float pk = warp_sum(to_f32(kin[at]) * dkv);
    if (cx == 0) {
      part_q[(tbase + u) * ntiles + blockIdx.y] = pq;
      part_k[(tbase + u) * ntiles + blockIdx.y] = pk;
    }
  }
}

// ---------------------------------------------------------------- dv
// CTA (chunk, 32 columns of d_v, head).  M2_ut = E_ut (q_u . khat_t) (the forward's decay-weighted
// score matrix), then dv = M2^T g + w (khat G^(k+1)^T) for the CTA's columns.
template <typename T, int L>
__global__ void __launch_bounds__(256) bwd_dv_kernel(
    const T *__restrict__ qin, const T *__restrict__ kin, const T *__restrict__ dh, const float *__restrict__ invD,
    const float *__restrict__ gb, const float *__restrict__ gx, const float *__restrict__ gu,
    const float *__restrict__ cm, const float *__restrict__ Gs, int S, int DQK, int DV, T *__restrict__ dv,
    const float *__restrict__ yv, const float *__restrict__ pm) {
  constexpr int RB = L / 16;
  constexpr int RR = L / 8;
  constexpr int KR = L > kSlab ? L : kSlab;
  extern __shared__ float smem[];
  float *sM = smem;                  // [L][L+1]  M2
  float *sA = sM + L * (L + 1);      // [L][kSlab+1]
  float *sB = sA + L * (kSlab + 1);  // [KR][kSlab+1]
  float *sInv = sB + KR * (kSlab + 1);
  float *sMx = sInv + L, *sGx = sMx + L, *sW = sGx + L;

  const int kc = blockIdx.x, a0 = blockIdx.y * kCols, p = blockIdx.z;
  const int NC = S / L;
  const int tid = threadIdx.x;
  const size_t tbase = (size_t)p * S + (size_t)kc * L;
  const float scale = rsqrtf((float)DQK);
  const float m_in = cm[(size_t)p * (NC + 1) + kc], m_out = cm[(size_t)p * (NC + 1) + kc + 1];
  const float bl = gb[tbase + L - 1];
  if (tid < L) {
    const size_t u = tbase + tid;
    sInv[tid] = invD[u];
    sMx[tid] = fmaxf(m_in, gu[u]);
    sGx[tid] = gx[u];
    sW[tid] = expf(bl + gx[u] - m_out);
  }
  const int ty = tid >> 4, tx = tid & 15;
  float s[RB][RB];
#pragma unroll
  for (int i = 0; i < RB; ++i)
#pragma unroll
    for (int j = 0; j < RB; ++j) s[i][j] = 0.f;
  for (int c0 = 0; c0 < DQK && pm == nullptr; c0 += kSlab) {
    __syncthreads();
    for (int e = tid; e < L * kSlab; e += blockDim.x) {
      const int r = e / kSlab, c = e - r * kSlab;
      sA[r * (kSlab + 1) + c] = to_f32(qin[(tbase + r) * DQK + c0 + c]);
      sB[r * (kSlab + 1) + c] = to_f32(kin[(tbase + r) * DQK + c0 + c]);
    }
    __syncthreads();
#pragma unroll 4
    for (int c = 0; c < kSlab; ++c) {
      float qa[RB], kb[RB];
#pragma unroll
      for (int i = 0; i < RB; ++i) qa[i] = sA[(ty + 16 * i) * (kSlab + 1) + c];
#pragma unroll
      for (int j = 0; j < RB; ++j) kb[j] = sB[(tx + 16 * j) * (kSlab + 1) + c];
#pragma unroll
      for (int i = 0; i < RB; ++i)
#pragma unroll
        for (int j = 0; j < RB; ++j) s[i][j] = fmaf(qa[i], kb[j], s[i][j]);
    }
  }
  if (pm != nullptr) {  // the chunk's P, formed once
    __syncthreads();
    const float *pc = pm + ((size_t)p * NC + kc) * L * L;
    for (int e = tid; e < L * L; e += blockDim.x) sM[(e / L) * (L + 1) + e % L] = pc[e];
  } else {
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      const int u = ty + 16 * i;
#pragma unroll
      for (int j = 0; j < RB; ++j) {
        const int t = tx + 16 * j;
        sM[u * (L + 1) + t] = t <= u ? s[i][j] * scale * expf(sGx[t] - sMx[u]) : 0.f;
      }
    }
  }
  const int ry = tid >> 5, ax = tid & 31;
  float dv_in[RR], dv_x[RR];
#pragma unroll
  for (int i = 0; i < RR; ++i) dv_in[i] = dv_x[i] = 0.f;
  __syncthreads();
  for (int e = tid; e < L * kCols; e += blockDim.x) {
    const int r = e / kCols, a = e - r * kCols;
    sA[r * (kSlab + 1) + a] = to_f32(dh[(tbase + r) * DV + a0 + a]) * sInv[r];
  }
  __syncthreads();
  {
    // register tiles of L/16 rows x 2 columns, as in the dq/dk kernel: sum_u M2[u][t] g_u
    constexpr int RQ = L / 16;
    const int cq = tid & 15, rq = tid >> 4;
    float av[RQ][2];
#pragma unroll
    for (int i = 0; i < RQ; ++i) av[i][0] = av[i][1] = 0.f;
#pragma unroll 4
    for (int u = 0; u < L; ++u) {
      const float g0 = sA[u * (kSlab + 1) + 2 * cq], g1 = sA[u * (kSlab + 1) + 2 * cq + 1];
#pragma unroll
      for (int i = 0; i < RQ; ++i) {
        const float mc = sM[u * (L + 1) + RQ * rq + i];
        av[i][0] = fmaf(mc, g0, av[i][0]);
        av[i][1] = fmaf(mc, g1, av[i][1]);
      }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < RQ; ++i)
#pragma unroll
      for (int j = 0; j < 2; ++j) sB[(RQ * rq + i) * (kSlab + 1) + 2 * cq + j] = av[i][j];
    __syncthreads();
#pragma unroll
    for (int i = 0; i < RR; ++i) dv_in[i] = sB[(ry + 8 * i) * (kSlab + 1) + ax];
    __syncthreads();  // the inter-chunk part below restages sA and sB
  }
  const float *Gk = Gs + ((size_t)p * (NC + 1) + kc + 1) * (size_t)DV * DQK;
  for (int c0 = 0; c0 < DQK && yv == nullptr; c0 += kSlab) {
    __syncthreads();
    for (int e = tid; e < L * kSlab; e += blockDim.x) {
      const int r = e / kSlab, c = e - r * kSlab;
      sA[r * (kSlab + 1) + c] = to_f32(kin[(tbase + r) * DQK + c0 + c]) * scale;
    }
    for (int e = tid; e < kCols * kSlab; e += blockDim.x) {
      const int a = e / kSlab, c = e - a * kSlab;
      sB[a * (kSlab + 1) + c] = Gk[(size_t)(a0 + a) * DQK + c0 + c];
    }
    __syncthreads();
#pragma unroll 4
    for (int c = 0; c < kSlab; ++c) {
      const float gv = sB[ax * (kSlab + 1) + c];
#pragma unroll
      for (int i = 0; i < RR; ++i) dv_x[i] = fmaf(sA[(ry + 8 * i) * (kSlab + 1) + c], gv, dv_x[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < RR; ++i) {
    const int t = ry + 8 * i;
    if (yv != nullptr) dv_x[i] = yv[(tbase + t) * DV + a0 + ax];
    dv[(tbase + t) * DV + a0 + ax] = from_f32<T>(dv_in[i] + sW[t] * dv_x[i]);
  }
}

// ---------------------------------------------------------------- di~, df~, dm0
// One CTA per head.  Each thread owns a contiguous run of tokens; the suffix sums of
// R_t = q_t . dq_t - k_t . dk_t run in double precision.
__global__ void __launch_bounds__(256) bwd_gates_kernel(
    const float *__restrict__ fg, int exp_fg, const float *__restrict__ part_q, const float *__restrict__ part_k,
    int S, int ntiles, const float *__restrict__ Gs0, const float *__restrict__ Ns0, size_t gs_stride,
    size_t ns_stride, const float *__restrict__ C_init, const float *__restrict__ n_init, int DQK, int DV,
    float *__restrict__ dig, float *__restrict__ dfg, float *__restrict__ dm_init) {
  __shared__ double s_run[256];
  const int p = blockIdx.x, tid = threadIdx.x;
  const int seg = (S + blockDim.x - 1) / blockDim.x;
  const int t0 = tid * seg < S ? tid * seg : S, t1 = t0 + seg < S ? t0 + seg : S;
  auto R = [&](int t, float &kdk) {
    const size_t base = ((size_t)p * S + t) * ntiles;
    float qdq = 0.f;
    kdk = 0.f;
    for (int j = 0; j < ntiles; ++j) {
      qdq += part_q[base + j];
      kdk += part_k[base + j];
    }
    return (double)qdq - (double)kdk;
  };
  double local = 0.0;
  for (int t = t0; t < t1; ++t) {
    float kdk;
    local += R(t, kdk);
  }
  s_run[tid] = local;
  __syncthreads();
  if (tid == 0) {
    double run = 0.0;
    for (int i = (int)blockDim.x - 1; i >= 0; --i) {
      const double x = s_run[i];
      s_run[i] = run;
      run += x;
    }
  }
  __syncthreads();
  double run = s_run[tid];  // R summed over the tokens after this thread's run
  for (int t = t1 - 1; t >= t0; --t) {
    float kdk;
    run += R(t, kdk);
    const size_t at = (size_t)p * S + t;
    const float f = fg[at];
    // d log f / d f~: 1 - sigmoid(f~) = 1 / (1 + exp(f~)) for the sigmoid gate, 1 for f = exp(f~)
    const float dlogf = exp_fg ? 1.f : 1.f / (1.f + expf(f));
    dig[at] = kdk;
    dfg[at] = (float)run * dlogf;
  }
  if (dm_init != nullptr) {
    // dm0 = <G^(0), C0> + N^(0) . n0 (zero without an initial state)
    double acc = 0.0;
    if (C_init != nullptr) {
      const float *G = Gs0 + (size_t)p * gs_stride, *C0 = C_init + (size_t)p * DV * DQK;
      for (size_t i = tid; i < (size_t)DV * DQK; i += blockDim.x) acc += (double)G[i] * C0[i];
      const float *N = Ns0 + (size_t)p * ns_stride, *n0 = n_init + (size_t)p * DQK;
      for (int i = tid; i < DQK; i += blockDim.x) acc += (double)N[i] * n0[i];
    }
    __syncthreads();
    s_run[tid] = acc;
    __syncthreads();
    for (int o = blockDim.x / 2; o > 0; o >>= 1) {
      if (tid < o) s_run[tid] += s_run[tid + o];
      __syncthreads();
    }
    if (tid == 0) dm_init[p] = (float)s_run[0];
  }
}

// ---------------------------------------------------------------- a chunk's L x L matrices
// CTA (chunk, head), 256 threads, once per chunk (the column-tile kernels then read them):
//   mode 0: P_ut = E_ut (q_u . khat_t) -- the forward's decay-weighted scores -- and n^(k) . q_u;
//   mode 1: M1_ut = E_ut (g_u . v_t + c_u) with g_u = dh_u / D_u;
// t <= u, zero above the diagonal; out [P, NC, L, L] fp32 (row u, column t).
template <typename T, int L>
__global__ void __launch_bounds__(256) bwd_mat_kernel(
    int mode, const T *__restrict__ xin, const T *__restrict__ yin, int K, const float *__restrict__ invD,
    const float *__restrict__ cc, const float *__restrict__ gx, const float *__restrict__ gu,
    const float *__restrict__ cm, const float *__restrict__ ns, int S, int DQK, float *__restrict__ out,
    float *__restrict__ nq) {
  constexpr int RB = L / 16;
  __shared__ float sX[L][kSlab + 1], sY[L][kSlab + 1];
  __shared__ float sMx[L], sGx[L], sW[L], sC[L];
  const int kc = blockIdx.x, p = blockIdx.y, tid = threadIdx.x;
  const int NC = S / L;
  const size_t tbase = (size_t)p * S + (size_t)kc * L;
  const float m_in = cm[(size_t)p * (NC + 1) + kc];
  if (tid < L) {
    sMx[tid] = fmaxf(m_in, gu[tbase + tid]);
    sGx[tid] = gx[tbase + tid];
    sW[tid] = mode == 1 ? invD[tbase + tid] : 1.f;
    sC[tid] = mode == 1 ? cc[tbase + tid] : 0.f;
  }
  const float *nv = ns + ((size_t)p * (NC + 1) + kc) * (size_t)DQK;
  const int ty = tid >> 4, tx = tid & 15, lane = tid & 31, warp = tid >> 5;
  float s[RB][RB];
#pragma unroll
  for (int i = 0; i < RB; ++i)
#pragma unroll
    for (int j = 0; j < RB; ++j) s[i][j] = 0.f;
  float nqa[L / 8];
#pragma unroll
  for (int i = 0; i < L / 8; ++i) nqa[i] = 0.f;
  for (int c0 = 0; c0 < K; c0 += kSlab) {
    __syncthreads();
    for (int e = tid; e < L * kSlab; e += blockDim.x) {
      const int r = e / kSlab, c = e - r * kSlab;
      sX[r][c] = to_f32(xin[(tbase + r) * K + c0 + c]) * sW[r];
      sY[r][c] = to_f32(yin[(tbase + r) * K + c0 + c]);
    }
    __syncthreads();
#pragma unroll 4
    for (int c = 0; c < kSlab; ++c) {
      float xa[RB], yb[RB];
#pragma unroll
      for (int i = 0; i < RB; ++i) xa[i] = sX[ty + 16 * i][c];
#pragma unroll
      for (int j = 0; j < RB; ++j) yb[j] = sY[tx + 16 * j][c];
#pragma unroll
      for (int i = 0; i < RB; ++i)
#pragma unroll
        for (int j = 0; j < RB; ++j) s[i][j] = fmaf(xa[i], yb[j], s[i][j]);
    }
    if (mode == 0) {  // n^(k) . q_u for this slab: warp w takes rows w, w + 8, ...
#pragma unroll
      for (int i = 0; i < L / 8; ++i) nqa[i] = fmaf(sX[warp + 8 * i][lane], nv[c0 + lane], nqa[i]);
    }
  }
  const float scale = mode == 0 ? rsqrtf((float)DQK) : 1.f;
  float *o = out + ((size_t)p * NC + kc) * L * L;
#pragma unroll
  for (int i = 0; i < RB; ++i) {
    const int u = ty + 16 * i;
#pragma unroll
    for (int j = 0; j < RB; ++j) {
      const int t = tx + 16 * j;
      o[u * L + t] = t <= u ? (s[i][j] * scale + sC[u]) * expf(sGx[t] - sMx[u]) : 0.f;
    }
  }
  if (mode == 0) {
#pragma unroll
    for (int i = 0; i < L / 8; ++i) {
      const float x = warp_sum(nqa[i]);
      if (lane == 0) nq[tbase + warp + 8 * i] = x;
    }
  }
}

// ---------------------------------------------------------------- bf16 (or fp32) to fp32
// Eight elements per thread and step: a 16-byte load of bf16 (or two of fp32), two 16-byte stores
// (n a multiple of 8, both pointers 16-byte aligned).
__global__ void to_f32_kernel(const void *__restrict__ src, int bf16, float *__restrict__ dst, size_t n) {
  const size_t n8 = n / 8;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    float4 a, b;
    if (bf16) {
      const uint4 u = reinterpret_cast<const uint4 *>(src)[i];
      a = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                      __uint_as_float(u.y & 0xffff0000u));
      b = make_float4(__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xffff0000u), __uint_as_float(u.w << 16),
                      __uint_as_float(u.w & 0xffff0000u));
    } else {
      a = reinterpret_cast<const float4 *>(src)[2 * i];
      b = reinterpret_cast<const float4 *>(src)[2 * i + 1];
    }
    reinterpret_cast<float4 *>(dst)[2 * i] = a;
    reinterpret_cast<float4 *>(dst)[2 * i + 1] = b;
  }
}

// ---------------------------------------------------------------- launchers
cudaError_t launch_bwd_mat(int mode, const void *x, const void *y, bool bf16, int K, const float *invD,
                           const float *cc, const float *gx, const float *gu, const float *cm, const float *ns, int P,
                           int S, int L, int DQK, float *out, float *nq, cudaStream_t stream) {
  if (P == 0 || S == 0) return cudaSuccess;
  dim3 grid(S / L, P);
#define MLSTM_BWD_MAT(T_, L_)                                                                                  \
  bwd_mat_kernel<T_, L_><<<grid, 256, 0, stream>>>(mode, (const T_ *)x, (const T_ *)y, K, invD, cc, gx, gu, cm, \
                                                    ns, S, DQK, out, nq);                                       \
  return cudaGetLastError()
  if (bf16) {
    switch (L) {
      case 16: MLSTM_BWD_MAT(__nv_bfloat16, 16);
      case 32: MLSTM_BWD_MAT(__nv_bfloat16, 32);
      case 64: MLSTM_BWD_MAT(__nv_bfloat16, 64);
      case 128: MLSTM_BWD_MAT(__nv_bfloat16, 128);
    }
  } else {
    switch (L) {
      case 16: MLSTM_BWD_MAT(float, 16);
      case 32: MLSTM_BWD_MAT(float, 32);
      case 64: MLSTM_BWD_MAT(float, 64);
      case 128: MLSTM_BWD_MAT(float, 128);
    }
  }
#undef MLSTM_BWD_MAT
  return cudaErrorInvalidValue;
}

cudaError_t launch_to_f32(const void *src, bool bf16, float *dst, size_t n, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  if (n % 8 != 0) return cudaErrorInvalidValue;
  const size_t n8 = n / 8, blocks = (n8 + 255) / 256 < 4096 ? (n8 + 255) / 256 : 4096;
  to_f32_kernel<<<(unsigned)blocks, 256, 0, stream>>>(src, bf16 ? 1 : 0, dst, n);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep(const void *dh, bool bf16, const float *h32, const float *den, const float *gb,
                            const float *gu, const float *cm, int P, int S, int L, int DV, float *invD, float *cc,
                            cudaStream_t stream) {
  const long long tokens = (long long)P * S;
  if (tokens == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((tokens + 7) / 8);
  if (bf16)
    bwd_prep_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>((const __nv_bfloat16 *)dh, h32, den, gb, gu, cm, S,
                                                                L, DV, tokens, invD, cc);
  else
    bwd_prep_kernel<float><<<blocks, 256, 0, stream>>>((const float *)dh, h32, den, gb, gu, cm, S, L, DV, tokens,
                                                       invD, cc);
  return cudaGetLastError();
}

cudaError_t launch_bwd_states(const void *q, const void *dh, bool bf16, const float *invD, const float *cc,
                              const float *gb, const float *gu, const float *cm, int P, int S, int L, int DQK,
                              int DV, float *Gs, float *Ns, cudaStream_t stream) {
  if (P == 0) return cudaSuccess;
  dim3 grid(DV / kRows, P);
  if (bf16)
    bwd_states_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>((const __nv_bfloat16 *)q, (const __nv_bfloat16 *)dh,
                                                               invD, cc, gb, gu, cm, S, L, DQK, DV, Gs, Ns);
  else
    bwd_states_kernel<float><<<grid, 256, 0, stream>>>((const float *)q, (const float *)dh, invD, cc, gb, gu, cm, S,
                                                       L, DQK, DV, Gs, Ns);
  return cudaGetLastError();
}

namespace {
template <int L>
size_t chunk_smem(int scalars) {
  constexpr int KR = L > kSlab ? L : kSlab;
  return sizeof(float) * ((size_t)L * (L + 1) + (size_t)(L + KR) * (kSlab + 1) + (size_t)scalars * L);
}

template <typename T, int L>
cudaError_t dqdk_t(const void *q, const void *k, const void *v, const void *dh, const float *invD, const float *cc,
                   const float *gb, const float *gx, const float *gu, const float *cm, const float *Cs,
                   const float *ns, const float *Gs, const float *Ns, int P, int S, int DQK, int DV, void *dq,
                   void *dk, float *part_q, float *part_k, const float *yq, const float *yk, const float *m1,
                   cudaStream_t stream) {
  auto kern = bwd_dqdk_kernel<T, L>;
  const size_t smem = chunk_smem<L>(6);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(S / L, DQK / kCols, P), 256, smem, stream>>>((const T *)q, (const T *)k, (const T *)v, (const T *)dh,
                                                           invD, cc, gb, gx, gu, cm, Cs, ns, Gs, Ns, S, DQK, DV,
                                                           (T *)dq, (T *)dk, part_q, part_k, yq, yk, m1);
  return cudaGetLastError();
}

template <typename T, int L>
cudaError_t dv_t(const void *q, const void *k, const void *dh, const float *invD, const float *gb, const float *gx,
                 const float *gu, const float *cm, const float *Gs, int P, int S, int DQK, int DV, void *dv,
                 const float *yv, const float *pm, cudaStream_t stream) {
  auto kern = bwd_dv_kernel<T, L>;
  const size_t smem = chunk_smem<L>(4);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(S / L, DV / kCols, P), 256, smem, stream>>>((const T *)q, (const T *)k, (const T *)dh, invD, gb, gx,
                                                          gu, cm, Gs, S, DQK, DV, (T *)dv, yv, pm);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_bwd_dqdk(const void *q, const void *k, const void *v, const void *dh, bool bf16,
                            const float *invD, const float *cc, const float *gb, const float *gx, const float *gu,
                            const float *cm, const float *Cs, const float *ns, const float *Gs, const float *Ns,
                            int P, int S, int L, int DQK, int DV, void *dq, void *dk, float *part_q,
                            float *part_k, cudaStream_t stream, const float *yq, const float *yk,
                            const float *m1) {
  if (P == 0 || S == 0) return cudaSuccess;
#define MLSTM_BWD_DQDK(T_, L_)                                                                                   \
  return dqdk_t<T_, L_>(q, k, v, dh, invD, cc, gb, gx, gu, cm, Cs, ns, Gs, Ns, P, S, DQK, DV, dq, dk, part_q, \
                        part_k, yq, yk, m1, stream)
  if (bf16) {
    switch (L) {
      case 16: MLSTM_BWD_DQDK(__nv_bfloat16, 16);
      case 32: MLSTM_BWD_DQDK(__nv_bfloat16, 32);
      case 64: MLSTM_BWD_DQDK(__nv_bfloat16, 64);
      case 128: MLSTM_BWD_DQDK(__nv_bfloat16, 128);
    }
  } else {
    switch (L) {
      case 16: MLSTM_BWD_DQDK(float, 16);
      case 32: MLSTM_BWD_DQDK(float, 32);
      case 64: MLSTM_BWD_DQDK(float, 64);
      case 128: MLSTM_BWD_DQDK(float, 128);
    }
  }
#undef MLSTM_BWD_DQDK
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_dv(const void *q, const void *k, const void *dh, bool bf16, const float *invD,
                          const float *gb, const float *gx, const float *gu, const float *cm, const float *Gs,
                          int P, int S, int L, int DQK, int DV, void *dv, cudaStream_t stream, const float *yv,
                          const float *pm) {
  if (P == 0 || S == 0) return cudaSuccess;
#define MLSTM_BWD_DV(T_, L_) return dv_t<T_, L_>(q, k, dh, invD, gb, gx, gu, cm, Gs, P, S, DQK, DV, dv, yv, pm, stream)
  if (bf16) {
    switch (L) {
      case 16: MLSTM_BWD_DV(__nv_bfloat16, 16);
      case 32: MLSTM_BWD_DV(__nv_bfloat16, 32);
      case 64: MLSTM_BWD_DV(__nv_bfloat16, 64);
      case 128: MLSTM_BWD_DV(__nv_bfloat16, 128);
    }
  } else {
    switch (L) {
      case 16: MLSTM_BWD_DV(float, 16);
      case 32: MLSTM_BWD_DV(float, 32);
      case 64: MLSTM_BWD_DV(float, 64);
      case 128: MLSTM_BWD_DV(float, 128);
    }
  }
#undef MLSTM_BWD_DV
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_gates(const float *fg, bool exp_fg, const float *part_q, const float *part_k, int P, int S,
                             int ntiles, const float *Gs0, const float *Ns0, size_t gs_stride, size_t ns_stride,
                             const float *C_init, const float *n_init, int DQK, int DV, float *dig, float *dfg,
                             float *dm_init, cudaStream_t stream) {
  if (P == 0) return cudaSuccess;
  bwd_gates_kernel<<<P, 256, 0, stream>>>(fg, exp_fg ? 1 : 0, part_q, part_k, S, ntiles, Gs0, Ns0, gs_stride,
                                          ns_stride, C_init, n_init, DQK, DV, dig, dfg, dm_init);
  return cudaGetLastError();
}

}  // namespace mlstm
