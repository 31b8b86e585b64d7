// gates.cu -- kernel (a): gate preprocessing for the chunkwise mLSTM forward.
//
// Page "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural Networks"
// (llms.blog), section 2 "The Normalizer State and Numerical Stabilization": the
// stabiliser m_t = max(log f_t + m_{t-1}, i~_t), here with log f_t = log sigmoid(f~_t)
// (section 3 allows the sigmoid forget gate); section 3 "The Parallel Dual Form" and
// section 5: the chunked form is built on prefix sums ("associative prefix scans").
//
// Inside chunk k (tokens t = kL + r, r = 0..L-1) with m_in = m after chunk k-1:
//   b_r = sum_{rho <= r} log f            (in-chunk inclusive prefix sum)
//   x_r = i~_r - b_r                      u_r = max_{rho <= r} x_rho
// Unrolling the stabiliser gives, for the token at r and for the chunk end,
//   m_t   = b_r + max(m_in, u_r)
//   m_out = b_{L-1} + max(m_in, u_{L-1})
// so every decay and gate factor of the chunk is an exponential of a difference of these
// quantities and never exceeds 1.
#include "common.cuh"
#include "kernels.cuh"

namespace mlstm {

// One CTA per (batch, head) pair; warp w walks chunks w, w + nwarps, ...  Each lane owns
// E = max(L/32, 1) consecutive tokens of the chunk.
__global__ void __launch_bounds__(256) gates_kernel(const float *__restrict__ ig,
                                                    const float *__restrict__ fg, int S, int L,
                                                    const float *__restrict__ m_init,
                                                    float *__restrict__ gb, float *__restrict__ gx,
                                                    float *__restrict__ gu, float *__restrict__ cm,
                                                    float *__restrict__ m_tok, int exp_fg) {
  const int p = blockIdx.x;
  const int NC = S / L;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int E = L >= 32 ? L / 32 : 1;
  const bool active = lane * E < L;
  const size_t base = (size_t)p * S;

  for (int kc = warp; kc < NC; kc += nwarps) {
    const size_t t0 = base + (size_t)kc * L + (size_t)lane * E;
    float lf[4], xi[4];
    float bsum = 0.f;
    for (int e = 0; e < E; ++e) {
      lf[e] = active ? log_forget(fg[t0 + e], exp_fg) : 0.f;
      bsum += lf[e];
      lf[e] = bsum;  // lane-local inclusive prefix
    }
    // warp-wide exclusive prefix of the lane totals
    float incl = bsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const float excl = incl - bsum;
    float xmax = -INFINITY;
    for (int e = 0; e < E; ++e) {
      lf[e] += excl;  // b_r
      xi[e] = active ? ig[t0 + e] - lf[e] : -INFINITY;
      xmax = fmaxf(xmax, xi[e]);
    }
    // warp-wide exclusive running max of the lane maxima
    float imax = xmax;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, imax, o);
      if (lane >= o) imax = fmaxf(imax, y);
    }
    float run = __shfl_up_sync(0xffffffffu, imax, 1);
    if (lane == 0) run = -INFINITY;
    if (active) {
      for (int e = 0; e < E; ++e) {
        run = fmaxf(run, xi[e]);
        gb[t0 + e] = lf[e];
        gx[t0 + e] = xi[e];
        gu[t0 + e] = run;
      }
    }
  }
  __syncthreads();  // makes this CTA's global writes visible to its own threads

  // Chunk-level stabiliser chain m^{(k+1)} = b_L + max(m^{(k)}, u_L), in token order.
  // Warp 0: lanes fetch 32 chunk ends at a time, lane 0 walks them.
  if (warp == 0) {
    float m = m_init ? m_init[p] : 0.f;
    if (lane == 0) cm[(size_t)p * (NC + 1)] = m;
    for (int k0 = 0; k0 < NC; k0 += 32) {
      const int kc = k0 + lane;
      float bl = 0.f, ul = 0.f;
      if (kc < NC) {
        const size_t te = base + (size_t)kc * L + (L - 1);
        bl = gb[te];
        ul = gu[te];
      }
      float mine = 0.f;
      for (int j = 0; j < 32 && k0 + j < NC; ++j) {
        const float b_ = __shfl_sync(0xffffffffu, bl, j);
        const float u_ = __shfl_sync(0xffffffffu, ul, j);
        m = b_ + fmaxf(m, u_);
        if (lane == j) mine = m;
      }
      if (kc < NC) cm[(size_t)p * (NC + 1) + kc + 1] = mine;
    }
  }
  if (m_tok == nullptr) return;
  __syncthreads();
  for (int i = threadIdx.x; i < S; i += blockDim.x) {
    const int kc = i / L;
    const float m_in = cm[(size_t)p * (NC + 1) + kc];
    m_tok[base + i] = gb[base + i] + fmaxf(m_in, gu[base + i]);
  }
}

cudaError_t launch_gates(const float *ig, const float *fg, int P, int S, int L, const float *m_init,
                         float *gb, float *gx, float *gu, float *cm, float *m_tok,
                         cudaStream_t stream, bool exp_fg) {
  if (P == 0) return cudaSuccess;
  gates_kernel<<<P, 256, 0, stream>>>(ig, fg, S, L, m_init, gb, gx, gu, cm, m_tok, exp_fg ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace mlstm
