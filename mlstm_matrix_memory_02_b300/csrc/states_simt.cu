// states_simt.cu -- kernel (b), CUDA-core version: the inter-chunk recurrence.
//
// Page "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural Networks"
// (llms.blog), section 3 "Associative Matrix Cell State" (C_t = f_t C_{t-1} + i_t v_t k_t^T,
// n_t = f_t n_{t-1} + i_t k_t, k scaled by 1/sqrt(d)) unrolled over one chunk as in
// "The Parallel Dual Form" (C_T = sum_t prod f * i_t v_t k_t^T), with the section 2 stabiliser:
//   C^{(k+1)} = alpha C^{(k)} + sum_r w_r v_r khat_r^T,   n^{(k+1)} = alpha n^{(k)} + sum_r w_r khat_r
//   alpha = exp(b_{L-1} + m^{(k)} - m^{(k+1)}),          w_r = exp(b_{L-1} + x_r - m^{(k+1)})
// (b, x from the gate kernel; both factors are <= 1).
//
// Used for fp32 inputs, for every shape, and to materialise the boundary states.  The
// state is elementwise-parallel: CTA (a-tile, pair) owns 16 rows of C for all chunks and
// keeps them in registers; each thread holds 4 rows x ceil(DQK/64) columns.
#include "common.cuh"
#include "kernels.cuh"

namespace mlstm {

namespace {
constexpr int kRows = 16;     // rows of C per CTA
constexpr int kTok = 16;      // tokens staged in shared memory at a time
constexpr int kMaxCols = 8;   // DQK <= 512 = 64 threads x 8
}  // namespace

template <typename T>
__global__ void __launch_bounds__(256) states_simt_kernel(
    const T *__restrict__ kin, const T *__restrict__ vin, const float *__restrict__ gb,
    const float *__restrict__ gx, const float *__restrict__ cm, int S, int L, int DQK, int DV,
    const float *__restrict__ C_init, const float *__restrict__ n_init, float *__restrict__ Cs,
    float *__restrict__ ns, float *__restrict__ C_last, float *__restrict__ n_last) {
  __shared__ float sK[kTok][512];
  __shared__ float sV[kTok][kRows];
  __shared__ float sW[kTok];

  const int p = blockIdx.y;
  const int a0 = blockIdx.x * kRows;
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;  // 64 x 4
  const int NC = S / L;
  const float scale = rsqrtf((float)DQK);
  const int ncol = (DQK + 63) / 64;
  const bool do_n = blockIdx.x == 0 && ty == 0;

  float acc[4][kMaxCols];
  float nacc[kMaxCols];
#pragma unroll
  for (int j = 0; j < kMaxCols; ++j) {
    const int c = tx + 64 * j;
    nacc[j] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i][j] = 0.f;
    if (j < ncol && c < DQK) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int a = a0 + ty * 4 + i;
        if (C_init) acc[i][j] = C_init[((size_t)p * DV + a) * DQK + c];
      }
      if (do_n && n_init) nacc[j] = n_init[(size_t)p * DQK + c];
    }
  }

  auto store_state = [&](float *Cdst, float *ndst) {
#pragma unroll
    for (int j = 0; j < kMaxCols; ++j) {
      const int c = tx + 64 * j;
      if (j < ncol && c < DQK) {
#pragma unroll
        for (int i = 0; i < 4; ++i) Cdst[(size_t)(a0 + ty * 4 + i) * DQK + c] = acc[i][j];
        if (do_n) ndst[c] = nacc[j];
      }
    }
  };

  const size_t cs_stride = (size_t)DV * DQK;
  if (Cs) store_state(Cs + (size_t)p * (NC + 1) * cs_stride, ns + (size_t)p * (NC + 1) * DQK);

  for (int kc = 0; kc < NC; ++kc) {
    const size_t tbase = (size_t)p * S + (size_t)kc * L;
    const float m_in = cm[(size_t)p * (NC + 1) + kc];
    const float m_out = cm[(size_t)p * (NC + 1) + kc + 1];
    const float bl = gb[tbase + L - 1];
    const float alpha = expf(bl + m_in - m_out);
#pragma unroll
    for (int j = 0; j < kMaxCols; ++j) {
      nacc[j] *= alpha;
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i][j] *= alpha;
    }
    for (int r0 = 0; r0 < L; r0 += kTok) {
      __syncthreads();
      if (threadIdx.x < kTok) sW[threadIdx.x] = expf(bl + gx[tbase + r0 + threadIdx.x] - m_out);
      __syncthreads();
      for (int e = threadIdx.x; e < kTok * DQK; e += blockDim.x) {
        const int r = e / DQK, c = e - r * DQK;
        sK[r][c] = to_f32(kin[(tbase + r0 + r) * DQK + c]) * scale * sW[r];
      }
      for (int e = threadIdx.x; e < kTok * kRows; e += blockDim.x) {
        const int r = e / kRows, a = e - r * kRows;
        sV[r][a] = to_f32(vin[(tbase + r0 + r) * DV + a0 + a]);
      }
      __syncthreads();
#pragma unroll 4
      for (int r = 0; r < kTok; ++r) {
        float vv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) vv[i] = sV[r][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < kMaxCols; ++j) {
          if (j < ncol) {
            const int c = tx + 64 * j;
            const float kk = c < DQK ? sK[r][c] : 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i][j] = fmaf(vv[i], kk, acc[i][j]);
            if (do_n) nacc[j] += kk;
          }
        }
      }
    }
    if (Cs) {
      store_state(Cs + ((size_t)p * (NC + 1) + kc + 1) * cs_stride,
                  ns + ((size_t)p * (NC + 1) + kc + 1) * DQK);
    }
  }
  if (C_last) store_state(C_last + (size_t)p * cs_stride, n_last + (size_t)p * DQK);
}

cudaError_t launch_states_simt(const void *k, const void *v, bool bf16, const float *gb,
                               const float *gx, const float *cm, int P, int S, int L, int DQK,
                               int DV, const float *C_init, const float *n_init, float *Cs,
                               float *ns, float *C_last, float *n_last, cudaStream_t stream) {
  if (P == 0) return cudaSuccess;
  dim3 grid(DV / kRows, P);
  if (bf16) {
    states_simt_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
        (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, gb, gx, cm, S, L, DQK, DV, C_init,
        n_init, Cs, ns, C_last, n_last);
  } else {
    states_simt_kernel<float><<<grid, 256, 0, stream>>>((const float *)k, (const float *)v, gb,
                                                        gx, cm, S, L, DQK, DV, C_init, n_init, Cs,
                                                        ns, C_last, n_last);
  }
  return cudaGetLastError();
}

}  // namespace mlstm
