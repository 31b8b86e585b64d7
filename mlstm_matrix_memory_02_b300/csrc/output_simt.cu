// output_simt.cu -- kernel (c), CUDA-core version: the intra-chunk output.
//
// Page "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural Networks"
// (llms.blog), section 3 "The Parallel Dual Form" (H = ((Q K^T) o S) V with the causal decay
// matrix S_ij = prod_{tau=j+1..i} f_tau * i_j), applied inside one chunk, plus the state
// entering the chunk (the unrolled C_T written from the chunk start); section 3 retrieval
// h~_t = C_t q_t / max(|n_t^T q_t|, .) and section 2 stabiliser.  For row r of chunk k with
// entering state (C, n, m_in) and gate quantities b, x, u from the gate kernel:
//   m_r   = b_r + max(m_in, u_r)
//   D_rj  = exp(x_j - max(m_in, u_r))            (j <= r; 0 above the diagonal)
//   beta_r = exp(m_in - max(m_in, u_r))
//   num_r = sum_j D_rj (q_r . khat_j) v_j + beta_r C q_r
//   den_r = sum_j D_rj (q_r . khat_j)     + beta_r n . q_r
//   h_r   = num_r / max(|den_r|, exp(-m_r))
// Every exponent is <= 0.
//
// CTA = (chunk, 32 output columns, pair); 256 threads.  fp32 throughout (CUDA cores):
// the path for fp32 inputs and the reference-precision path for every shape.
#include "common.cuh"
#include "kernels.cuh"

namespace mlstm {

namespace {
constexpr int kCols = 32;  // output columns (of d_v) per CTA
constexpr int kSlab = 32;  // d_qk columns staged at a time
}  // namespace

template <typename T, typename TO, int L>
__global__ void __launch_bounds__(256) output_simt_kernel(
    const T *__restrict__ qin, const T *__restrict__ kin, const T *__restrict__ vin,
    const float *__restrict__ gb, const float *__restrict__ gx, const float *__restrict__ gu,
    const float *__restrict__ cm, const float *__restrict__ Cs, const float *__restrict__ ns,
    int S, int DQK, int DV, TO *__restrict__ h, float *__restrict__ den_out, const float *__restrict__ xq,
    const float *__restrict__ pm, const float *__restrict__ nq) {
  constexpr int RB = L / 16;  // S-tile rows/cols per thread (16 x 16 thread grid)
  extern __shared__ float smem[];
  float *sP = smem;                        // [L][L+1]   S, then P = S o D
  float *sQ = sP + L * (L + 1);            // [L][kSlab+1]
  constexpr int KR = L > kCols ? L : kCols;
  float *sK = sQ + L * (kSlab + 1);        // [KR][kSlab+1]  (keys, later the C slab rows)
  float *sV = sK + KR * (kSlab + 1);       // [L][kCols]
  float *sRow = sV + L * kCols;            // [L]: den (intra, then full)
  float *sMr = sRow + L;                   // [L]: max(m_in, u_r)
  float *sDenX = sMr + L;                  // [L]: n . q_r

  const int kc = blockIdx.x, a0 = blockIdx.y * kCols, p = blockIdx.z;
  const int NC = S / L;
  const int tid = threadIdx.x;
  const size_t tbase = (size_t)p * S + (size_t)kc * L;
  const float scale = rsqrtf((float)DQK);
  const float m_in = cm[(size_t)p * (NC + 1) + kc];
  const float *C = Cs + ((size_t)p * (NC + 1) + kc) * (size_t)DV * DQK;  // entering state
  const float *nv = ns + ((size_t)p * (NC + 1) + kc) * (size_t)DQK;

  if (tid < L) {
    sMr[tid] = fmaxf(m_in, gu[tbase + tid]);
    sDenX[tid] = pm != nullptr ? nq[tbase + tid] : 0.f;
  }

  // ---- S = Q K^T over d_qk in slabs; thread (ty, tx) owns rows ty + 16 i, cols tx + 16 j
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
      sQ[r * (kSlab + 1) + c] = to_f32(qin[(tbase + r) * DQK + c0 + c]);
      sK[r * (kSlab + 1) + c] = to_f32(kin[(tbase + r) * DQK + c0 + c]);
    }
    __syncthreads();
#pragma unroll 4
    for (int c = 0; c < kSlab; ++c) {
      float qa[RB], ka[RB];
#pragma unroll
      for (int i = 0; i < RB; ++i) qa[i] = sQ[(ty + 16 * i) * (kSlab + 1) + c];
#pragma unroll
      for (int j = 0; j < RB; ++j) ka[j] = sK[(tx + 16 * j) * (kSlab + 1) + c];
#pragma unroll
      for (int i = 0; i < RB; ++i)
#pragma unroll
        for (int j = 0; j < RB; ++j) s[i][j] = fmaf(qa[i], ka[j], s[i][j]);
    }
    // n . q_r for this slab: warp w handles rows w, w + 8, ...
    {
      const int lane = tid & 31, warp = tid >> 5;
      for (int r = warp; r < L; r += 8) {
        float part = sQ[r * (kSlab + 1) + lane] * nv[c0 + lane];
        part = warp_sum(part);
        if (lane == 0) sDenX[r] += part;
      }
    }
  }
  // ---- P = S o D (causal), fp32 (or the chunk's P formed once elsewhere); row sums give the
  // intra-chunk denominator
  if (pm != nullptr) {
    const float *pc = pm + ((size_t)p * NC + kc) * L * L;
    for (int e = tid; e < L * L; e += blockDim.x) sP[(e / L) * (L + 1) + e % L] = pc[e];
  } else {
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      const int r = ty + 16 * i;
#pragma unroll
      for (int j = 0; j < RB; ++j) {
        const int jj = tx + 16 * j;
        float pv = 0.f;
        if (jj <= r) pv = s[i][j] * scale * expf(gx[tbase + jj] - sMr[r]);
        sP[r * (L + 1) + jj] = pv;
      }
    }
  }
  __syncthreads();
  if (tid < L) {
    float acc = 0.f;
    for (int j = 0; j <= tid; ++j) acc += sP[tid * (L + 1) + j];
    sRow[tid] = acc;
  }

  // ---- num = P V + beta Q C^T for 32 columns; thread (ry, ax) owns rows ry + 8 i
  constexpr int RR = L / 8;
  const int ry = tid >> 5, ax = tid & 31;
  float num_in[RR], num_x[RR];
#pragma unroll
  for (int i = 0; i < RR; ++i) num_in[i] = num_x[i] = 0.f;
  for (int e = tid; e < L * kCols; e += blockDim.x) {
    const int r = e / kCols, a = e - r * kCols;
    sV[r * kCols + a] = to_f32(vin[(tbase + r) * DV + a0 + a]);
  }
  __syncthreads();
  {
    // register tiles of L/16 rows x 2 columns (thread (rq, cq): rows RQ rq + i, columns 2 cq + j),
    // so that each shared-memory read feeds two or more products; then back to the
    // row-per-thread layout through shared memory
    constexpr int RQ = L / 16;
    const int cq = tid & 15, rq = tid >> 4;
    float an[RQ][2];
#pragma unroll
    for (int i = 0; i < RQ; ++i) an[i][0] = an[i][1] = 0.f;
#pragma unroll 4
    for (int j = 0; j < L; ++j) {
      const float v0 = sV[j * kCols + 2 * cq], v1 = sV[j * kCols + 2 * cq + 1];
#pragma unroll
      for (int i = 0; i < RQ; ++i) {
        const float pr = sP[(RQ * rq + i) * (L + 1) + j];
        an[i][0] = fmaf(pr, v0, an[i][0]);
        an[i][1] = fmaf(pr, v1, an[i][1]);
      }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < RQ; ++i) {
      sV[(RQ * rq + i) * kCols + 2 * cq] = an[i][0];
      sV[(RQ * rq + i) * kCols + 2 * cq + 1] = an[i][1];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < RR; ++i) num_in[i] = sV[(ry + 8 * i) * kCols + ax];
  }
  for (int c0 = 0; c0 < DQK && xq == nullptr; c0 += kSlab) {
    __syncthreads();
    for (int e = tid; e < L * kSlab; e += blockDim.x) {
      const int r = e / kSlab, c = e - r * kSlab;
      sQ[r * (kSlab + 1) + c] = to_f32(qin[(tbase + r) * DQK + c0 + c]);
    }
    for (int e = tid; e < kCols * kSlab; e += blockDim.x) {
      const int a = e / kSlab, c = e - a * kSlab;
      sK[a * (kSlab + 1) + c] = C[(size_t)(a0 + a) * DQK + c0 + c];
    }
    __syncthreads();
#pragma unroll 4
    for (int c = 0; c < kSlab; ++c) {
      const float cv = sK[ax * (kSlab + 1) + c];
#pragma unroll
      for (int i = 0; i < RR; ++i) num_x[i] = fmaf(sQ[(ry + 8 * i) * (kSlab + 1) + c], cv, num_x[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < RR; ++i) {
    const int r = ry + 8 * i;
    if (xq != nullptr) num_x[i] = xq[(tbase + r) * DV + a0 + ax];  // C q_r, from the state product
    const float mr = sMr[r];
    const float beta = expf(m_in - mr);
    const float den = sRow[r] + beta * sDenX[r];
    const float floor_ = expf(-(gb[tbase + r] + mr));
    const float out = (num_in[i] + beta * num_x[i]) / fmaxf(fabsf(den), floor_);
    h[(tbase + r) * DV + a0 + ax] = from_f32<TO>(out);
    if (den_out != nullptr && blockIdx.y == 0 && ax == 0) den_out[tbase + r] = den;
  }
}

template <typename T, typename TO, int L>
static cudaError_t launch_output_simt_t(const void *q, const void *k, const void *v, const float *gb,
                                        const float *gx, const float *gu, const float *cm,
                                        const float *Cs, const float *ns, int P, int S, int DQK,
                                        int DV, void *h, float *den_out, const float *xq, const float *pm,
                                        const float *nq, cudaStream_t stream) {
  constexpr int KR = L > kCols ? L : kCols;
  const size_t smem = sizeof(float) * ((size_t)L * (L + 1) + (size_t)(L + KR) * (kSlab + 1) +
                                       (size_t)L * kCols + 3 * (size_t)L);
  auto kern = output_simt_kernel<T, TO, L>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  dim3 grid(S / L, DV / kCols, P);
  kern<<<grid, 256, smem, stream>>>((const T *)q, (const T *)k, (const T *)v, gb, gx, gu, cm, Cs,
                                    ns, S, DQK, DV, (TO *)h, den_out, xq, pm, nq);
  return cudaGetLastError();
}

template <typename T, typename TO>
static cudaError_t dispatch_L(int L, const void *q, const void *k, const void *v, const float *gb,
                              const float *gx, const float *gu, const float *cm, const float *Cs,
                              const float *ns, int P, int S, int DQK, int DV, void *h,
                              float *den, const float *xq, const float *pm, const float *nq, cudaStream_t st) {
  switch (L) {
    case 16: return launch_output_simt_t<T, TO, 16>(q, k, v, gb, gx, gu, cm, Cs, ns, P, S, DQK, DV, h, den, xq, pm, nq, st);
    case 32: return launch_output_simt_t<T, TO, 32>(q, k, v, gb, gx, gu, cm, Cs, ns, P, S, DQK, DV, h, den, xq, pm, nq, st);
    case 64: return launch_output_simt_t<T, TO, 64>(q, k, v, gb, gx, gu, cm, Cs, ns, P, S, DQK, DV, h, den, xq, pm, nq, st);
    case 128: return launch_output_simt_t<T, TO, 128>(q, k, v, gb, gx, gu, cm, Cs, ns, P, S, DQK, DV, h, den, xq, pm, nq, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_output_simt(const void *q, const void *k, const void *v, bool bf16, bool out_bf16,
                               const float *gb, const float *gx, const float *gu, const float *cm,
                               const float *Cs, const float *ns, int P, int S, int L, int DQK, int DV,
                               void *h, cudaStream_t stream, float *den_out, const float *xq, const float *pm,
                               const float *nq) {
  if (P == 0 || S == 0) return cudaSuccess;
  if (bf16) {
    if (out_bf16)
      return dispatch_L<__nv_bfloat16, __nv_bfloat16>(L, q, k, v, gb, gx, gu, cm, Cs, ns, P, S, DQK, DV, h, den_out, xq, pm, nq, stream);
    return dispatch_L<__nv_bfloat16, float>(L, q, k, v, gb, gx, gu, cm, Cs, ns, P, S, DQK, DV, h, den_out, xq, pm, nq, stream);
  }
  if (out_bf16)
    return dispatch_L<float, __nv_bfloat16>(L, q, k, v, gb, gx, gu, cm, Cs, ns, P, S, DQK, DV, h, den_out, xq, pm, nq, stream);
  return dispatch_L<float, float>(L, q, k, v, gb, gx, gu, cm, Cs, ns, P, S, DQK, DV, h, den_out, xq, pm, nq, stream);
}

}  // namespace mlstm
