// step.cu -- kernel (d): one recurrent decode step of the mLSTM cell, in place.
//
// Page "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural Networks"
// (llms.blog): section 5 "Inference Memory and Throughput Trade-Offs" (decoding carries the
// constant-size state C, n per head), section 3 "Associative Matrix Cell State" (updates and
// retrieval, k scaled by 1/sqrt(d)) and section 2 (stabiliser), for one token:
//   m' = max(log sigmoid(f~) + m, i~),  alpha = exp(log sigmoid(f~) + m - m'),  w = exp(i~ - m')
//   C <- alpha C + w v khat^T,  n <- alpha n + w khat,  h = C q / max(|n . q|, exp(-m'))
//
// HBM-bound: C is read once and written once (2 * DV * DQK * 4 bytes per head); everything
// else is a few KB.  One CTA of 256 threads per (batch, head) -- the head's n and m are
// updated in place by the only CTA that reads them.  Rows of C are streamed with 16-byte
// loads and stores; each warp keeps several rows in flight.
#include "common.cuh"
#include "kernels.cuh"

namespace mlstm {

namespace {
constexpr int kThreads = 256;
constexpr int kMaxD = 512;
}  // namespace

template <typename T, typename TO>
__global__ void __launch_bounds__(kThreads) step_kernel(const T *__restrict__ qin, const T *__restrict__ kin,
                                                        const T *__restrict__ vin, const float *__restrict__ ig,
                                                        const float *__restrict__ fg, float *__restrict__ C,
                                                        float *__restrict__ n, float *__restrict__ m,
                                                        TO *__restrict__ h, int DQK, int DV, int exp_fg) {
  __shared__ __align__(16) float sq[kMaxD];
  __shared__ __align__(16) float sk[kMaxD];  // w * khat
  __shared__ float sv[kMaxD];
  __shared__ float sred[kThreads / 32];
  __shared__ float sden;

  const int p = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float scale = rsqrtf((float)DQK);

  const float m_old = m[p];
  const float lf = log_forget(fg[p], exp_fg);
  const float m_new = fmaxf(lf + m_old, ig[p]);
  const float alpha = expf(lf + m_old - m_new);
  const float w = expf(ig[p] - m_new);

  // n <- alpha n + w khat and its dot with q
  float part = 0.f;
  for (int c = tid; c < DQK; c += kThreads) {
    const float qc = to_f32(qin[(size_t)p * DQK + c]);
    const float kc = to_f32(kin[(size_t)p * DQK + c]) * scale * w;
    sq[c] = qc;
    sk[c] = kc;
    const float nn = fmaf(alpha, n[(size_t)p * DQK + c], kc);
    n[(size_t)p * DQK + c] = nn;
    part = fmaf(nn, qc, part);
  }
  for (int a = tid; a < DV; a += kThreads) sv[a] = to_f32(vin[(size_t)p * DV + a]);
  part = warp_sum(part);
  if (lane == 0) sred[warp] = part;
  __syncthreads();
  if (warp == 0) {
    float x = lane < kThreads / 32 ? sred[lane] : 0.f;
    x = warp_sum(x);
    if (lane == 0) sden = fmaxf(fabsf(x), expf(-m_new));
  }
  __syncthreads();
  const float inv_den = 1.f / sden;
  if (tid == 0) m[p] = m_new;

  // C rows: warp w streams rows w, w + 8, ...; lane owns float4 columns lane + 32 j.
  const int nv4 = DQK / 4;            // float4 per row (a multiple of 8)
  const int per_lane = (nv4 + 31) / 32;  // 1..4
  float4 qv[4], kv[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c4 = lane + 32 * j;
    if (j < per_lane && c4 < nv4) {
      qv[j] = reinterpret_cast<const float4 *>(sq)[c4];
      kv[j] = reinterpret_cast<const float4 *>(sk)[c4];
    } else {
      qv[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      kv[j] = qv[j];
    }
  }
  float4 *C4 = reinterpret_cast<float4 *>(C + (size_t)p * DV * DQK);
  constexpr int kRowsInFlight = 4;
  for (int a0 = warp * kRowsInFlight; a0 < DV; a0 += (kThreads / 32) * kRowsInFlight) {
    float4 x[kRowsInFlight][4];
#pragma unroll
    for (int i = 0; i < kRowsInFlight; ++i) {
      const int a = a0 + i;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c4 = lane + 32 * j;
        if (a < DV && j < per_lane && c4 < nv4) x[i][j] = __ldcs(&C4[(size_t)a * nv4 + c4]);
      }
    }
#pragma unroll
    for (int i = 0; i < kRowsInFlight; ++i) {
      const int a = a0 + i;
      if (a >= DV) break;
      const float va = sv[a];
      float dot = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c4 = lane + 32 * j;
        if (j < per_lane && c4 < nv4) {
          float4 y = x[i][j];
          y.x = fmaf(alpha, y.x, va * kv[j].x);
          y.y = fmaf(alpha, y.y, va * kv[j].y);
          y.z = fmaf(alpha, y.z, va * kv[j].z);
          y.w = fmaf(alpha, y.w, va * kv[j].w);
          __stcs(&C4[(size_t)a * nv4 + c4], y);
          dot = fmaf(y.x, qv[j].x, dot);
          dot = fmaf(y.y, qv[j].y, dot);
          dot = fmaf(y.z, qv[j].z, dot);
          dot = fmaf(y.w, qv[j].w, dot);
        }
      }
      dot = warp_sum(dot);
      if (lane == 0) h[(size_t)p * DV + a] = from_f32<TO>(dot * inv_den);
    }
  }
}

cudaError_t launch_step(const void *q, const void *k, const void *v, bool bf16, bool out_bf16,
                        const float *ig, const float *fg, float *C, float *n, float *m, void *h,
                        int P, int DQK, int DV, cudaStream_t stream, bool exp_fg) {
  if (P == 0) return cudaSuccess;
  const int ef = exp_fg ? 1 : 0;
  if (bf16) {
    if (out_bf16)
      step_kernel<__nv_bfloat16, __nv_bfloat16><<<P, kThreads, 0, stream>>>(
          (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, ig, fg, C, n,
          m, (__nv_bfloat16 *)h, DQK, DV, ef);
    else
      step_kernel<__nv_bfloat16, float><<<P, kThreads, 0, stream>>>(
          (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, ig, fg, C, n,
          m, (float *)h, DQK, DV, ef);
  } else {
    if (out_bf16)
      step_kernel<float, __nv_bfloat16><<<P, kThreads, 0, stream>>>(
          (const float *)q, (const float *)k, (const float *)v, ig, fg, C, n, m, (__nv_bfloat16 *)h,
          DQK, DV, ef);
    else
      step_kernel<float, float><<<P, kThreads, 0, stream>>>((const float *)q, (const float *)k,
                                                            (const float *)v, ig, fg, C, n, m,
                                                            (float *)h, DQK, DV, ef);
  }
  return cudaGetLastError();
}

}  // namespace mlstm
