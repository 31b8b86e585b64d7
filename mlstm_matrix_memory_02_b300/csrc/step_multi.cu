// step_multi.cu -- T consecutive recurrent decode steps of the mLSTM cell in one launch, in place.
//
// Page "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural Networks"
// (llms.blog): section 5 "Inference Memory and Throughput Trade-Offs" (decoding carries the
// constant-size state C, n per head), section 3 "Associative Matrix Cell State" (updates and
// retrieval, k scaled by 1/sqrt(d)) and section 2 (stabiliser).  For tokens t = 1..T in order:
//   m_t = max(log sigmoid(f~_t) + m_{t-1}, i~_t)
//   alpha_t = exp(log sigmoid(f~_t) + m_{t-1} - m_t),  w_t = exp(i~_t - m_t)
//   C_t = alpha_t C_{t-1} + w_t v_t khat_t^T,  n_t = alpha_t n_{t-1} + w_t khat_t
//   h_t = C_t q_t / max(|n_t . q_t|, exp(-m_t))
// exactly as T single steps, but the state (2 * DV * DQK * 4 bytes per head) crosses HBM once
// for the T tokens instead of T times: row a of C_t depends only on row a of C_{t-1}, so each
// warp carries its rows through all T tokens in registers.  One CTA of 256 threads per
// (batch, head); the scalar gate chain, the n chain and the T denominators are formed first.
#include "common.cuh"
#include "kernels.cuh"

namespace mlstm {

namespace {
constexpr int kThreads = 256;
constexpr int kMaxT = 16;
}  // namespace

// Reduces 32 per-lane partial sums at once: afterwards lane l holds slot l summed over the
// warp (five butterfly stages, 31 shuffles, instead of 5 shuffles per slot).
__device__ __forceinline__ float transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const bool up = lane & 16;
    const float send = up ? v[i] : v[i + 16], keep = up ? v[i + 16] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool up = lane & 8;
    const float send = up ? v[i] : v[i + 8], keep = up ? v[i + 8] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool up = lane & 4;
    const float send = up ? v[i] : v[i + 4], keep = up ? v[i + 4] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool up = lane & 2;
    const float send = up ? v[i] : v[i + 2], keep = up ? v[i + 2] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  {
    const bool up = lane & 1;
    const float send = up ? v[0] : v[1], keep = up ? v[1] : v[0];
    v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
  }
  return v[0];
}

// BUTTERFLY: reduce the 2 T dot products of a row pair together (worth it from T = 8 on; below
// that the per-dot warp sums are cheaper and the kernel needs half the registers).
template <typename T, typename TO, bool BUTTERFLY>
__global__ void __launch_bounds__(kThreads) step_multi_kernel(
    const T *__restrict__ qin, const T *__restrict__ kin, const T *__restrict__ vin, const float *__restrict__ ig,
    const float *__restrict__ fg, float *__restrict__ C, float *__restrict__ n, float *__restrict__ m,
    TO *__restrict__ h, int NT, int DQK, int DV, int exp_fg) {
  extern __shared__ __align__(16) float dsm[];
  float *sq = dsm;                // [NT][DQK]  q_t
  float *sk = dsm + NT * DQK;     // [NT][DQK]  w_t khat_t
  float *sv = dsm + 2 * NT * DQK; // [NT][DV]   v_t
  __shared__ float s_alpha[kMaxT], s_w[kMaxT], s_floor[kMaxT], s_inv[kMaxT];
  __shared__ float s_part[kMaxT][kThreads / 32];

  const int p = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float scale = rsqrtf((float)DQK);

  // gate chain over the T tokens
  if (tid == 0) {
    float mm = m[p];
    for (int t = 0; t < NT; ++t) {
      const float lf = log_forget(fg[(size_t)p * NT + t], exp_fg);
      const float it = ig[(size_t)p * NT + t];
      const float mn = fmaxf(lf + mm, it);
      s_alpha[t] = expf(lf + mm - mn);
      s_w[t] = expf(it - mn);
      s_floor[t] = expf(-mn);
      mm = mn;
    }
    m[p] = mm;
  }
  __syncthreads();
  for (int i = tid; i < NT * DQK; i += kThreads) {
    const int t = i / DQK;
    sq[i] = to_f32(qin[(size_t)p * NT * DQK + i]);
    sk[i] = to_f32(kin[(size_t)p * NT * DQK + i]) * scale * s_w[t];
  }
  for (int i = tid; i < NT * DV; i += kThreads) sv[i] = to_f32(vin[(size_t)p * NT * DV + i]);
  __syncthreads();

  // n chain and the dots n_t . q_t (each thread owns columns tid, tid + 256)
  float part[kMaxT];
#pragma unroll
  for (int t = 0; t < kMaxT; ++t) part[t] = 0.f;
  for (int c = tid; c < DQK; c += kThreads) {
    float nn = n[(size_t)p * DQK + c];
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) {
      if (t < NT) {
        nn = fmaf(s_alpha[t], nn, sk[t * DQK + c]);
        part[t] = fmaf(nn, sq[t * DQK + c], part[t]);
      }
    }
    n[(size_t)p * DQK + c] = nn;
  }
#pragma unroll
  for (int t = 0; t < kMaxT; ++t) {
    if (t < NT) {
      const float x = warp_sum(part[t]);
      if (lane == 0) s_part[t][warp] = x;
    }
  }
  __syncthreads();
  if (tid < NT) {
    float x = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) x += s_part[tid][w];
    s_inv[tid] = 1.f / fmaxf(fabsf(x), s_floor[tid]);
  }
  __syncthreads();

  // C rows: warp w carries rows w, w + 8, ... through the T tokens; lane owns float4 columns
  // lane + 32 j of the row.
  const int nv4 = DQK / 4;               // float4 per row (a multiple of 8)
  const int per_lane = (nv4 + 31) / 32;  // 1..4
  float4 *C4 = reinterpret_cast<float4 *>(C + (size_t)p * DV * DQK);
  const float4 *sq4 = reinterpret_cast<const float4 *>(sq);
  const float4 *sk4 = reinterpret_cast<const float4 *>(sk);
  constexpr int kRowsInFlight = 2;
  for (int a0 = warp * kRowsInFlight; a0 < DV; a0 += (kThreads / 32) * kRowsInFlight) {
    float4 x[kRowsInFlight][4];
#pragma unroll
    for (int i = 0; i < kRowsInFlight; ++i) {
      const int a = a0 + i;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c4 = lane + 32 * j;
        if (a < DV && j < per_lane && c4 < nv4) x[i][j] = __ldcs(&C4[(size_t)a * nv4 + c4]);
        else x[i][j] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (BUTTERFLY) {
      // the 2 NT dot products of this row pair (slot i NT + t) are reduced together at the end
      float dots[32];
#pragma unroll
      for (int sl = 0; sl < 32; ++sl) dots[sl] = 0.f;
#pragma unroll
      for (int t = 0; t < kMaxT; ++t) {
        if (t < NT) {
          const float al = s_alpha[t];
#pragma unroll
          for (int i = 0; i < kRowsInFlight; ++i) {
            const int a = a0 + i;
            const float va = a < DV ? sv[t * DV + a] : 0.f;
            float dot = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int c4 = lane + 32 * j;
              if (j < per_lane && c4 < nv4) {
                const float4 kv = sk4[t * nv4 + c4], qv = sq4[t * nv4 + c4];
                float4 y = x[i][j];
                y.x = fmaf(al, y.x, va * kv.x);
                y.y = fmaf(al, y.y, va * kv.y);
                y.z = fmaf(al, y.z, va * kv.z);
                y.w = fmaf(al, y.w, va * kv.w);
                x[i][j] = y;
                dot = fmaf(y.x, qv.x, dot);
                dot = fmaf(y.y, qv.y, dot);
                dot = fmaf(y.z, qv.z, dot);
                dot = fmaf(y.w, qv.w, dot);
              }
            }
            dots[i * kMaxT + t] = dot;
          }
        }
      }
      const float tot = transpose_reduce32(dots, lane);
      const int i = lane / kMaxT, t = lane % kMaxT, a = a0 + i;
      if (t < NT && a < DV) h[((size_t)p * NT + t) * DV + a] = from_f32<TO>(tot * s_inv[t]);
    } else {
      for (int t = 0; t < NT; ++t) {
        const float al = s_alpha[t], inv = s_inv[t];
#pragma unroll
        for (int i = 0; i < kRowsInFlight; ++i) {
          const int a = a0 + i;
          if (a >= DV) break;
          const float va = sv[t * DV + a];
          float dot = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int c4 = lane + 32 * j;
            if (j < per_lane && c4 < nv4) {
              const float4 kv = sk4[t * nv4 + c4], qv = sq4[t * nv4 + c4];
              float4 y = x[i][j];
              y.x = fmaf(al, y.x, va * kv.x);
              y.y = fmaf(al, y.y, va * kv.y);
              y.z = fmaf(al, y.z, va * kv.z);
              y.w = fmaf(al, y.w, va * kv.w);
              x[i][j] = y;
              dot = fmaf(y.x, qv.x, dot);
              dot = fmaf(y.y, qv.y, dot);
              dot = fmaf(y.z, qv.z, dot);
              dot = fmaf(y.w, qv.w, dot);
            }
          }
          dot = warp_sum(dot);
          if (lane == 0) h[((size_t)p * NT + t) * DV + a] = from_f32<TO>(dot * inv);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kRowsInFlight; ++i) {
      const int a = a0 + i;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c4 = lane + 32 * j;
        if (a < DV && j < per_lane && c4 < nv4) __stcs(&C4[(size_t)a * nv4 + c4], x[i][j]);
      }
    }
  }
}

template <typename T, typename TO>
cudaError_t launch_step_multi_t(const void *q, const void *k, const void *v, const float *ig, const float *fg,
                                float *C, float *n, float *m, void *h, int P, int NT, int DQK, int DV,
                                cudaStream_t stream, bool exp_fg) {
  auto kern = NT >= 8 ? step_multi_kernel<T, TO, true> : step_multi_kernel<T, TO, false>;
  const size_t smem = (size_t)NT * (2 * DQK + DV) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<P, kThreads, smem, stream>>>((const T *)q, (const T *)k, (const T *)v, ig, fg, C, n, m, (TO *)h, NT, DQK,
                                      DV, exp_fg ? 1 : 0);
  return cudaGetLastError();
}

int step_multi_max_tokens() { return kMaxT; }

cudaError_t launch_step_multi(const void *q, const void *k, const void *v, bool bf16, bool out_bf16,
                              const float *ig, const float *fg, float *C, float *n, float *m, void *h, int P,
                              int NT, int DQK, int DV, cudaStream_t stream, bool exp_fg) {
  if (P == 0 || NT == 0) return cudaSuccess;
  if (bf16)
    return out_bf16 ? launch_step_multi_t<__nv_bfloat16, __nv_bfloat16>(q, k, v, ig, fg, C, n, m, h, P, NT, DQK, DV,
                                                                         stream, exp_fg)
                    : launch_step_multi_t<__nv_bfloat16, float>(q, k, v, ig, fg, C, n, m, h, P, NT, DQK, DV, stream,
                                                               exp_fg);
  return out_bf16 ? launch_step_multi_t<float, __nv_bfloat16>(q, k, v, ig, fg, C, n, m, h, P, NT, DQK, DV, stream,
                                                               exp_fg)
                  : launch_step_multi_t<float, float>(q, k, v, ig, fg, C, n, m, h, P, NT, DQK, DV, stream, exp_fg);
}

}  // namespace mlstm
