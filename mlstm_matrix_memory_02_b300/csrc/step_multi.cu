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
// warp carries two rows at a time through all T tokens in registers.  One CTA of 256 threads per
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

// BUTTERFLY: reduce the T dot products of the rows in flight together (worth it from T = 8 on;
// below that the per-dot warp sums are cheaper and the kernel needs fewer registers).  PL: float4
// columns of a row per lane (DQK / 128, rounded up); RIF: rows a warp carries at once -- every
// k_t, q_t read from shared memory feeds RIF rows.
template <typename T, typename TO, bool BUTTERFLY, int PL, int RIF>
__global__ void __launch_bounds__(kThreads) step_multi_kernel(
    const T *__restrict__ qin, const T *__restrict__ kin, const T *__restrict__ vin, const float *__restrict__ ig,
    const float *__restrict__ fg, float *__restrict__ C, float *__restrict__ n, float *__restrict__ m,
    TO *__restrict__ h, int NT, int DQK, int DV, int exp_fg) {
  static_assert(!BUTTERFLY || (RIF * kMaxT) % 32 == 0, "dot slots fill whole butterflies");
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

  // C rows: warp w carries rows w RIF .. w RIF + RIF - 1 (then the next 8 RIF rows) through the T
  // tokens; lane owns float4 columns lane + 32 j of each row.
  const int nv4 = DQK / 4;  // float4 per row (a multiple of 8)
  float4 *C4 = reinterpret_cast<float4 *>(C + (size_t)p * DV * DQK);
  const float4 *sq4 = reinterpret_cast<const float4 *>(sq);
  const float4 *sk4 = reinterpret_cast<const float4 *>(sk);
  // the rows of the next pass are requested before this pass's arithmetic
  auto load_rows = [&](int b0, float4 (&y)[RIF][PL]) {
#pragma unroll
    for (int i = 0; i < RIF; ++i) {
      const int a = b0 + i;
#pragma unroll
      for (int j = 0; j < PL; ++j) {
        const int c4 = lane + 32 * j;
        if (a < DV && c4 < nv4) y[i][j] = __ldcs(&C4[(size_t)a * nv4 + c4]);
        else y[i][j] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  };
  constexpr int kPass = (kThreads / 32) * RIF;  // rows per pass of the CTA
  float4 xn[RIF][PL];
  load_rows(warp * RIF, xn);
  for (int a0 = warp * RIF; a0 < DV; a0 += kPass) {
    float4 x[RIF][PL];
#pragma unroll
    for (int i = 0; i < RIF; ++i)
#pragma unroll
      for (int j = 0; j < PL; ++j) x[i][j] = xn[i][j];
    if (a0 + kPass < DV) load_rows(a0 + kPass, xn);
    if (BUTTERFLY) {
      // the RIF NT dot products of these rows (slot i kMaxT + t) are reduced together at the end,
      // 32 slots per butterfly
      float dots[RIF * kMaxT / 32][32];
#pragma unroll
      for (int b = 0; b < RIF * kMaxT / 32; ++b)
#pragma unroll
        for (int sl = 0; sl < 32; ++sl) dots[b][sl] = 0.f;
#pragma unroll
      for (int t = 0; t < kMaxT; ++t) {
        if (t < NT) {
          const float al = s_alpha[t];
          float4 kv[PL], qv[PL];
#pragma unroll
          for (int j = 0; j < PL; ++j) {
            const int c4 = lane + 32 * j;
            kv[j] = c4 < nv4 ? sk4[t * nv4 + c4] : make_float4(0.f, 0.f, 0.f, 0.f);
            qv[j] = c4 < nv4 ? sq4[t * nv4 + c4] : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int i = 0; i < RIF; ++i) {
            const int a = a0 + i;
            const float va = a < DV ? sv[t * DV + a] : 0.f;
            // four partial sums (one per float4 component): dependent chains of PL, not 4 PL
            float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
#pragma unroll
            for (int j = 0; j < PL; ++j) {
              float4 y = x[i][j];
              y.x = fmaf(al, y.x, va * kv[j].x);
              y.y = fmaf(al, y.y, va * kv[j].y);
              y.z = fmaf(al, y.z, va * kv[j].z);
              y.w = fmaf(al, y.w, va * kv[j].w);
              x[i][j] = y;
              d0 = fmaf(y.x, qv[j].x, d0);
              d1 = fmaf(y.y, qv[j].y, d1);
              d2 = fmaf(y.z, qv[j].z, d2);
              d3 = fmaf(y.w, qv[j].w, d3);
            }
            dots[(i * kMaxT + t) / 32][(i * kMaxT + t) % 32] = (d0 + d1) + (d2 + d3);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < RIF * kMaxT / 32; ++b) {
        const float tot = transpose_reduce32(dots[b], lane);
        const int slot = 32 * b + lane, i = slot / kMaxT, t = slot % kMaxT, a = a0 + i;
        if (t < NT && a < DV) h[((size_t)p * NT + t) * DV + a] = from_f32<TO>(tot * s_inv[t]);
      }
    } else {
      for (int t = 0; t < NT; ++t) {
        const float al = s_alpha[t], inv = s_inv[t];
        float4 kv[PL], qv[PL];
#pragma unroll
        for (int j = 0; j < PL; ++j) {
          const int c4 = lane + 32 * j;
          kv[j] = c4 < nv4 ? sk4[t * nv4 + c4] : make_float4(0.f, 0.f, 0.f, 0.f);
          qv[j] = c4 < nv4 ? sq4[t * nv4 + c4] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < RIF; ++i) {
          const int a = a0 + i;
          const float va = a < DV ? sv[t * DV + a] : 0.f;
          float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
#pragma unroll
          for (int j = 0; j < PL; ++j) {
            float4 y = x[i][j];
            y.x = fmaf(al, y.x, va * kv[j].x);
            y.y = fmaf(al, y.y, va * kv[j].y);
            y.z = fmaf(al, y.z, va * kv[j].z);
            y.w = fmaf(al, y.w, va * kv[j].w);
            x[i][j] = y;
            d0 = fmaf(y.x, qv[j].x, d0);
            d1 = fmaf(y.y, qv[j].y, d1);
            d2 = fmaf(y.z, qv[j].z, d2);
            d3 = fmaf(y.w, qv[j].w, d3);
          }
          const float dot = warp_sum((d0 + d1) + (d2 + d3));
          if (lane == 0 && a < DV) h[((size_t)p * NT + t) * DV + a] = from_f32<TO>(dot * inv);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < RIF; ++i) {
      const int a = a0 + i;
#pragma unroll
      for (int j = 0; j < PL; ++j) {
        const int c4 = lane + 32 * j;
        if (a < DV && c4 < nv4) __stcs(&C4[(size_t)a * nv4 + c4], x[i][j]);
      }
    }
  }
}

template <typename T, typename TO, bool BUTTERFLY, int RIF>
cudaError_t launch_step_multi_k(const void *q, const void *k, const void *v, const float *ig, const float *fg,
                                float *C, float *n, float *m, void *h, int P, int NT, int DQK, int DV,
                                cudaStream_t stream, bool exp_fg) {
  const int pl = (DQK / 4 + 31) / 32;
  auto kern = pl == 1   ? step_multi_kernel<T, TO, BUTTERFLY, 1, RIF>
              : pl == 2 ? step_multi_kernel<T, TO, BUTTERFLY, 2, RIF>
              : pl == 3 ? step_multi_kernel<T, TO, BUTTERFLY, 3, RIF>
                        : step_multi_kernel<T, TO, BUTTERFLY, 4, RIF>;
  const size_t smem = (size_t)NT * (2 * DQK + DV) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<P, kThreads, smem, stream>>>((const T *)q, (const T *)k, (const T *)v, ig, fg, C, n, m, (TO *)h, NT, DQK,
                                      DV, exp_fg ? 1 : 0);
  return cudaGetLastError();
}

template <typename T, typename TO>
cudaError_t launch_step_multi_t(const void *q, const void *k, const void *v, const float *ig, const float *fg,
                                float *C, float *n, float *m, void *h, int P, int NT, int DQK, int DV,
                                cudaStream_t stream, bool exp_fg) {
  if (NT >= 8)
    return launch_step_multi_k<T, TO, true, 2>(q, k, v, ig, fg, C, n, m, h, P, NT, DQK, DV, stream, exp_fg);
  return launch_step_multi_k<T, TO, false, 2>(q, k, v, ig, fg, C, n, m, h, P, NT, DQK, DV, stream, exp_fg);
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
