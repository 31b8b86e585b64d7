// groupnorm_gate.cu -- the mLSTM block's step after the cell: per-head group normalisation of
// the cell output and the output gate, one pass over HBM.
//
// Page "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural Networks"
// (llms.blog): section 4 "xLSTM Block Architecture and Residual Stacking", the mLSTM block's
// item 5 "Group Normalization and Output Gating" (output heads normalised, then modulated by the
// output gate), and section 3 "Associative Matrix Cell State" (h_t = o_t (.) h~_t).  For every
// (batch, head, token) row of d_v channels:
//   mu = mean_c h~_c,  var = mean_c (h~_c - mu)^2,
//   y_c = sigmoid(o~_c) * (gamma_c (h~_c - mu) / sqrt(var + eps) + beta_c)
// with gamma, beta per (head, channel).  Memory bound: one warp per row, the row held in
// registers.  A lane owns chunks of 8 consecutive channels (chunk lane + 32 j), read and written
// with 16-byte accesses (two for fp32 data); h and o~ of the row are both requested before any
// arithmetic, so each warp has its whole row in flight at once.  The mean and the centred
// variance are two warp reductions over the register copy (no second read of the row).
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.cuh"

namespace mlstm {

namespace {
constexpr int kRowsPerBlock = 8;  // warps per CTA, one row each
constexpr int kMaxChunks = 2;     // 8-channel chunks per lane: d_v <= 512

// 8 consecutive values starting at element i (16-byte aligned) as fp32
__device__ __forceinline__ void load8(const void *p, size_t i, int bf16, float (&x)[8]) {
  if (bf16) {
    const uint4 u = *reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p) + i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = __uint_as_float(w[e] << 16);
      x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
  } else {
    const float4 a = *reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i);
    const float4 b = *reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}
__device__ __forceinline__ void store8(void *p, size_t i, int bf16, const float (&x)[8]) {
  if (bf16) {
    uint4 u;
    uint32_t *w = &u.x;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 v = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
      w[e] = *reinterpret_cast<const uint32_t *>(&v);
    }
    *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p) + i) = u;
  } else {
    *reinterpret_cast<float4 *>(static_cast<float *>(p) + i) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4 *>(static_cast<float *>(p) + i + 4) = make_float4(x[4], x[5], x[6], x[7]);
  }
}
}  // namespace

__global__ void __launch_bounds__(32 * kRowsPerBlock) groupnorm_gate_kernel(
    const void *h, const void *__restrict__ o_pre, const float *__restrict__ gamma,
    const float *__restrict__ beta, float eps, void *y, long long rows, int NH, int S, int DV, int h_bf16,
    int o_bf16, int y_bf16) {
  const long long row = (long long)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const int head = (int)((row / S) % NH);
  const int nchunks = DV / 8;
  const size_t base = (size_t)row * DV;
  float x[kMaxChunks][8], o[kMaxChunks][8];
#pragma unroll
  for (int j = 0; j < kMaxChunks; ++j) {
    const int ci = lane + 32 * j;
    if (ci < nchunks) {
      load8(h, base + 8 * ci, h_bf16, x[j]);
      load8(o_pre, base + 8 * ci, o_bf16, o[j]);
    }
  }
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxChunks; ++j)
    if (lane + 32 * j < nchunks)
#pragma unroll
      for (int e = 0; e < 8; ++e) sum += x[j][e];
  const float mu = warp_sum(sum) / (float)DV;
  float sq = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxChunks; ++j)
    if (lane + 32 * j < nchunks)
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float d = x[j][e] - mu;
        sq += d * d;
      }
  const float var = warp_sum(sq) / (float)DV;
  const float rstd = rsqrtf(var + eps);
  const float *g = gamma + (size_t)head * DV, *b = beta + (size_t)head * DV;
#pragma unroll
  for (int j = 0; j < kMaxChunks; ++j) {
    const int ci = lane + 32 * j;
    if (ci < nchunks) {
      const float4 g0 = *reinterpret_cast<const float4 *>(g + 8 * ci), g1 = *reinterpret_cast<const float4 *>(g + 8 * ci + 4);
      const float4 b0 = *reinterpret_cast<const float4 *>(b + 8 * ci), b1 = *reinterpret_cast<const float4 *>(b + 8 * ci + 4);
      const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
      float out[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float gate = 1.f / (1.f + __expf(-o[j][e]));
        out[e] = gate * fmaf(gg[e], (x[j][e] - mu) * rstd, bb[e]);
      }
      store8(y, base + 8 * ci, y_bf16, out);
    }
  }
}

cudaError_t launch_groupnorm_gate(const void *h, bool h_bf16, const void *o_pre, bool o_bf16, const float *gamma,
                                  const float *beta, float eps, void *y, bool y_bf16, int B, int NH, int S, int DV,
                                  cudaStream_t stream) {
  const long long rows = (long long)B * NH * S;
  if (rows == 0) return cudaSuccess;
  const long long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  groupnorm_gate_kernel<<<(unsigned)blocks, 32 * kRowsPerBlock, 0, stream>>>(
      h, o_pre, gamma, beta, eps, y, rows, NH, S, DV, h_bf16 ? 1 : 0, o_bf16 ? 1 : 0, y_bf16 ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace mlstm
