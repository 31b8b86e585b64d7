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
// registers (d_v <= 512: at most 16 values per lane), lane-strided loads and stores so that
// every warp access covers 128 contiguous bytes (fp32) or 64 (bf16).  The mean and the centred
// variance are two warp reductions over the register copy (no second read of the row).
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.cuh"

namespace mlstm {

namespace {
constexpr int kRowsPerBlock = 8;  // warps per CTA, one row each
constexpr int kMaxPerLane = 16;   // d_v <= 512

__device__ __forceinline__ float load_any(const void *p, size_t i, int bf16) {
  return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]) : static_cast<const float *>(p)[i];
}
__device__ __forceinline__ void store_any(void *p, size_t i, float x, int bf16) {
  if (bf16) static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(x);
  else static_cast<float *>(p)[i] = x;
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
  const int per = DV / 32;
  const size_t base = (size_t)row * DV;
  float x[kMaxPerLane];
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxPerLane; ++j) {
    if (j < per) {
      x[j] = load_any(h, base + lane + 32 * j, h_bf16);
      sum += x[j];
    }
  }
  const float mu = warp_sum(sum) / (float)DV;
  float sq = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxPerLane; ++j) {
    if (j < per) {
      const float d = x[j] - mu;
      sq += d * d;
    }
  }
  const float var = warp_sum(sq) / (float)DV;
  const float rstd = rsqrtf(var + eps);
  const float *g = gamma + (size_t)head * DV, *b = beta + (size_t)head * DV;
#pragma unroll
  for (int j = 0; j < kMaxPerLane; ++j) {
    if (j < per) {
      const int c = lane + 32 * j;
      const float gate = 1.f / (1.f + __expf(-load_any(o_pre, base + c, o_bf16)));
      store_any(y, base + c, gate * fmaf(g[c], (x[j] - mu) * rstd, b[c]), y_bf16);
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
