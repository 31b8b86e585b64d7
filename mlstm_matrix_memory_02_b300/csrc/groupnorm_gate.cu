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
// with gamma, beta per (head, channel).  Memory bound: a warp per row at a time, rows streamed
// into shared memory several rows ahead.  A lane owns chunks of 8 consecutive channels (chunk
// lane + 32 j), copied in and written out with 16-byte accesses (two for fp32 data).  The mean
// and the centred variance are two warp reductions over the lane's register copy (no second
// read of the row).
#include <cuda_bf16.h>

#include <atomic>

#include "common.cuh"
#include "kernels.cuh"

namespace mlstm {

namespace {
constexpr int kRowsPerBlock = 8;  // warps per CTA
constexpr int kMaxChunks = 2;     // 8-channel chunks per lane: d_v <= 512

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

// One row's group norm and gate from its register copy (x = h~, o = o~), stored to y.
template <int NCH>
__device__ __forceinline__ void finish_row(const float (&x)[NCH][8], const float (&o)[NCH][8], int lane, int nchunks,
                                           int DV, float eps, const float *g, const float *b, void *y, size_t base,
                                           int y_bf16) {
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < NCH; ++j)
    if (lane + 32 * j < nchunks)
#pragma unroll
      for (int e = 0; e < 8; ++e) sum += x[j][e];
  const float mu = warp_sum(sum) / (float)DV;
  float sq = 0.f;
#pragma unroll
  for (int j = 0; j < NCH; ++j)
    if (lane + 32 * j < nchunks)
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float d = x[j][e] - mu;
        sq += d * d;
      }
  const float var = warp_sum(sq) / (float)DV;
  const float rstd = rsqrtf(var + eps);
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int ci = lane + 32 * j;
    if (ci < nchunks) {
      const float4 g0 = *reinterpret_cast<const float4 *>(g + 8 * ci), g1 = *reinterpret_cast<const float4 *>(g + 8 * ci + 4);
      const float4 b0 = *reinterpret_cast<const float4 *>(b + 8 * ci), b1 = *reinterpret_cast<const float4 *>(b + 8 * ci + 4);
      const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
      float out[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float gate = __fdividef(1.f, 1.f + __expf(-o[j][e]));  // fast divide: 2 ulp
        out[e] = gate * fmaf(gg[e], (x[j][e] - mu) * rstd, bb[e]);
      }
      store8(y, base + 8 * ci, y_bf16, out);
    }
  }
}

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// 8 consecutive values at byte offset `off` of a shared-memory row, as fp32
__device__ __forceinline__ void smem8(const unsigned char *row, size_t off, int bf16, float (&x)[8]) {
  if (bf16) {
    const uint4 u = *reinterpret_cast<const uint4 *>(row + off);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = __uint_as_float(w[e] << 16);
      x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
  } else {
    const float4 a = *reinterpret_cast<const float4 *>(row + off);
    const float4 b = *reinterpret_cast<const float4 *>(row + off + 16);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

constexpr int kStages = 2;  // row buffers per warp: the row being reduced and the next one in flight

// A grid of as many CTAs as fit on each SM.  Each warp walks rows with a stride of all warps and streams
// them through a private ring of kStages row buffers in shared memory with 16-byte cp.async
// copies, kStages - 1 rows ahead of the one it reduces.
template <int NCH>
__global__ void __launch_bounds__(32 * kRowsPerBlock) groupnorm_gate_kernel(
    const void *h, const void *__restrict__ o_pre, const float *__restrict__ gamma,
    const float *__restrict__ beta, float eps, void *y, long long rows, int NH, int S, int DV, int h_bf16,
    int o_bf16, int y_bf16) {
  extern __shared__ __align__(16) unsigned char gn_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int hb = h_bf16 ? 2 : 4, ob = o_bf16 ? 2 : 4;
  const size_t hrow = (size_t)DV * hb, stage = hrow + (size_t)DV * ob;
  unsigned char *ring = gn_smem + (size_t)warp * kStages * stage;
  const long long stride = (long long)gridDim.x * kRowsPerBlock;
  const long long first = (long long)blockIdx.x * kRowsPerBlock + warp;
  const int nchunks = DV / 8;
  // Copies are made in 16-byte pieces, lane l taking pieces l, l + 32, ... of the row's h~ and o~
  // (each warp instruction covers 512 contiguous bytes); rows past the end still commit an
  // (empty) group, so that the group count stays uniform.
  const int hpieces = (int)(hrow / 16), opieces = (int)((size_t)DV * ob / 16);
  auto issue = [&](long long r, int slot) {
    if (r < rows) {
      unsigned char *sh = ring + (size_t)slot * stage, *so = sh + hrow;
      const unsigned char *gh = static_cast<const unsigned char *>(h) + (size_t)r * hrow;
      const unsigned char *go = static_cast<const unsigned char *>(o_pre) + (size_t)r * DV * ob;
      for (int i = lane; i < hpieces; i += 32) cp_async16(sh + 16 * i, gh + 16 * i);
      for (int i = lane; i < opieces; i += 32) cp_async16(so + 16 * i, go + 16 * i);
    }
    cp_async_commit();
  };
#pragma unroll
  for (int st = 0; st < kStages - 1; ++st) issue(first + st * stride, st);
  int slot = 0;
  for (long long row = first; row < rows; row += stride) {
    issue(row + (kStages - 1) * stride, (slot + kStages - 1) % kStages);
    cp_async_wait<kStages - 1>();  // this lane's copies of the row have landed ...
    __syncwarp();                  // ... and every other lane's
    const unsigned char *sh = ring + (size_t)slot * stage, *so = sh + hrow;
    float x[NCH][8], o[NCH][8];
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int ci = lane + 32 * j;
      if (ci < nchunks) {
        smem8(sh, (size_t)8 * ci * hb, h_bf16, x[j]);
        smem8(so, (size_t)8 * ci * ob, o_bf16, o[j]);
      }
    }
    const int head = (int)((row / S) % NH);
    finish_row<NCH>(x, o, lane, nchunks, DV, eps, gamma + (size_t)head * DV, beta + (size_t)head * DV, y,
                    (size_t)row * DV, y_bf16);
    __syncwarp();  // every lane has read the slot before any lane refills it
    slot = (slot + 1) % kStages;
  }
  cp_async_wait<0>();
}

namespace {
constexpr size_t kMaxSmem = (size_t)kRowsPerBlock * kStages * 512 * 8;  // d_v = 512, fp32 h~ and o~

// CTAs per SM for each (chunks per lane, shared-memory size in 4 KB units), found once per process
std::atomic<int> g_per_sm[kMaxChunks][kMaxSmem / 4096 + 1];
std::atomic<bool> g_attr_set[kMaxChunks];
}  // namespace

cudaError_t launch_groupnorm_gate(const void *h, bool h_bf16, const void *o_pre, bool o_bf16, const float *gamma,
                                  const float *beta, float eps, void *y, bool y_bf16, int B, int NH, int S, int DV,
                                  cudaStream_t stream) {
  const long long rows = (long long)B * NH * S;
  if (rows == 0) return cudaSuccess;
  const int nch = DV <= 256 ? 1 : kMaxChunks;
  auto kern = nch == 1 ? groupnorm_gate_kernel<1> : groupnorm_gate_kernel<kMaxChunks>;
  const size_t smem = (size_t)kRowsPerBlock * kStages * DV * ((h_bf16 ? 2 : 4) + (o_bf16 ? 2 : 4));
  if (!g_attr_set[nch - 1].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem);
    if (e != cudaSuccess) return e;
    g_attr_set[nch - 1].store(true, std::memory_order_release);
  }
  std::atomic<int> &slot = g_per_sm[nch - 1][smem / 4096];
  int per_sm = slot.load(std::memory_order_relaxed);
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * kRowsPerBlock, smem) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    slot.store(per_sm, std::memory_order_relaxed);
  }
  const long long need = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  const long long cap = (long long)sm_count() * per_sm;
  const long long blocks = need < cap ? need : cap;
  kern<<<(unsigned)blocks, 32 * kRowsPerBlock, smem, stream>>>(h, o_pre, gamma, beta, eps, y, rows, NH, S, DV,
                                                               h_bf16 ? 1 : 0, o_bf16 ? 1 : 0, y_bf16 ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace mlstm
