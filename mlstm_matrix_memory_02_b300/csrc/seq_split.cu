// seq_split.cu -- the sequence-parallel forward's two helper kernels.
//
// Page "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural Networks"
// (llms.blog), section 3 "The Parallel Dual Form" (the state after a stretch of tokens is the
// unrolled sum of their decayed contributions, so stretches compose by parallel associative
// scans) and section 2 (the max stabiliser, whose recurrence m_t = max(log f_t + m_{t-1}, i~_t)
// is max-plus linear in m_{t-1}).
//
// A head's sequence is cut into G segments of Sg tokens.  Run from the zero state with
// m = -inf, segment g yields its own map: the state (dC, dn) relative to its own stabiliser
// M_g, and B_g = sum of log f over its tokens.  Entering the segment with (C, n, m), the state
// after it is then exactly
//     m' = max(m + B_g, M_g)
//     C' = exp(m + B_g - m') C + exp(M_g - m') dC,   n' likewise,
// the unrolled recurrence split at the segment boundary (each term keeps its own decay).  A
// first pass computes every segment's map at once (gate preprocessing and the tensor-core state
// walk, no outputs; its segments may be finer than the second pass's, to fill the GPU), the scan
// below composes the maps from the initial state into the entering state of every second-pass
// segment and the final state, and the fused forward then runs those segments from their
// entering states.
#include "common.cuh"
#include "kernels.cuh"

namespace mlstm {
namespace {

// One block per (head, segment): B_g, and m = -inf as the first pass's entering stabiliser.
__global__ void seg_init_kernel(const float *__restrict__ fg, int exp_fg, int G, int Sg, float *__restrict__ min,
                                float *__restrict__ Bg) {
  const int pg = blockIdx.x;
  // B_g = sum of log f over the segment's tokens (double accumulation, tree reduction)
  double acc = 0.0;
  const float *f = fg + (size_t)pg * Sg;
  for (int t = threadIdx.x; t < Sg; t += blockDim.x) acc += (double)log_forget(f[t], exp_fg);
  __shared__ double red[32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double b = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) b += red[w];
    Bg[pg] = (float)b;
    min[pg] = -INFINITY;
  }
}

// Blocks over (head, range of C and n elements): the entering state of every R-th of the G
// first-pass segments (the second pass's segments, G / R per head), composed from the initial
// state (the caller's, or the zero state with m = 0) through the maps of the segments before
// it, and the final state.  Segment g's map: its own state (Cseg, nseg) and stabiliser M_g = the
// last entry of its chunk stabiliser chain (cm, NCg + 1 entries per segment), and B_g.  C_init
// may alias C_last (each element is read before it is written).
__global__ void seg_scan_kernel(int G, int R, int DQK, int DV, int NCg, const float *__restrict__ Bg,
                                const float *__restrict__ Cseg, const float *__restrict__ nseg,
                                const float *__restrict__ cm, const float *C_init, const float *n_init,
                                const float *m_init, float *__restrict__ Cin, float *__restrict__ nin,
                                float *__restrict__ min, float *C_last, float *n_last, float *m_last) {
  const int p = blockIdx.y;
  const size_t E = (size_t)DV * DQK;
  const size_t i4 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;  // float4 index over [C | n]
  const bool isC = i4 < E / 4;
  const bool isn = !isC && i4 < (E + DQK) / 4;
  float m = m_init ? m_init[p] : 0.f;
  float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
  if (isC && C_init) x = reinterpret_cast<const float4 *>(C_init + (size_t)p * E)[i4];
  if (isn && n_init) x = reinterpret_cast<const float4 *>(n_init + (size_t)p * DQK)[i4 - E / 4];
  for (int g = 0; g < G; ++g) {
    const size_t pg = (size_t)p * G + g;
    if (g % R == 0) {
      const size_t pe = (size_t)p * (G / R) + g / R;
      if (isC) reinterpret_cast<float4 *>(Cin + pe * E)[i4] = x;
      if (isn) reinterpret_cast<float4 *>(nin + pe * DQK)[i4 - E / 4] = x;
      if (i4 == 0) min[pe] = m;
    }
    const float Mg = cm[pg * (NCg + 1) + NCg], mb = m + Bg[pg];
    const float mn = fmaxf(mb, Mg);
    const float a = __expf(mb - mn), b = __expf(Mg - mn);
    float4 d = make_float4(0.f, 0.f, 0.f, 0.f);
    if (isC) d = reinterpret_cast<const float4 *>(Cseg + pg * E)[i4];
    if (isn) d = reinterpret_cast<const float4 *>(nseg + pg * DQK)[i4 - E / 4];
    x = make_float4(a * x.x + b * d.x, a * x.y + b * d.y, a * x.z + b * d.z, a * x.w + b * d.w);
    m = mn;
  }
  if (isC) reinterpret_cast<float4 *>(C_last + (size_t)p * E)[i4] = x;
  if (isn) reinterpret_cast<float4 *>(n_last + (size_t)p * DQK)[i4 - E / 4] = x;
  if (i4 == 0) m_last[p] = m;
}

}  // namespace

cudaError_t launch_seg_init(const float *fg, bool exp_fg, int P, int G, int Sg, float *min, float *Bg,
                            cudaStream_t stream) {
  seg_init_kernel<<<P * G, 256, 0, stream>>>(fg, exp_fg ? 1 : 0, G, Sg, min, Bg);
  return cudaGetLastError();
}

cudaError_t launch_seg_scan(int P, int G, int R, int DQK, int DV, int NCg, const float *Bg, const float *Cseg,
                            const float *nseg, const float *cm, const float *C_init, const float *n_init,
                            const float *m_init, float *Cin, float *nin, float *min, float *C_last, float *n_last,
                            float *m_last, cudaStream_t stream) {
  const size_t n4 = ((size_t)DV * DQK + DQK) / 4;
  dim3 grid((unsigned)((n4 + 255) / 256), (unsigned)P);
  seg_scan_kernel<<<grid, 256, 0, stream>>>(G, R, DQK, DV, NCg, Bg, Cseg, nseg, cm, C_init, n_init, m_init, Cin, nin,
                                            min, C_last, n_last, m_last);
  return cudaGetLastError();
}

}  // namespace mlstm
