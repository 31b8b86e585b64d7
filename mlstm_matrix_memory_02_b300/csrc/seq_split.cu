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
// the unrolled recurrence split at the segment boundary (each term keeps its own decay).  The
// first pass runs every segment at once (segment 0 from the true initial state), the scan below
// composes the maps into every segment's true entering state, and a second pass recomputes
// segments 1..G-1 from those states.
#include "common.cuh"
#include "kernels.cuh"

namespace mlstm {
namespace {

// One block per (head, segment): the entering state of the first pass and B_g.
__global__ void seg_init_kernel(const float *__restrict__ C_init, const float *__restrict__ n_init,
                                const float *__restrict__ m_init, const float *__restrict__ fg, int exp_fg, int G,
                                int Sg, int DQK, int DV, float *__restrict__ Cin, float *__restrict__ nin,
                                float *__restrict__ min, float *__restrict__ Bg) {
  const int pg = blockIdx.x, p = pg / G, g = pg % G;
  const size_t E = (size_t)DV * DQK;
  float4 *C4 = reinterpret_cast<float4 *>(Cin + (size_t)pg * E);
  float4 *n4 = reinterpret_cast<float4 *>(nin + (size_t)pg * DQK);
  if (g == 0 && C_init != nullptr) {
    const float4 *src = reinterpret_cast<const float4 *>(C_init + (size_t)p * E);
    for (size_t i = threadIdx.x; i < E / 4; i += blockDim.x) C4[i] = src[i];
    const float4 *ns = reinterpret_cast<const float4 *>(n_init + (size_t)p * DQK);
    for (int i = threadIdx.x; i < DQK / 4; i += blockDim.x) n4[i] = ns[i];
  } else {
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (size_t i = threadIdx.x; i < E / 4; i += blockDim.x) C4[i] = z;
    for (int i = threadIdx.x; i < DQK / 4; i += blockDim.x) n4[i] = z;
  }
  // B_g = sum of log f over the segment's tokens (double accumulation, tree reduction)
  double acc = 0.0;
  const float *f = fg + ((size_t)p * G + g) * Sg;
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
    min[pg] = g == 0 ? (m_init ? m_init[p] : 0.f) : -INFINITY;
  }
}

// Blocks over (head, range of C and n elements): every segment's entering state and the final state.
__global__ void seg_scan_kernel(int G, int DQK, int DV, const float *__restrict__ Bg, const float *__restrict__ Cseg,
                                const float *__restrict__ nseg, const float *__restrict__ mseg, float *__restrict__ Cin,
                                float *__restrict__ nin, float *__restrict__ min, float *__restrict__ C_last,
                                float *__restrict__ n_last, float *__restrict__ m_last) {
  const int p = blockIdx.y;
  const size_t E = (size_t)DV * DQK;
  const size_t i4 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;  // float4 index over [C | n]
  const bool isC = i4 < E / 4;
  const bool isn = !isC && i4 < (E + DQK) / 4;
  // the stabiliser chain across the segments (every thread, G is small)
  float m = mseg[(size_t)p * G];
  float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
  if (isC) x = reinterpret_cast<const float4 *>(Cseg + (size_t)p * G * E)[i4];
  if (isn) x = reinterpret_cast<const float4 *>(nseg + (size_t)p * G * DQK)[i4 - E / 4];
  for (int g = 1; g < G; ++g) {
    const size_t pg = (size_t)p * G + g;
    if (isC) reinterpret_cast<float4 *>(Cin + pg * E)[i4] = x;
    if (isn) reinterpret_cast<float4 *>(nin + pg * DQK)[i4 - E / 4] = x;
    if (i4 == 0) min[pg] = m;
    const float Mg = mseg[pg], mb = m + Bg[pg];
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

cudaError_t launch_seg_init(const float *C_init, const float *n_init, const float *m_init, const float *fg,
                            bool exp_fg, int P, int G, int Sg, int DQK, int DV, float *Cin, float *nin, float *min,
                            float *Bg, cudaStream_t stream) {
  seg_init_kernel<<<P * G, 256, 0, stream>>>(C_init, n_init, m_init, fg, exp_fg ? 1 : 0, G, Sg, DQK, DV, Cin, nin,
                                             min, Bg);
  return cudaGetLastError();
}

cudaError_t launch_seg_scan(int P, int G, int DQK, int DV, const float *Bg, const float *Cseg, const float *nseg,
                            const float *mseg, float *Cin, float *nin, float *min, float *C_last, float *n_last,
                            float *m_last, cudaStream_t stream) {
  const size_t n4 = ((size_t)DV * DQK + DQK) / 4;
  dim3 grid((unsigned)((n4 + 255) / 256), (unsigned)P);
  seg_scan_kernel<<<grid, 256, 0, stream>>>(G, DQK, DV, Bg, Cseg, nseg, mseg, Cin, nin, min, C_last, n_last, m_last);
  return cudaGetLastError();
}

}  // namespace mlstm
