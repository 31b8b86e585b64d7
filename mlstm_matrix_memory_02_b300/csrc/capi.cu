// capi.cu -- the extern "C" boundary of the mLSTM library: argument checks, workspace
// layout and kernel launches.  Declarations and their contracts are in include/mlstm.h.
#include <stdint.h>

#include "../../include/mlstm.h"
#include "common.cuh"
#include "kernels.cuh"

namespace mlstm {

__global__ void copy_chunk_m_kernel(const float *__restrict__ cm, int P, int NC, float *__restrict__ m_last) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p < P) m_last[p] = cm[(size_t)p * (NC + 1) + NC];
}

cudaError_t launch_copy_chunk_m(const float *cm, int P, int NC, float *m_last, cudaStream_t stream) {
  if (P == 0) return cudaSuccess;
  copy_chunk_m_kernel<<<(P + 255) / 256, 256, 0, stream>>>(cm, P, NC, m_last);
  return cudaGetLastError();
}

namespace {

constexpr size_t kAlign = 256;
constexpr int kTcChunk = 64;  // the fused tensor-core kernel's chunk
constexpr int kMaxPairs = 65535;  // grid.z limit of the output kernel

inline size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Layout {
  size_t err, gb, gx, gu, cm, Cs, ns, ncopy, gates_end, total;
  // the sequence-parallel forward's buffers (G segments per head, the fused path only), after
  // `total`: per (head, segment) the sum of log f, the segment's own state and stabiliser, and
  // its entering state
  size_t Bg, Cseg, nseg, mseg, Cin, nin, min, m1, cmseg, wx, wn;
  // the three-kernel forward's buffers (per-chunk operands prepared ahead of the state walk)
  size_t qb, kw, pm, pden, pinv, pdn, ptok4, ptok2, pcdat;
  size_t split_total;  // the end of the optional buffers: the size mlstm_fwd_workspace_bytes reports
  int G, G1, Ls;  // segments per head (second pass, first pass); the first pass's chunk
  bool tc;  // the forward runs on the fused tensor-core kernel (no materialised states)
  bool pre;  // the sizes suit the three-kernel forward (used when the workspace holds its buffers)
};

// The three-kernel forward (pre-pass, n chain, state walk) instead of the single fused kernel:
// for heads split over a CTA pair, where the per-chunk work it does once per head would
// otherwise be repeated by each d_v tile, and for sequences of at most 64 chunks of 64 tokens.
bool use_prepass(int P, int S, int DQK, int DV) {
  return fwd_prep_supported(S, DQK) && fwd_tc_pair(P, DQK, DV);
}

bool use_tc(int B, int NH, int S, int DQK, int DV, int chunk, mlstm_dtype dt) {
  return fwd_tc_supported(S, chunk, DQK, DV, dt == MLSTM_BF16) && (long long)B * NH * S < (1LL << 31);
}

bool sizes_ok(int B, int NH, int S, int DQK, int DV, int chunk) {
  if (B < 1 || NH < 1 || S < 0) return false;
  if ((long long)B * NH > kMaxPairs) return false;
  if (chunk != 16 && chunk != 32 && chunk != 64 && chunk != 128) return false;
  if (S % chunk != 0) return false;
  if (DQK < 32 || DQK > 512 || DQK % 32 != 0) return false;
  if (DV < 32 || DV > 512 || DV % 32 != 0) return false;
  if ((long long)B * NH * S > (1LL << 40)) return false;
  return true;
}

// Workspace layout for the kernels of one chunk size.  The wait-error word of the kernels with
// bounded waits sits at offset 0 of every layout, so that mlstm_fwd_check finds it whatever path
// or chunk a forward took.
Layout layout(int B, int NH, int S, int DQK, int DV, int chunk, mlstm_dtype dt) {
  const size_t P = (size_t)B * NH, NC = (size_t)S / chunk;
  Layout L{};
  L.tc = use_tc(B, NH, S, DQK, DV, chunk, dt);
  size_t off = 0;
  L.err = off; off = round_up(off + sizeof(int));
  L.gb = off; off = round_up(off + P * S * sizeof(float));
  L.gx = off; off = round_up(off + P * S * sizeof(float));
  L.gu = off; off = round_up(off + P * S * sizeof(float));
  L.cm = off; off = round_up(off + P * (NC + 1) * sizeof(float));
  L.gates_end = off;
  const size_t states = L.tc ? 0 : P * (NC + 1);
  L.Cs = off; off = round_up(off + states * DV * DQK * sizeof(float));
  L.ns = off; off = round_up(off + states * DQK * sizeof(float));
  // tensor-core path: a copy of n_init (every d_v tile reads it; one of them writes n_last,
  // which may alias n_init)
  L.ncopy = off; off = round_up(off + (L.tc ? P * DQK : 0) * sizeof(float));
  L.total = off;
  L.G = L.tc && S > 0 && states_tc_supported(64, DQK, DV, true) ? fwd_tc_segments((int)P, S, DQK, DV) : 1;
  const size_t PG = L.G > 1 ? P * L.G : 0;
  // the first pass (states only) fills the GPU with finer segments where that keeps at least
  // 128 tokens a segment
  L.G1 = L.G;
  if (L.G > 1) {
    const long long ctas = (long long)P * (DV / 128);
    while (ctas * 2 * L.G1 <= sm_count() && S % (64 * 2 * L.G1) == 0 && S / (2 * L.G1) >= 128) L.G1 *= 2;
  }
  const size_t PG1 = L.G > 1 ? P * L.G1 : 0;
  L.Ls = L.G > 1 && (S / L.G1) % 128 == 0 ? 128 : 64;
  const size_t PS1 = L.G > 1 ? P * (size_t)S : 0, NC1 = L.G > 1 ? PS1 / L.Ls : 0;
  L.Bg = off; off = round_up(off + PG1 * sizeof(float));
  L.Cseg = off; off = round_up(off + PG1 * DV * DQK * sizeof(float));
  L.nseg = off; off = round_up(off + PG1 * DQK * sizeof(float));
  L.mseg = off; off = round_up(off + PG * sizeof(float));
  L.Cin = off; off = round_up(off + PG * DV * DQK * sizeof(float));
  L.nin = off; off = round_up(off + PG * DQK * sizeof(float));
  L.min = off; off = round_up(off + PG * sizeof(float));
  L.m1 = off; off = round_up(off + PG1 * sizeof(float));
  L.cmseg = off; off = round_up(off + (NC1 + PG1) * sizeof(float));  // PG1 chains of S / (G1 Ls) + 1
  L.wx = off; off = round_up(off + PS1 * sizeof(float));
  L.wn = off; off = round_up(off + PS1 * sizeof(float));
  L.pre = L.tc && L.G == 1 && use_prepass((int)P, S, DQK, DV);
  const size_t PSp = L.pre ? P * (size_t)S : 0, PNCp = L.pre ? P * (size_t)(S / 64) : 0;
  L.qb = off; off = round_up(off + PSp * DQK * 2);
  L.kw = off; off = round_up(off + PSp * DQK * 2);
  L.pm = off; off = round_up(off + PSp * 64 * 2);
  L.pden = off; off = round_up(off + PSp * sizeof(float));
  L.pinv = off; off = round_up(off + PSp * sizeof(float));
  L.ptok4 = off; off = round_up(off + PSp * 4 * sizeof(float));
  L.ptok2 = off; off = round_up(off + PSp * 2 * sizeof(float));
  L.pdn = off; off = round_up(off + PNCp * DQK * sizeof(float));
  L.pcdat = off; off = round_up(off + PNCp * 2 * 4 * sizeof(float));
  L.split_total = off;
  return L;
}

// Bytes that mlstm_fwd_chunkwise (and mlstm_fwd_chunk_states, mlstm_fwd_gates) need on the
// path the forward actually takes: the fused kernel runs in its own chunks of kTcChunk tokens
// whatever chunk is asked for, and needs no boundary states; the gate stage of the asked-for
// chunk must still fit (mlstm_fwd_chunk_states and mlstm_fwd_gates use it).  With `split` the
// fused path's size includes the sequence-parallel buffers (the size mlstm_fwd_workspace_bytes
// reports); without, it is the least workspace the forward accepts.
size_t fwd_need(int B, int NH, int S, int DQK, int DV, int chunk, mlstm_dtype dt, bool split = true) {
  if (use_tc(B, NH, S, DQK, DV, kTcChunk, dt)) {
    const Layout L = layout(B, NH, S, DQK, DV, kTcChunk, dt);
    const size_t tc = split ? L.split_total : L.total;
    const size_t gates = layout(B, NH, S, DQK, DV, chunk, dt).gates_end;
    return tc > gates ? tc : gates;
  }
  return layout(B, NH, S, DQK, DV, chunk, dt).total;
}

inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// The forget-gate variant rides in the dtype argument of the calls that read raw gate
// pre-activations: MLSTM_FORGET_EXP OR-ed into dt selects f = exp(f~) (log f = f~).
inline mlstm_dtype split_forget(mlstm_dtype dt, bool &exp_fg) {
  exp_fg = ((int)dt & (int)MLSTM_FORGET_EXP) != 0;
  return (mlstm_dtype)((int)dt & ~(int)MLSTM_FORGET_EXP);
}

thread_local int g_last_cuda_error = 0;
unsigned long long g_launches = 0;  // kernels launched by this library (all host threads)

mlstm_status launch_status(cudaError_t e, int kernels = 1) {
  if (e == cudaSuccess) {
    __atomic_fetch_add(&g_launches, (unsigned long long)kernels, __ATOMIC_RELAXED);
    return MLSTM_OK;
  }
  g_last_cuda_error = (int)e;
  return MLSTM_ERR_LAUNCH;
}

// Synchronises `s`, then reads the wait-error word at offset 0 of a forward workspace.
mlstm_status read_error_word(const void *workspace, cudaStream_t s) {
  int word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    g_last_cuda_error = (int)cudaGetLastError();
    return MLSTM_ERR_LAUNCH;
  }
  if (word != 0) {
    g_last_cuda_error = word;  // the code of the wait that gave up
    return MLSTM_ERR_TIMEOUT;
  }
  return MLSTM_OK;
}

mlstm_status check_device() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return MLSTM_ERR_DEVICE; }
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return MLSTM_ERR_DEVICE;
  }
  if (major != 10 || minor != 3) return MLSTM_ERR_DEVICE;
  return MLSTM_OK;
}

}  // namespace
}  // namespace mlstm

using namespace mlstm;

extern "C" {

const char *mlstm_status_str(mlstm_status s) {
  switch (s) {
    case MLSTM_OK: return "MLSTM_OK";
    case MLSTM_ERR_NULL: return "MLSTM_ERR_NULL: a required pointer is NULL";
    case MLSTM_ERR_ALIGN: return "MLSTM_ERR_ALIGN: a pointer is not 16-byte aligned";
    case MLSTM_ERR_SHAPE: return "MLSTM_ERR_SHAPE: unsupported sizes (S % chunk, chunk, DQK/DV range)";
    case MLSTM_ERR_DTYPE: return "MLSTM_ERR_DTYPE: unsupported dtype code";
    case MLSTM_ERR_WORKSPACE: return "MLSTM_ERR_WORKSPACE: workspace too small";
    case MLSTM_ERR_LAUNCH: return "MLSTM_ERR_LAUNCH: a kernel launch failed";
    case MLSTM_ERR_TIMEOUT: return "MLSTM_ERR_TIMEOUT: a bounded device-side wait gave up";
    case MLSTM_ERR_DEVICE: return "MLSTM_ERR_DEVICE: no usable sm_103 device";
  }
  return "MLSTM_ERR_UNKNOWN";
}

// CUDA error code of the last failed launch on this host thread (0 if none).
int mlstm_last_cuda_error(void) { return g_last_cuda_error; }

unsigned long long mlstm_kernel_launches(void) { return __atomic_load_n(&g_launches, __ATOMIC_RELAXED); }

int mlstm_fwd_path(int B, int NH, int S, int DQK, int DV, int chunk, mlstm_dtype dt) {
  bool exp_fg;
  dt = split_forget(dt, exp_fg);
  if (dt != MLSTM_F32 && dt != MLSTM_BF16) return -1;
  if (!sizes_ok(B, NH, S, DQK, DV, chunk)) return -1;
  if (!use_tc(B, NH, S, DQK, DV, kTcChunk, dt)) return 0;
  return fwd_tc_pair(B * NH, DQK, DV) ? 2 : 1;
}

size_t mlstm_fwd_workspace_min_bytes(int B, int NH, int S, int DQK, int DV, int chunk, mlstm_dtype dt) {
  bool exp_fg;
  dt = split_forget(dt, exp_fg);
  if (dt != MLSTM_F32 && dt != MLSTM_BF16) return 0;
  if (!sizes_ok(B, NH, S, DQK, DV, chunk)) return 0;
  return fwd_need(B, NH, S, DQK, DV, chunk, dt, false);
}

int mlstm_fwd_segments(int B, int NH, int S, int DQK, int DV, int chunk, mlstm_dtype dt, size_t ws_bytes) {
  bool exp_fg;
  dt = split_forget(dt, exp_fg);
  if (dt != MLSTM_F32 && dt != MLSTM_BF16) return -1;
  if (!sizes_ok(B, NH, S, DQK, DV, chunk)) return -1;
  if (!use_tc(B, NH, S, DQK, DV, kTcChunk, dt)) return 1;
  const Layout L = layout(B, NH, S, DQK, DV, kTcChunk, dt);
  return L.G > 1 && ws_bytes >= L.split_total ? L.G : 1;
}

size_t mlstm_fwd_workspace_bytes(int B, int NH, int S, int DQK, int DV, int chunk, mlstm_dtype dt) {
  bool exp_fg;
  dt = split_forget(dt, exp_fg);
  if (dt != MLSTM_F32 && dt != MLSTM_BF16) return 0;
  if (!sizes_ok(B, NH, S, DQK, DV, chunk)) return 0;
  return fwd_need(B, NH, S, DQK, DV, chunk, dt);
}

static mlstm_status check_init(const float *C_init, const float *n_init, const float *m_init) {
  const int given = (C_init != nullptr) + (n_init != nullptr) + (m_init != nullptr);
  if (given != 0 && given != 3) return MLSTM_ERR_NULL;
  if (given && (!aligned16(C_init) || !aligned16(n_init) || !aligned16(m_init))) return MLSTM_ERR_ALIGN;
  return MLSTM_OK;
}

static mlstm_status check_fwd_args(const void *q, const void *k, const void *v, int B, int NH, int S,
                                   int DQK, int DV, int chunk, mlstm_dtype dt, const float *C_init,
                                   const float *n_init, const void *h, mlstm_dtype h_dt,
                                   const float *C_last, const float *n_last, const float *m_last,
                                   const void *workspace, size_t ws_bytes, size_t ws_need) {
  if (dt != MLSTM_F32 && dt != MLSTM_BF16) return MLSTM_ERR_DTYPE;
  if (h_dt != MLSTM_F32 && h_dt != MLSTM_BF16) return MLSTM_ERR_DTYPE;
  if (!sizes_ok(B, NH, S, DQK, DV, chunk)) return MLSTM_ERR_SHAPE;
  // per-token arrays may be NULL for an empty sequence (zero-size tensors have no storage)
  if (S > 0 && (!q || !k || !v || !h)) return MLSTM_ERR_NULL;
  if (!C_last || !n_last || !m_last || !workspace) return MLSTM_ERR_NULL;
  if ((C_init == nullptr) != (n_init == nullptr)) return MLSTM_ERR_NULL;
  for (const void *ptr : {q, k, v, h, (const void *)C_last, (const void *)n_last, (const void *)m_last, workspace})
    if (!aligned16(ptr)) return MLSTM_ERR_ALIGN;
  if ((C_init && !aligned16(C_init)) || (n_init && !aligned16(n_init))) return MLSTM_ERR_ALIGN;
  if (ws_bytes < ws_need) return MLSTM_ERR_WORKSPACE;
  return MLSTM_OK;
}

// The fused forward over G segments of each head's sequence at once, for long sequences over
// few heads: a first pass computes the own map of each of G1 >= G finer segments from the zero
// state with m = -inf (gate preprocessing and the tensor-core state walk over P G1 heads of
// S / G1 tokens, final state only), a scan composes the maps from the caller's initial state
// into the entering state of each of the G segments and the final state, and the fused kernel
// then runs all P G segments from their entering states.  Each (head, segment) is a head of S / G tokens to the kernels: the
// token-major arrays need no copies.
static mlstm_status run_segments(const void *q, const void *k, const void *v, const Layout &Lw, int P, int S,
                                 int DQK, int DV, const float *C_init, const float *n_init, const float *m_init,
                                 const float *ig, const float *fg, bool exp_fg, void *h, mlstm_dtype h_dt,
                                 float *C_last, float *n_last, float *m_last, char *ws, cudaStream_t s) {
  const int G = Lw.G, PG = P * G, Sg = S / G, G1 = Lw.G1, PG1 = P * G1, Sg1 = S / G1, Ls = Lw.Ls;
  auto F = [&](size_t off) { return (float *)(ws + off); };
  int *err = (int *)(ws + Lw.err);
  const bool hb = h_dt == MLSTM_BF16;
  cudaError_t e = launch_seg_init(fg, exp_fg, P, G1, Sg1, F(Lw.m1), F(Lw.Bg), s);
  if (e == cudaSuccess)
    e = launch_gates(ig, fg, PG1, Sg1, Ls, F(Lw.m1), F(Lw.gb), F(Lw.gx), F(Lw.gu), F(Lw.cmseg), nullptr, s, exp_fg);
  if (e == cudaSuccess)
    e = launch_state_weights(2, F(Lw.gb), F(Lw.gx), F(Lw.gu), F(Lw.cmseg), nullptr, nullptr, PG1, Sg1, Ls, DQK,
                             F(Lw.wx), F(Lw.wn), nullptr, nullptr, s);
  if (e == cudaSuccess)
    e = launch_states_tc(v, k, F(Lw.wx), F(Lw.wn), nullptr, nullptr, PG1, Sg1, Ls, DQK, DV, false, nullptr, nullptr,
                         nullptr, nullptr, F(Lw.Cseg), F(Lw.nseg), err, s);
  if (e == cudaSuccess)
    e = launch_seg_scan(P, G1, G1 / G, DQK, DV, Sg1 / Ls, F(Lw.Bg), F(Lw.Cseg), F(Lw.nseg), F(Lw.cmseg), C_init,
                        n_init, m_init, F(Lw.Cin), F(Lw.nin), F(Lw.min), C_last, n_last, m_last, s);
  if (e != cudaSuccess) return launch_status(e);
  if (mlstm_status st = launch_status(cudaSuccess, 5)) return st;
  // the segments' own final states land in the first pass's buffers, which are free by now
  return launch_status(launch_fwd_tc(q, k, v, hb, F(Lw.gb), F(Lw.gx), F(Lw.gu), F(Lw.cm), ig, fg, F(Lw.min), PG,
                                     Sg, DQK, DV, F(Lw.Cin), F(Lw.nin), h, F(Lw.Cseg), F(Lw.nseg), F(Lw.mseg), err, s,
                                     exp_fg, P));
}

// The forward in three kernels: the pre-pass (per head and chunk: Q K^T on tensor cores, P,
// beta q, w k, the n increment, the chunk's stabiliser and frame), the n chain with every token's
// 1/den, and the state walk (U, X and P V on tensor cores).  n_init is read by every chunk's CTA
// of the second kernel while one of them writes n_last, which may alias it: a copy is read.
static mlstm_status run_prepass(const void *q, const void *k, const void *v, const Layout &Lw, int P, int S, int DQK,
                                int DV, const float *C_init, const float *n_init, const float *m_init, const float *ig,
                                const float *fg, bool exp_fg, void *h, mlstm_dtype h_dt, float *C_last,
                                float *n_last, float *m_last, char *ws, cudaStream_t s) {
  PrepBuffers b;
  b.qb = (__half *)(ws + Lw.qb);
  b.kw = (__half *)(ws + Lw.kw);
  b.pm = (__half *)(ws + Lw.pm);
  b.den = (float *)(ws + Lw.pden);
  b.inv = (float *)(ws + Lw.pinv);
  b.dn = (float *)(ws + Lw.pdn);
  b.tok4 = (float4 *)(ws + Lw.ptok4);
  b.tok2 = (float2 *)(ws + Lw.ptok2);
  b.cdat = (float4 *)(ws + Lw.pcdat);
  int *err = (int *)(ws + Lw.err);
  if (n_init) {
    float *ncopy = (float *)(ws + Lw.ncopy);
    if (cudaMemcpyAsync(ncopy, n_init, sizeof(float) * (size_t)P * DQK, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return launch_status(cudaGetLastError());
    n_init = ncopy;
  }
  if (mlstm_status st = launch_status(
          launch_fwd_prep(q, k, ig, fg, m_init, P, S, DQK, exp_fg, b, n_init, n_last, m_last, err, s), 4))
    return st;
  return launch_status(launch_fwd_state(b, v, h_dt == MLSTM_BF16, P, S, DQK, DV, C_init, h, C_last, err, s));
}

// Everything after kernel (a), on a workspace that kernel (a) has filled for these sizes -- or,
// on the tensor-core path when ig is given, from the raw gate pre-activations (ig, fg, m_init),
// whose preprocessing the fused kernel then does itself.
static mlstm_status run_from_gates(const void *q, const void *k, const void *v, int B, int NH, int S,
                                   int DQK, int DV, int chunk, mlstm_dtype dt, const float *C_init,
                                   const float *n_init, void *h, mlstm_dtype h_dt, float *C_last,
                                   float *n_last, float *m_last, void *workspace, size_t ws_bytes,
                                   cudaStream_t s, const float *ig = nullptr, const float *fg = nullptr,
                                   const float *m_init = nullptr, bool exp_fg = false) {
  const Layout Lw = layout(B, NH, S, DQK, DV, chunk, dt);
  // The wait-error word reports on this forward only: it is cleared in stream order before the
  // first kernel, on every path (the CUDA-core kernels have no bounded waits and leave it 0).
  char *ws = (char *)workspace;
  float *gb = (float *)(ws + Lw.gb), *gx = (float *)(ws + Lw.gx), *gu = (float *)(ws + Lw.gu);
  float *cm = (float *)(ws + Lw.cm), *Cs = (float *)(ws + Lw.Cs), *ns = (float *)(ws + Lw.ns);
  int *err = (int *)(ws + Lw.err);
  const int P = B * NH, NC = S / chunk;
  const bool bf16 = dt == MLSTM_BF16;
  if (cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess) return launch_status(cudaGetLastError());
  if (Lw.tc && ig != nullptr && Lw.G > 1 && ws_bytes >= Lw.split_total)
    return run_segments(q, k, v, Lw, P, S, DQK, DV, C_init, n_init, m_init, ig, fg, exp_fg, h, h_dt, C_last,
                        n_last, m_last, ws, s);
  if (Lw.tc && ig != nullptr && Lw.pre && ws_bytes >= Lw.split_total)
    return run_prepass(q, k, v, Lw, P, S, DQK, DV, C_init, n_init, m_init, ig, fg, exp_fg, h, h_dt, C_last, n_last,
                       m_last, ws, s);
  if (Lw.tc) {
    if (n_init) {
      float *ncopy = (float *)(ws + Lw.ncopy);
      if (cudaMemcpyAsync(ncopy, n_init, sizeof(float) * (size_t)P * DQK, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return launch_status(cudaGetLastError());
      n_init = ncopy;
    }
    return launch_status(launch_fwd_tc(q, k, v, h_dt == MLSTM_BF16, gb, gx, gu, cm, ig, fg, m_init, P, S, DQK,
                                       DV, C_init, n_init, h, C_last, n_last, m_last, err, s, exp_fg));
  }
  if (mlstm_status st = launch_status(launch_states_simt(k, v, bf16, gb, gx, cm, P, S, chunk, DQK, DV, C_init,
                                                         n_init, Cs, ns, C_last, n_last, s)))
    return st;
  if (S > 0) {
    if (mlstm_status st = launch_status(launch_output_simt(q, k, v, bf16, h_dt == MLSTM_BF16, gb, gx, gu, cm,
                                                           Cs, ns, P, S, chunk, DQK, DV, h, s)))
      return st;
  }
  return launch_status(launch_copy_chunk_m(cm, P, NC, m_last, s));
}

mlstm_status mlstm_fwd_from_gates(const void *q, const void *k, const void *v, int B, int NH, int S,
                                  int DQK, int DV, int chunk, mlstm_dtype dt, const float *C_init,
                                  const float *n_init, void *h, mlstm_dtype h_dt, float *C_last,
                                  float *n_last, float *m_last, void *workspace, size_t ws_bytes,
                                  void *stream) {
  bool exp_fg;  // the variant is that of the gates already in the workspace
  dt = split_forget(dt, exp_fg);
  if (mlstm_status st = check_fwd_args(q, k, v, B, NH, S, DQK, DV, chunk, dt, C_init, n_init, h, h_dt,
                                       C_last, n_last, m_last, workspace, ws_bytes,
                                       sizes_ok(B, NH, S, DQK, DV, chunk) && (dt == MLSTM_F32 || dt == MLSTM_BF16)
                                           ? layout(B, NH, S, DQK, DV, chunk, dt).total
                                           : 0))
    return st;
  if (mlstm_status st = check_device()) return st;
  return run_from_gates(q, k, v, B, NH, S, DQK, DV, chunk, dt, C_init, n_init, h, h_dt, C_last, n_last,
                        m_last, workspace, ws_bytes, (cudaStream_t)stream);
}

mlstm_status mlstm_fwd_chunkwise(const void *q, const void *k, const void *v, const float *igate_pre,
                                 const float *fgate_pre, int B, int NH, int S, int DQK, int DV,
                                 int chunk, mlstm_dtype dt, const float *C_init, const float *n_init,
                                 const float *m_init, void *h, mlstm_dtype h_dt, float *C_last,
                                 float *n_last, float *m_last, void *workspace, size_t ws_bytes,
                                 void *stream) {
  bool exp_fg;
  dt = split_forget(dt, exp_fg);
  if (mlstm_status st = check_fwd_args(q, k, v, B, NH, S, DQK, DV, chunk, dt, C_init, n_init, h, h_dt,
                                       C_last, n_last, m_last, workspace, ws_bytes,
                                       sizes_ok(B, NH, S, DQK, DV, chunk) && (dt == MLSTM_F32 || dt == MLSTM_BF16)
                                           ? fwd_need(B, NH, S, DQK, DV, chunk, dt, false)
                                           : 0))
    return st;
  if (S > 0 && (!igate_pre || !fgate_pre)) return MLSTM_ERR_NULL;
  if (mlstm_status st = check_init(C_init, n_init, m_init)) return st;
  if (!aligned16(igate_pre) || !aligned16(fgate_pre)) return MLSTM_ERR_ALIGN;
  if (mlstm_status st = check_device()) return st;

  cudaStream_t s = (cudaStream_t)stream;
  char *ws = (char *)workspace;
  const int P = B * NH;
  // The fused kernel preprocesses the gates itself and walks the sequence in its own chunks of
  // 64 tokens, whatever chunk was asked for (the result is the same function up to rounding);
  // its workspace needs are below those of the asked-for chunk's layout, which was checked.
  if (use_tc(B, NH, S, DQK, DV, kTcChunk, dt))
    return run_from_gates(q, k, v, B, NH, S, DQK, DV, kTcChunk, dt, C_init, n_init, h, h_dt, C_last, n_last,
                          m_last, workspace, ws_bytes, s, igate_pre, fgate_pre, m_init, exp_fg);
  const Layout Lw = layout(B, NH, S, DQK, DV, chunk, dt);
  if (mlstm_status st = launch_status(launch_gates(igate_pre, fgate_pre, P, S, chunk, m_init, (float *)(ws + Lw.gb),
                                                   (float *)(ws + Lw.gx), (float *)(ws + Lw.gu),
                                                   (float *)(ws + Lw.cm), nullptr, s, exp_fg)))
    return st;
  return run_from_gates(q, k, v, B, NH, S, DQK, DV, chunk, dt, C_init, n_init, h, h_dt, C_last, n_last,
                        m_last, workspace, ws_bytes, s);
}

mlstm_status mlstm_fwd_chunk_states(const void *k, const void *v, const float *igate_pre,
                                    const float *fgate_pre, int B, int NH, int S, int DQK, int DV,
                                    int chunk, mlstm_dtype dt, const float *C_init, const float *n_init,
                                    const float *m_init, float *C_states, float *n_states,
                                    float *m_states, void *workspace, size_t ws_bytes, void *stream) {
  bool exp_fg;
  dt = split_forget(dt, exp_fg);
  if (dt != MLSTM_F32 && dt != MLSTM_BF16) return MLSTM_ERR_DTYPE;
  if (!sizes_ok(B, NH, S, DQK, DV, chunk)) return MLSTM_ERR_SHAPE;
  if (S > 0 && (!k || !v || !igate_pre || !fgate_pre)) return MLSTM_ERR_NULL;
  if (!C_states || !n_states || !m_states || !workspace) return MLSTM_ERR_NULL;
  if (mlstm_status st = check_init(C_init, n_init, m_init)) return st;
  for (const void *ptr : {(const void *)k, (const void *)v, (const void *)igate_pre, (const void *)fgate_pre,
                          (const void *)C_states, (const void *)n_states, (const void *)m_states,
                          (const void *)workspace})
    if (!aligned16(ptr)) return MLSTM_ERR_ALIGN;
  const Layout Lw = layout(B, NH, S, DQK, DV, chunk, dt);
  if (ws_bytes < Lw.gates_end) return MLSTM_ERR_WORKSPACE;
  if (mlstm_status st = check_device()) return st;

  cudaStream_t s = (cudaStream_t)stream;
  char *ws = (char *)workspace;
  float *gb = (float *)(ws + Lw.gb), *gx = (float *)(ws + Lw.gx), *gu = (float *)(ws + Lw.gu);
  float *cm = (float *)(ws + Lw.cm);
  const int P = B * NH, NC = S / chunk;
  if (mlstm_status st = launch_status(launch_gates(igate_pre, fgate_pre, P, S, chunk, m_init, gb, gx, gu, cm, nullptr, s,
                                                   exp_fg)))
    return st;
  if (mlstm_status st = launch_status(launch_states_simt(k, v, dt == MLSTM_BF16, gb, gx, cm, P, S, chunk, DQK,
                                                         DV, C_init, n_init, C_states, n_states, nullptr,
                                                         nullptr, s)))
    return st;
  return launch_status(cudaMemcpyAsync(m_states, cm, sizeof(float) * (size_t)P * (NC + 1),
                                       cudaMemcpyDeviceToDevice, s));
}

mlstm_status mlstm_fwd_gates(const float *igate_pre, const float *fgate_pre, int B, int NH, int S,
                             int chunk, const float *m_init, float *m_tok, float *m_states,
                             void *workspace, size_t ws_bytes, void *stream) {
  if (!sizes_ok(B, NH, S, 32, 32, chunk)) return MLSTM_ERR_SHAPE;
  if ((S > 0 && (!igate_pre || !fgate_pre)) || !workspace) return MLSTM_ERR_NULL;
  for (const void *ptr : {(const void *)igate_pre, (const void *)fgate_pre, (const void *)workspace})
    if (!aligned16(ptr)) return MLSTM_ERR_ALIGN;
  if ((m_init && !aligned16(m_init)) || (m_tok && !aligned16(m_tok)) || (m_states && !aligned16(m_states)))
    return MLSTM_ERR_ALIGN;
  const Layout Lw = layout(B, NH, S, 32, 32, chunk, MLSTM_F32);
  if (ws_bytes < Lw.gates_end) return MLSTM_ERR_WORKSPACE;
  if (mlstm_status st = check_device()) return st;

  cudaStream_t s = (cudaStream_t)stream;
  char *ws = (char *)workspace;
  float *gb = (float *)(ws + Lw.gb), *gx = (float *)(ws + Lw.gx), *gu = (float *)(ws + Lw.gu);
  float *cm = (float *)(ws + Lw.cm);
  const int P = B * NH, NC = S / chunk;
  if (mlstm_status st = launch_status(launch_gates(igate_pre, fgate_pre, P, S, chunk, m_init, gb, gx, gu, cm, m_tok, s)))
    return st;
  if (m_states)
    return launch_status(cudaMemcpyAsync(m_states, cm, sizeof(float) * (size_t)P * (NC + 1),
                                         cudaMemcpyDeviceToDevice, s));
  return MLSTM_OK;
}

mlstm_status mlstm_fwd_check(const void *workspace, size_t ws_bytes, int B, int NH, int S, int DQK, int DV,
                             int chunk, mlstm_dtype dt, void *stream) {
  bool exp_fg;
  dt = split_forget(dt, exp_fg);
  if (dt != MLSTM_F32 && dt != MLSTM_BF16) return MLSTM_ERR_DTYPE;
  if (!sizes_ok(B, NH, S, DQK, DV, chunk)) return MLSTM_ERR_SHAPE;
  if (!workspace) return MLSTM_ERR_NULL;
  if (ws_bytes < kAlign) return MLSTM_ERR_WORKSPACE;  // the error word's header
  if (mlstm_status st = check_device()) return st;
  return read_error_word(workspace, (cudaStream_t)stream);
}

mlstm_status mlstm_wait_selftest(void *workspace, size_t ws_bytes, int B, int NH, int S, int DQK, int DV,
                                 int chunk, mlstm_dtype dt, void *stream) {
  bool exp_fg;
  dt = split_forget(dt, exp_fg);
  if (dt != MLSTM_F32 && dt != MLSTM_BF16) return MLSTM_ERR_DTYPE;
  if (!sizes_ok(B, NH, S, DQK, DV, chunk)) return MLSTM_ERR_SHAPE;
  if (!workspace) return MLSTM_ERR_NULL;
  if (!aligned16(workspace)) return MLSTM_ERR_ALIGN;
  if (ws_bytes < kAlign) return MLSTM_ERR_WORKSPACE;  // the error word's header
  if (mlstm_status st = check_device()) return st;
  return launch_status(launch_wait_selftest((int *)workspace, MLSTM_SELFTEST_WAIT_CODE, (cudaStream_t)stream));
}

// ---------------------------------------------------------------- backward
namespace {
struct BwdLayout {
  size_t gb, gx, gu, cm, Cs, ns, Gs, Ns, h32, den, invD, cc, pq, pk, wx, wn, al, sc;
  size_t Cst, Gst, q32, k32, v32, dh32, xq, yq, yk, yv, pm, m1, nq, total;
  bool tc_states, tc_prod;  // state walks / state products on tensor cores
};

BwdLayout bwd_layout(int B, int NH, int S, int DQK, int DV, int chunk, bool bf16) {
  const size_t P = (size_t)B * NH, NC = (size_t)S / chunk, PS = P * S, nt = (size_t)DQK / 32;
  BwdLayout L{};
  L.tc_states = S > 0 && states_tc_supported(chunk, DQK, DV, bf16);
  L.tc_prod = L.tc_states && state_prod_supported(chunk, DQK, DV);
  size_t off = kAlign;  // offset 0: the error-word header every workspace keeps
  auto take = [&](size_t &at, size_t floats) {
    at = off;
    off = round_up(off + floats * sizeof(float));
  };
  take(L.gb, PS);
  take(L.gx, PS);
  take(L.gu, PS);
  take(L.cm, P * (NC + 1));
  take(L.Cs, P * (NC + 1) * DV * DQK);
  take(L.ns, P * (NC + 1) * DQK);
  take(L.Gs, P * (NC + 1) * DV * DQK);
  take(L.Ns, P * (NC + 1) * DQK);
  take(L.h32, PS * DV);
  take(L.den, PS);
  take(L.invD, PS);
  take(L.cc, PS);
  take(L.pq, PS * nt);
  take(L.pk, PS * nt);
  take(L.wx, PS);  // tensor-core state walks: per-token weights and per-chunk factors
  take(L.wn, PS);
  take(L.al, P * NC);
  take(L.sc, P * NC);
  // tensor-core state products: transposed states, fp32 copies of the tokens, the products
  const size_t SQ = L.tc_prod ? P * (NC + 1) * DV * DQK : 0, TQ = L.tc_prod ? PS * DQK : 0, TV = L.tc_prod ? PS * DV : 0;
  take(L.Cst, SQ);
  take(L.Gst, SQ);
  take(L.q32, TQ);
  take(L.k32, TQ);
  take(L.v32, TV);
  take(L.dh32, TV);
  take(L.xq, TV);
  take(L.yq, TQ);
  take(L.yk, TQ);
  take(L.yv, TV);
  take(L.pm, P * NC * chunk * chunk);  // each chunk's L x L matrices, formed once
  take(L.m1, P * NC * chunk * chunk);
  take(L.nq, PS);
  L.total = off;
  return L;
}
}  // namespace

size_t mlstm_bwd_workspace_bytes(int B, int NH, int S, int DQK, int DV, int chunk, mlstm_dtype dt) {
  bool exp_fg;
  dt = split_forget(dt, exp_fg);
  if (dt != MLSTM_F32 && dt != MLSTM_BF16) return 0;
  if (!sizes_ok(B, NH, S, DQK, DV, chunk)) return 0;
  return bwd_layout(B, NH, S, DQK, DV, chunk, dt == MLSTM_BF16).total;
}

mlstm_status mlstm_bwd_chunkwise(const void *q, const void *k, const void *v, const float *igate_pre,
                                 const float *fgate_pre, const void *dh, int B, int NH, int S, int DQK, int DV,
                                 int chunk, mlstm_dtype dt, const float *C_init, const float *n_init,
                                 const float *m_init, void *dq, void *dk, void *dv, float *dig, float *dfg,
                                 float *dC_init, float *dn_init, float *dm_init, void *workspace, size_t ws_bytes,
                                 void *stream) {
  bool exp_fg;
  dt = split_forget(dt, exp_fg);
  if (dt != MLSTM_F32 && dt != MLSTM_BF16) return MLSTM_ERR_DTYPE;
  if (!sizes_ok(B, NH, S, DQK, DV, chunk)) return MLSTM_ERR_SHAPE;
  if (S > 0 && (!q || !k || !v || !igate_pre || !fgate_pre || !dh || !dq || !dk || !dv || !dig || !dfg))
    return MLSTM_ERR_NULL;
  if (!workspace) return MLSTM_ERR_NULL;
  if (mlstm_status st = check_init(C_init, n_init, m_init)) return st;
  const int dgiven = (dC_init != nullptr) + (dn_init != nullptr) + (dm_init != nullptr);
  if (dgiven != 0 && dgiven != 3) return MLSTM_ERR_NULL;
  for (const void *ptr : {q, k, v, (const void *)igate_pre, (const void *)fgate_pre, dh, (const void *)dq,
                          (const void *)dk, (const void *)dv, (const void *)dig, (const void *)dfg,
                          (const void *)dC_init, (const void *)dn_init, (const void *)dm_init,
                          (const void *)workspace})
    if (ptr && !aligned16(ptr)) return MLSTM_ERR_ALIGN;
  const BwdLayout Lw = bwd_layout(B, NH, S, DQK, DV, chunk, dt == MLSTM_BF16);
  if (ws_bytes < Lw.total) return MLSTM_ERR_WORKSPACE;
  if (mlstm_status st = check_device()) return st;

  cudaStream_t s = (cudaStream_t)stream;
  char *ws = (char *)workspace;
  auto F = [&](size_t off) { return (float *)(ws + off); };
  const int P = B * NH, NC = S / chunk;
  const bool bf16 = dt == MLSTM_BF16;
  if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return launch_status(cudaGetLastError());
  int kernels = 0;
  cudaError_t e = cudaSuccess;
  if (S > 0) {
    e = launch_gates(igate_pre, fgate_pre, P, S, chunk, m_init, F(Lw.gb), F(Lw.gx), F(Lw.gu), F(Lw.cm), nullptr, s,
                     exp_fg);
    ++kernels;
  } else {
    // no tokens: the only boundary is the initial one
    e = m_init ? cudaMemcpyAsync(F(Lw.cm), m_init, sizeof(float) * P, cudaMemcpyDeviceToDevice, s)
               : cudaMemsetAsync(F(Lw.cm), 0, sizeof(float) * P, s);
  }
  // the boundary states walk on tensor cores where the shapes allow (bf16, chunk 64 or 128,
  // d_qk a power of two from 64, d_v a multiple of 128), on CUDA cores otherwise; with d_qk a
  // multiple of 128 too, the products of the tokens with the states also run on tensor cores
  const bool tc_states = Lw.tc_states, tc_prod = Lw.tc_prod;
  int *err = (int *)ws;
  if (e == cudaSuccess && tc_states) {
    e = launch_state_weights(0, F(Lw.gb), F(Lw.gx), F(Lw.gu), F(Lw.cm), nullptr, nullptr, P, S, chunk, DQK, F(Lw.wx),
                             F(Lw.wn), F(Lw.al), F(Lw.sc), s);
    if (e == cudaSuccess)
      e = launch_states_tc(v, k, F(Lw.wx), F(Lw.wn), F(Lw.al), F(Lw.sc), P, S, chunk, DQK, DV, false, C_init, n_init,
                           F(Lw.Cs), F(Lw.ns), nullptr, nullptr, err, s, tc_prod ? F(Lw.Cst) : nullptr);
    kernels += 2;
  }
  if (e == cudaSuccess && tc_prod) {
    // fp32 copies of the tokens (the tf32 operands), then C^(k) q_t for every token
    const size_t nq = (size_t)P * S * DQK, nv = (size_t)P * S * DV;
    e = launch_to_f32(q, bf16, F(Lw.q32), nq, s);
    if (e == cudaSuccess) e = launch_to_f32(k, bf16, F(Lw.k32), nq, s);
    if (e == cudaSuccess) e = launch_to_f32(v, bf16, F(Lw.v32), nv, s);
    if (e == cudaSuccess) e = launch_to_f32(dh, bf16, F(Lw.dh32), nv, s);
    if (e == cudaSuccess)
      e = launch_state_prod(F(Lw.Cs), DV, DQK, 0, F(Lw.q32), nullptr, 1.f, P, S, chunk, F(Lw.xq), err, s);
    kernels += 5;
  } else if (e == cudaSuccess) {
    e = launch_states_simt(k, v, bf16, F(Lw.gb), F(Lw.gx), F(Lw.cm), P, S, chunk, DQK, DV, C_init, n_init, F(Lw.Cs),
                           F(Lw.ns), nullptr, nullptr, s);
    ++kernels;
  }
  // a chunk's L x L matrix (mode 0: E (q k^T) / sqrt(d) and n^(k) . q; mode 1: E (g v^T + c)): on
  // tensor cores for bf16 chunks of 64, else on CUDA cores
  auto chunk_mat = [&](int mode, const void *x, const void *y, int K, const float *invD, const float *cc, float *out,
                       float *nq) {
    if (bf16 && chunk_gram_tc_supported(chunk, K))
      return launch_chunk_gram_tc(mode, x, y, K, invD, cc, F(Lw.gx), F(Lw.gu), F(Lw.cm), F(Lw.ns), P, S, DQK, out, nq,
                                  err, s);
    return launch_bwd_mat(mode, x, y, bf16, K, invD, cc, F(Lw.gx), F(Lw.gu), F(Lw.cm), F(Lw.ns), P, S, chunk, DQK, out,
                          nq, s);
  };
  if (e == cudaSuccess && S > 0) {
    // each chunk's decay-weighted scores P (also the dv kernel's matrix) and n^(k) . q_t, once
    e = chunk_mat(0, q, k, DQK, nullptr, nullptr, F(Lw.pm), F(Lw.nq));
    if (e == cudaSuccess)
      e = launch_output_simt(q, k, v, bf16, false, F(Lw.gb), F(Lw.gx), F(Lw.gu), F(Lw.cm), F(Lw.Cs), F(Lw.ns), P, S,
                             chunk, DQK, DV, F(Lw.h32), s, F(Lw.den), tc_prod ? F(Lw.xq) : nullptr, F(Lw.pm),
                             F(Lw.nq));
    kernels += 2;
  }
  if (e == cudaSuccess && S > 0) {
    e = launch_bwd_prep(dh, bf16, F(Lw.h32), F(Lw.den), F(Lw.gb), F(Lw.gu), F(Lw.cm), P, S, chunk, DV, F(Lw.invD),
                        F(Lw.cc), s);
    // each chunk's M1 = E (g v^T + c), once
    if (e == cudaSuccess) e = chunk_mat(1, dh, v, DV, F(Lw.invD), F(Lw.cc), F(Lw.m1), nullptr);
    kernels += 2;
  }
  if (e == cudaSuccess && tc_states) {
    e = launch_state_weights(1, F(Lw.gb), F(Lw.gx), F(Lw.gu), F(Lw.cm), F(Lw.invD), F(Lw.cc), P, S, chunk, DQK,
                             F(Lw.wx), F(Lw.wn), F(Lw.al), F(Lw.sc), s);
    if (e == cudaSuccess)
      e = launch_states_tc(dh, q, F(Lw.wx), F(Lw.wn), F(Lw.al), F(Lw.sc), P, S, chunk, DQK, DV, true, nullptr,
                           nullptr, F(Lw.Gs), F(Lw.Ns), nullptr, nullptr, err, s, tc_prod ? F(Lw.Gst) : nullptr);
    kernels += 2;
  }
  if (e == cudaSuccess && tc_prod) {
    // C^(k)^T g_t = C^(k)^T dh_t / D_t, G^(k+1)^T v_t and G^(k+1) khat_t for every token
    e = launch_state_prod(F(Lw.Cst), DQK, DV, 0, F(Lw.dh32), F(Lw.invD), 1.f, P, S, chunk, F(Lw.yq), err, s);
    if (e == cudaSuccess)
      e = launch_state_prod(F(Lw.Gst), DQK, DV, 1, F(Lw.v32), nullptr, 1.f, P, S, chunk, F(Lw.yk), err, s);
    if (e == cudaSuccess)
      e = launch_state_prod(F(Lw.Gs), DV, DQK, 1, F(Lw.k32), nullptr, 1.f / sqrtf((float)DQK), P, S, chunk,
                            F(Lw.yv), err, s);
    kernels += 3;
  } else if (e == cudaSuccess) {
    e = launch_bwd_states(q, dh, bf16, F(Lw.invD), F(Lw.cc), F(Lw.gb), F(Lw.gu), F(Lw.cm), P, S, chunk, DQK, DV,
                          F(Lw.Gs), F(Lw.Ns), s);
    ++kernels;
  }
  if (e == cudaSuccess && S > 0) {
    e = launch_bwd_dqdk(q, k, v, dh, bf16, F(Lw.invD), F(Lw.cc), F(Lw.gb), F(Lw.gx), F(Lw.gu), F(Lw.cm), F(Lw.Cs),
                        F(Lw.ns), F(Lw.Gs), F(Lw.Ns), P, S, chunk, DQK, DV, dq, dk, F(Lw.pq), F(Lw.pk), s,
                        tc_prod ? F(Lw.yq) : nullptr, tc_prod ? F(Lw.yk) : nullptr, F(Lw.m1));
    ++kernels;
  }
  if (e == cudaSuccess && S > 0) {
    e = launch_bwd_dv(q, k, dh, bf16, F(Lw.invD), F(Lw.gb), F(Lw.gx), F(Lw.gu), F(Lw.cm), F(Lw.Gs), P, S, chunk,
                      DQK, DV, dv, s, tc_prod ? F(Lw.yv) : nullptr, F(Lw.pm));
    ++kernels;
  }
  if (e == cudaSuccess) {
    const size_t gs_stride = (size_t)(NC + 1) * DV * DQK, ns_stride = (size_t)(NC + 1) * DQK;
    e = launch_bwd_gates(fgate_pre, exp_fg, F(Lw.pq), F(Lw.pk), P, S, DQK / 32, F(Lw.Gs), F(Lw.Ns), gs_stride,
                         ns_stride, C_init, n_init, DQK, DV, dig, dfg, dm_init, s);
    ++kernels;
  }
  if (e == cudaSuccess && dC_init) {
    // the adjoint entering boundary 0 is the gradient of the initial state
    e = cudaMemcpy2DAsync(dC_init, sizeof(float) * DV * DQK, F(Lw.Gs), sizeof(float) * (NC + 1) * DV * DQK,
                          sizeof(float) * DV * DQK, P, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(dn_init, sizeof(float) * DQK, F(Lw.Ns), sizeof(float) * (NC + 1) * DQK,
                            sizeof(float) * DQK, P, cudaMemcpyDeviceToDevice, s);
  }
  return launch_status(e, kernels);
}

mlstm_status mlstm_step(const void *q, const void *k, const void *v, const float *ig, const float *fg,
                        float *C, float *n, float *m, void *h, int B, int NH, int DQK, int DV,
                        mlstm_dtype dt, mlstm_dtype h_dt, void *stream) {
  bool exp_fg;
  dt = split_forget(dt, exp_fg);
  if (dt != MLSTM_F32 && dt != MLSTM_BF16) return MLSTM_ERR_DTYPE;
  if (h_dt != MLSTM_F32 && h_dt != MLSTM_BF16) return MLSTM_ERR_DTYPE;
  if (!sizes_ok(B, NH, 0, DQK, DV, 16)) return MLSTM_ERR_SHAPE;
  if (!q || !k || !v || !ig || !fg || !C || !n || !m || !h) return MLSTM_ERR_NULL;
  for (const void *ptr : {(const void *)q, (const void *)k, (const void *)v, (const void *)ig, (const void *)fg,
                          (const void *)C, (const void *)n, (const void *)m, (const void *)h})
    if (!aligned16(ptr)) return MLSTM_ERR_ALIGN;
  if (mlstm_status st = check_device()) return st;
  return launch_status(launch_step(q, k, v, dt == MLSTM_BF16, h_dt == MLSTM_BF16, ig, fg, C, n, m, h,
                                   B * NH, DQK, DV, (cudaStream_t)stream, exp_fg));
}

mlstm_status mlstm_step_multi(const void *q, const void *k, const void *v, const float *ig, const float *fg,
                              float *C, float *n, float *m, void *h, int B, int NH, int T, int DQK, int DV,
                              mlstm_dtype dt, mlstm_dtype h_dt, void *stream) {
  bool exp_fg;
  dt = split_forget(dt, exp_fg);
  if (dt != MLSTM_F32 && dt != MLSTM_BF16) return MLSTM_ERR_DTYPE;
  if (h_dt != MLSTM_F32 && h_dt != MLSTM_BF16) return MLSTM_ERR_DTYPE;
  if (!sizes_ok(B, NH, 0, DQK, DV, 16) || T < 1 || T > step_multi_max_tokens()) return MLSTM_ERR_SHAPE;
  if (!q || !k || !v || !ig || !fg || !C || !n || !m || !h) return MLSTM_ERR_NULL;
  for (const void *ptr : {(const void *)q, (const void *)k, (const void *)v, (const void *)ig, (const void *)fg,
                          (const void *)C, (const void *)n, (const void *)m, (const void *)h})
    if (!aligned16(ptr)) return MLSTM_ERR_ALIGN;
  if (mlstm_status st = check_device()) return st;
  return launch_status(launch_step_multi(q, k, v, dt == MLSTM_BF16, h_dt == MLSTM_BF16, ig, fg, C, n, m, h,
                                         B * NH, T, DQK, DV, (cudaStream_t)stream, exp_fg));
}

mlstm_status mlstm_groupnorm_gate(const void *h, const void *o_pre, const float *gamma, const float *beta,
                                  float eps, void *y, int B, int NH, int S, int DV, mlstm_dtype h_dt,
                                  mlstm_dtype o_dt, mlstm_dtype y_dt, void *stream) {
  for (mlstm_dtype d : {h_dt, o_dt, y_dt})
    if (d != MLSTM_F32 && d != MLSTM_BF16) return MLSTM_ERR_DTYPE;
  if (B < 1 || NH < 1 || S < 0 || (long long)B * NH * S > (1LL << 40)) return MLSTM_ERR_SHAPE;
  if (DV < 32 || DV > 512 || DV % 32 != 0) return MLSTM_ERR_SHAPE;
  if (!(eps > 0.f) || !(eps < 3.0e38f)) return MLSTM_ERR_SHAPE;  // also rejects NaN
  if (!gamma || !beta || (S > 0 && (!h || !o_pre || !y))) return MLSTM_ERR_NULL;
  for (const void *ptr : {h, o_pre, (const void *)gamma, (const void *)beta, (const void *)y})
    if (!aligned16(ptr)) return MLSTM_ERR_ALIGN;
  if (mlstm_status st = check_device()) return st;
  return launch_status(launch_groupnorm_gate(h, h_dt == MLSTM_BF16, o_pre, o_dt == MLSTM_BF16, gamma, beta, eps, y,
                                             y_dt == MLSTM_BF16, B, NH, S, DV, (cudaStream_t)stream));
}

// ---------------------------------------------------------------- forward without allocation
// The scratch of mlstm_fwd_chunkwise_noalloc: a fixed array in device memory, part of the
// library's image, so that every GPU that loads the library holds it until the process exits.
// Host code only ever sees a host-side stand-in for its name; the device address is resolved
// per device with cudaGetSymbolAddress and passed to the kernels as an ordinary workspace.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MLSTM_NOALLOC_SCRATCH_BYTES];

static void *g_noalloc_ptr[64];  // device address of g_noalloc_scratch, per device ordinal

// The array's device address on the current device, resolved on first use (set-up, once per
// device, with that device current).
static mlstm_status noalloc_scratch_ptr(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    g_last_cuda_error = (int)cudaGetLastError();
    return MLSTM_ERR_DEVICE;
  }
  if (dev < 0 || dev >= 64) return MLSTM_ERR_DEVICE;
  void *scratch = __atomic_load_n(&g_noalloc_ptr[dev], __ATOMIC_ACQUIRE);
  if (scratch == nullptr) {
    const cudaError_t e = cudaGetSymbolAddress(&scratch, g_noalloc_scratch);
    if (e != cudaSuccess || scratch == nullptr) {
      g_last_cuda_error = (int)e;
      cudaGetLastError();
      return MLSTM_ERR_LAUNCH;
    }
    __atomic_store_n(&g_noalloc_ptr[dev], scratch, __ATOMIC_RELEASE);
  }
  *out = scratch;
  return MLSTM_OK;
}

mlstm_status mlstm_fwd_chunkwise_noalloc(const void *q, const void *k, const void *v,
                                         const float *igate_pre, const float *fgate_pre, int B,
                                         int NH, int S, int DQK, int DV, int chunk, mlstm_dtype dt,
                                         const float *C_init, const float *n_init,
                                         const float *m_init, void *h, mlstm_dtype h_dt,
                                         float *C_last, float *n_last, float *m_last,
                                         void *stream) {
  bool exp_fg;
  const mlstm_dtype bare = split_forget(dt, exp_fg);  // dt itself (variant included) is passed on
  if (bare != MLSTM_F32 && bare != MLSTM_BF16) return MLSTM_ERR_DTYPE;
  if (!sizes_ok(B, NH, S, DQK, DV, chunk)) return MLSTM_ERR_SHAPE;
  // sizes whose scratch (on the path the forward takes) would not fit in the fixed array are
  // refused before anything runs
  if (fwd_need(B, NH, S, DQK, DV, chunk, bare, false) > (size_t)MLSTM_NOALLOC_SCRATCH_BYTES)
    return MLSTM_ERR_WORKSPACE;
  if (mlstm_status st = check_device()) return st;
  void *scratch = nullptr;
  if (mlstm_status st = noalloc_scratch_ptr(&scratch)) return st;
  // Everything the forward reads from its workspace is written by the same call first (the
  // gate arrays, the chunk stabiliser, the copy of n_init, the sequence-parallel buffers) and
  // the one word that must start at zero (the kernels' wait-error word) is cleared by the
  // forward itself, so the stale contents of an earlier call never matter.
  return mlstm_fwd_chunkwise(q, k, v, igate_pre, fgate_pre, B, NH, S, DQK, DV, chunk, dt, C_init,
                             n_init, m_init, h, h_dt, C_last, n_last, m_last, scratch,
                             (size_t)MLSTM_NOALLOC_SCRATCH_BYTES, stream);
}

mlstm_status mlstm_fwd_check_noalloc(void *stream) {
  if (mlstm_status st = check_device()) return st;
  void *scratch = nullptr;
  if (mlstm_status st = noalloc_scratch_ptr(&scratch)) return st;
  return read_error_word(scratch, (cudaStream_t)stream);
}

mlstm_status mlstm_noalloc_scratch(void **ptr, size_t *bytes) {
  if (!ptr) return MLSTM_ERR_NULL;
  if (mlstm_status st = check_device()) return st;
  if (mlstm_status st = noalloc_scratch_ptr(ptr)) return st;
  if (bytes) *bytes = (size_t)MLSTM_NOALLOC_SCRATCH_BYTES;
  return MLSTM_OK;
}

}  // extern "C"
