// kernels.cuh -- launch wrappers of the mLSTM kernels (internal to the library).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace mlstm {

// Streaming multiprocessors of the current device (148, a B300's count, when no device can be
// queried: the path queries also run on hosts without a GPU).
int sm_count();

// exp_fg selects the exponential forget gate f = exp(f~) (log f = f~) instead of sigmoid(f~).
//
// (a) gate preprocessing: per-token b, x, u [P, S] and per-chunk m [P, NC+1].
cudaError_t launch_gates(const float *ig, const float *fg, int P, int S, int L, const float *m_init,
                         float *gb, float *gx, float *gu, float *cm, float *m_tok,
                         cudaStream_t stream, bool exp_fg = false);

// (b) inter-chunk recurrence on CUDA cores; Cs/ns [P, NC+1, ...] (optional) and the final state.
cudaError_t launch_states_simt(const void *k, const void *v, bool bf16, const float *gb,
                               const float *gx, const float *cm, int P, int S, int L, int DQK,
                               int DV, const float *C_init, const float *n_init, float *Cs,
                               float *ns, float *C_last, float *n_last, cudaStream_t stream);

// (c) intra-chunk output on CUDA cores, reading the entering states Cs/ns; den_out (optional,
// [P, S]) receives each token's signed denominator n_t . q_t; xq (optional, [P, S, DV]) holds
// C^(k) q_t for every token, computed elsewhere, in place of the kernel's own product.
cudaError_t launch_output_simt(const void *q, const void *k, const void *v, bool bf16, bool out_bf16,
                               const float *gb, const float *gx, const float *gu, const float *cm,
                               const float *Cs, const float *ns, int P, int S, int L, int DQK, int DV,
                               void *h, cudaStream_t stream, float *den_out = nullptr, const float *xq = nullptr,
                               const float *pm = nullptr, const float *nq = nullptr);

// Backward of the chunkwise forward on CUDA cores (bwd_simt.cu), after the gate kernel, the
// boundary states (Cs, ns) and the output kernel (h in fp32 and den) have run for chunk L:
//   prep:   per token 1 / D_t and c_t = -(dh_t . h_t) s_t / D_t
//   states: adjoint states G, N entering every chunk boundary, walking the chunks backwards
//   dqdk:   dq, dk of every token and the per-tile partial sums of q . dq and k . dk
//   dv:     dv of every token
//   gates:  di~, df~ and (with an initial state) dm0
cudaError_t launch_bwd_prep(const void *dh, bool bf16, const float *h32, const float *den, const float *gb,
                            const float *gu, const float *cm, int P, int S, int L, int DV, float *invD, float *cc,
                            cudaStream_t stream);
cudaError_t launch_bwd_states(const void *q, const void *dh, bool bf16, const float *invD, const float *cc,
                              const float *gb, const float *gu, const float *cm, int P, int S, int L, int DQK,
                              int DV, float *Gs, float *Ns, cudaStream_t stream);
// With yq, yk (dqdk) or yv (dv) given ([P, S, DQK] or [P, S, DV]: C^(k)^T g_t, G^(k+1)^T v_t,
// G^(k+1) khat_t computed elsewhere), the kernels read them instead of forming those products.
cudaError_t launch_bwd_dqdk(const void *q, const void *k, const void *v, const void *dh, bool bf16,
                            const float *invD, const float *cc, const float *gb, const float *gx, const float *gu,
                            const float *cm, const float *Cs, const float *ns, const float *Gs, const float *Ns,
                            int P, int S, int L, int DQK, int DV, void *dq, void *dk, float *part_q,
                            float *part_k, cudaStream_t stream, const float *yq = nullptr,
                            const float *yk = nullptr, const float *m1 = nullptr);
cudaError_t launch_bwd_dv(const void *q, const void *k, const void *dh, bool bf16, const float *invD,
                          const float *gb, const float *gx, const float *gu, const float *cm, const float *Gs,
                          int P, int S, int L, int DQK, int DV, void *dv, cudaStream_t stream,
                          const float *yv = nullptr, const float *pm = nullptr);
// A chunk's L x L matrices, formed once per (chunk, head) for the kernels above ([P, NC, L, L]):
// mode 0, x = q, y = k, K = DQK: P_ut = E_ut (q_u . khat_t), and nq = n^(k) . q_u per token;
// mode 1, x = dh, y = v, K = DV: M1_ut = E_ut (dh_u . v_t / D_u + c_u).  (pm, m1 and nq also
// feed launch_output_simt, launch_bwd_dqdk and launch_bwd_dv.)
// The same two matrices on tensor cores (chunk_gram_tc.cu) for bf16 inputs, chunks of 64 and K in
// {64, 128, 256, 512}: the raw products bf16 x bf16 with fp32 sums, the factors applied in fp32.
bool chunk_gram_tc_supported(int L, int K);
cudaError_t launch_chunk_gram_tc(int mode, const void *x, const void *y, int K, const float *invD, const float *cc,
                                 const float *gx, const float *gu, const float *cm, const float *ns, int P, int S,
                                 int DQK, float *out, float *nq, int *err, cudaStream_t stream);
cudaError_t launch_bwd_mat(int mode, const void *x, const void *y, bool bf16, int K, const float *invD,
                           const float *cc, const float *gx, const float *gu, const float *cm, const float *ns, int P,
                           int S, int L, int DQK, float *out, float *nq, cudaStream_t stream);
// Chunk-boundary states on tensor cores (states_tc.cu): bf16 X [P, S, DV] and Y [P, S, DQK],
// L a multiple of 64 up to 128, DQK in {64, 128, 256, 512}, DV a multiple of 128, S > 0.  The
// weights come from launch_state_weights (mode 0: the forward state with X = v, Y = k; mode 1:
// the adjoint with X = dh, Y = q, needing invD and cc; mode 2: the final forward state alone,
// with no per-chunk factors).  Walks the chunks forwards, or backwards with `reverse`, from
// (C0, n0) (NULL = zero); states/nstates [P, NC+1, ...] and the final C_fin/n_fin are each
// optional.  With alpha == NULL (mode 2 weights) only C_fin/n_fin are written, from the zero
// state, forwards.  Bounded waits record a code in *err.
bool states_tc_supported(int L, int DQK, int DV, bool bf16);
cudaError_t launch_state_weights(int mode, const float *gb, const float *gx, const float *gu, const float *cm,
                                 const float *invD, const float *cc, int P, int S, int L, int DQK, float *wx,
                                 float *wn, float *alpha, float *sc, cudaStream_t stream);
// states_t (optional) receives every boundary state transposed, [P, NC+1, DQK, DV].
cudaError_t launch_states_tc(const void *X, const void *Y, const float *wx, const float *wn, const float *alpha,
                             const float *sc, int P, int S, int L, int DQK, int DV, bool reverse, const float *C0,
                             const float *n0, float *states, float *nstates, float *C_fin, float *n_fin, int *err,
                             cudaStream_t stream, float *states_t = nullptr);
// Products of every 64-token slab with the state at its chunk's boundary (+ bshift) on tensor
// cores (state_prod_tc.cu, tf32): Out[t][r] = scale (tok_scale[t]) sum_c A[r][c] Y[t][c], with A
// the states [P, S/L + 1, MA, K] fp32 and Y [P, S, K] fp32; L a multiple of 64, MA and K
// multiples of 128.
bool state_prod_supported(int L, int DQK, int DV);
cudaError_t launch_state_prod(const float *A, int MA, int K, int bshift, const float *Y, const float *tok_scale,
                              float scale, int P, int S, int L, float *out, int *err, cudaStream_t stream);
// bf16 or fp32 elements to fp32 (n a multiple of 8, pointers 16-byte aligned).
cudaError_t launch_to_f32(const void *src, bool bf16, float *dst, size_t n, cudaStream_t stream);
cudaError_t launch_bwd_gates(const float *fg, bool exp_fg, const float *part_q, const float *part_k, int P, int S,
                             int ntiles, const float *Gs0, const float *Ns0, size_t gs_stride, size_t ns_stride,
                             const float *C_init, const float *n_init, int DQK, int DV, float *dig, float *dfg,
                             float *dm_init, cudaStream_t stream);

// (d) single decode step, in place.
cudaError_t launch_step(const void *q, const void *k, const void *v, bool bf16, bool out_bf16,
                        const float *ig, const float *fg, float *C, float *n, float *m, void *h,
                        int P, int DQK, int DV, cudaStream_t stream, bool exp_fg = false);

// (b)+(c) fused on tensor cores (fwd_tc.cu): bf16 inputs, chunk 64, d_qk in {64, 128, 256, 512},
// d_v a multiple of 128.  fwd_tc_pair says whether a head's d_qk is split over a CTA pair.
bool fwd_tc_supported(int S, int L, int D, int DV, bool bf16);
bool fwd_tc_pair(int P, int D, int DV);
// Sequence segments the forward runs in parallel for these sizes (1 = none).
int fwd_tc_segments(int P, int S, int D, int DV);
// The gate factors come from the raw pre-activations ig, fg (and m_init) when ig is not NULL,
// otherwise from the gate kernel's b, x, u and chunk stabiliser in the workspace.
cudaError_t launch_fwd_tc(const void *q, const void *k, const void *v, bool out_bf16, const float *gb,
                          const float *gx, const float *gu, const float *cm, const float *ig, const float *fg,
                          const float *m_init, int P, int S, int D, int DV, const float *C_init,
                          const float *n_init, void *h, float *C_last, float *n_last, float *m_last, int *err,
                          cudaStream_t stream, bool exp_fg = false, int pair_heads = 0);
// The forward in three kernels (fwd_prep.cu, fwd_state.cu) for bf16 heads of d_qk 256 or 512
// split over a CTA pair: per (head, chunk) the state-independent work once (P, its row sums,
// beta q and w k in fp16, the n increment, the chunk's stabiliser and frame), then n over the
// chunks and every token's 1/den, then the state walk with the products U, X and P V only.
struct PrepBuffers {
  __half *qb, *kw, *pm;  // beta q, w k [P*S][D]; P [P*NC][64][64]
  float *den, *inv, *dn;  // [P*S], [P*S], [P*NC][D] (the n increments, then n entering each chunk)
  float4 *tok4;          // per token (x, mr, beta, w in the walk's frame / sqrt(d))
  float2 *tok2;          // per token (w / sqrt(d), exp(-m))
  float4 *cdat;          // per chunk: (m_in, m_out, alpha, frame after), (exp(frame), exp(frame) alpha, lazy, 0)
};
bool fwd_prep_supported(int S, int D);
cudaError_t launch_fwd_prep(const void *q, const void *k, const float *ig, const float *fg, const float *m_init,
                            int P, int S, int D, bool exp_fg, const PrepBuffers &b, const float *n_init,
                            float *n_last, float *m_last, int *err, cudaStream_t stream);
cudaError_t launch_fwd_state(const PrepBuffers &b, const void *v, bool out_bf16, int P, int S, int D, int DV,
                             const float *C_init, void *h, float *C_last, int *err, cudaStream_t stream);
// The sequence-parallel forward's helpers (seq_split.cu), for G segments of Sg tokens per head:
// every segment's sum of log f (Bg, P*G floats) and m = -inf as its first-pass entering
// stabiliser (min) ...
cudaError_t launch_seg_init(const float *fg, bool exp_fg, int P, int G, int Sg, float *min, float *Bg,
                            cudaStream_t stream);
// ... and the scan that composes the G segments' maps (their states Cseg, nseg and the last
// entry of their chunk stabiliser chains cm, NCg + 1 per segment) from the initial state into
// the entering state of every R-th segment (Cin, nin, min: G / R per head) and the final state.
cudaError_t launch_seg_scan(int P, int G, int R, int DQK, int DV, int NCg, const float *Bg, const float *Cseg,
                            const float *nseg, const float *cm, const float *C_init, const float *n_init,
                            const float *m_init, float *Cin, float *nin, float *min, float *C_last, float *n_last,
                            float *m_last, cudaStream_t stream);

// (d') T consecutive decode steps in one launch, in place (T <= step_multi_max_tokens()).
int step_multi_max_tokens();
cudaError_t launch_step_multi(const void *q, const void *k, const void *v, bool bf16, bool out_bf16,
                              const float *ig, const float *fg, float *C, float *n, float *m, void *h, int P,
                              int NT, int DQK, int DV, cudaStream_t stream, bool exp_fg = false);

// The block step after the cell: per-head group normalisation of h~ and the output gate,
// y = sigmoid(o~) (gamma (h~ - mu) / sqrt(var + eps) + beta) per (batch, head, token) row.
cudaError_t launch_groupnorm_gate(const void *h, bool h_bf16, const void *o_pre, bool o_bf16, const float *gamma,
                                  const float *beta, float eps, void *y, bool y_bf16, int B, int NH, int S, int DV,
                                  cudaStream_t stream);

// One bounded device-side wait on a barrier nothing completes: gives up after about a second and
// records `code` in *err (the failure path of every wait of the fused forward).
cudaError_t launch_wait_selftest(int *err, int code, cudaStream_t stream);

// small helpers
cudaError_t launch_copy_chunk_m(const float *cm, int P, int NC, float *m_last, cudaStream_t stream);

}  // namespace mlstm
