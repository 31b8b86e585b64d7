/*
 * mlstm.h -- C ABI of the B300 (sm_103a) mLSTM matrix-memory cell library.
 *
 * The cell (page "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural
 * Networks", llms.blog):
 *   section 3 "Associative Matrix Cell State":  k_t is scaled by 1/sqrt(d_qk);
 *       C_t = f_t C_{t-1} + i_t v_t k_t^T,  n_t = f_t n_{t-1} + i_t k_t,
 *       h_t = C_t q_t / max(|n_t^T q_t|, exp(-m_t))          (stabilised form);
 *   section 2 "The Normalizer State and Numerical Stabilization": the log-space max
 *       stabiliser m_t = max(log f_t + m_{t-1}, i~_t), with i_t = exp(i~_t) and the
 *       sigmoid forget gate used in log space, log f_t = log sigmoid(f~_t) (or, with
 *       MLSTM_FORGET_EXP, the exponential gate: log f_t = f~_t);
 *   section 3 "The Parallel Dual Form" and section 5 (chunkwise scans): the forward is
 *       computed chunk by chunk -- the quadratic form inside each chunk, the recurrent
 *       state (C, n, m) passed across chunks;
 *   section 5 "Inference Memory and Throughput Trade-Offs": decoding carries only the
 *       constant-size state (C, n, m), updated in place one token at a time.
 *
 * Conventions for every entry point
 *   - Every array pointer is DEVICE memory owned by the caller; the library allocates
 *     nothing and keeps no state between calls.
 *   - All arrays are contiguous row-major with the layouts given below; every pointer
 *     must be 16-byte aligned.
 *   - q, k, v are given in `dt` (MLSTM_F32 or MLSTM_BF16); k is passed UNSCALED and the
 *     library applies 1/sqrt(DQK).  The gate pre-activations and every state array are
 *     float32.  h is written in `h_dt`.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream) and
 *     the call returns without synchronising.  Argument errors are detected on the host
 *     and returned before anything is launched; a failed launch returns MLSTM_ERR_LAUNCH.
 *   - Layout of the state: C[b][h][a][c] accumulates v_a * k_c (d_v rows, d_qk columns),
 *     n[b][h][c], m[b][h].  (C, n) are stored relative to the stabiliser: the
 *     unstabilised state is C * exp(m).
 *
 * Supported sizes: B, NH >= 1; S >= 0 with S % chunk == 0; chunk in {16, 32, 64, 128};
 * DQK and DV multiples of 32 in [32, 512].
 */
#ifndef MLSTM_B300_H
#define MLSTM_B300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLSTM_OK = 0,
  MLSTM_ERR_NULL = 1,      /* a required pointer is NULL */
  MLSTM_ERR_ALIGN = 2,     /* a pointer is not 16-byte aligned */
  MLSTM_ERR_SHAPE = 3,     /* a size is outside the supported set, or S % chunk != 0 */
  MLSTM_ERR_DTYPE = 4,     /* unsupported dtype code */
  MLSTM_ERR_WORKSPACE = 5, /* workspace smaller than mlstm_fwd_workspace_bytes() */
  MLSTM_ERR_LAUNCH = 6,    /* a kernel launch failed (see mlstm_last_cuda_error) */
  MLSTM_ERR_TIMEOUT = 7,   /* a bounded device-side wait gave up (reported by a kernel) */
  MLSTM_ERR_DEVICE = 8     /* no usable device, or the device is not sm_103 */
} mlstm_status;

/* Element type of q, k, v (and of h in h_dt).  The calls that read raw gate pre-activations
 * (mlstm_fwd_chunkwise, mlstm_fwd_chunkwise_noalloc, mlstm_fwd_chunk_states, mlstm_step,
 * mlstm_step_multi) also take MLSTM_FORGET_EXP OR-ed into `dt`: the forget gate is then the
 * exponential variant f_t = exp(f~_t), log f_t = f~_t (section 2 of the page allows "exp or
 * sigmoid"; the default is sigmoid).  The sizing and path queries accept and ignore it;
 * mlstm_fwd_from_gates uses whatever variant filled its workspace; mlstm_fwd_gates (which
 * has no dtype argument) is the sigmoid variant only.  In C++ the combined value needs a
 * cast: (mlstm_dtype)(MLSTM_BF16 | MLSTM_FORGET_EXP). */
typedef enum { MLSTM_F32 = 0, MLSTM_BF16 = 1, MLSTM_FORGET_EXP = 0x100 } mlstm_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char *mlstm_status_str(mlstm_status s);

/* The cudaError_t value (as int) behind the last MLSTM_ERR_LAUNCH returned on the calling
 * host thread, 0 if there was none.  The CUDA error itself has been consumed. */
int mlstm_last_cuda_error(void);

/* Number of kernels this library has launched in the process so far (all host threads);
 * the difference across a region counts the library's launches inside it. */
unsigned long long mlstm_kernel_launches(void);

/* Which kernels mlstm_fwd_chunkwise runs for these sizes:
 * 1 = the fused tensor-core kernel, one CTA per (head, 128 rows of d_v);
 * 2 = the same kernel with each head's d_qk split over a pair of CTAs (a thread-block
 *     cluster exchanging partial sums through distributed shared memory) -- always for
 *     d_qk = 512, and for smaller heads when the single-CTA grid would leave SMs idle;
 *     (both: bf16 inputs, S a multiple of 64, d_qk in {64, 128, 256, 512}, d_v a multiple
 *     of 128; the kernel walks the sequence in its own chunks of 64 tokens whatever `chunk`
 *     asks for -- the result is the same function up to rounding)
 * 0 = the CUDA-core kernels (every other supported size), -1 = unsupported sizes or dtype.
 * mlstm_fwd_from_gates runs the fused kernel only for chunk 64 (its workspace holds the gate
 * preprocessing of the asked-for chunk) and the CUDA-core kernels otherwise. */
int mlstm_fwd_path(int B, int NH, int S, int DQK, int DV, int chunk, mlstm_dtype dt);

/* Bytes of device workspace mlstm_fwd_chunkwise, mlstm_fwd_chunk_states and mlstm_fwd_gates
 * need for these sizes (0 if the sizes are unsupported), on the path mlstm_fwd_chunkwise takes
 * (mlstm_fwd_path): the fused tensor-core kernel materialises no boundary states, so its
 * workspace is small whatever chunk is asked for; the CUDA-core kernels keep every
 * chunk-boundary state.  The workspace holds the wait-error word at offset 0, the per-token
 * gate prefix sums, the per-chunk stabiliser and, on the CUDA-core path, the boundary states.
 * Its contents are scratch: nothing is read back by the caller except through mlstm_fwd_check.
 * mlstm_fwd_from_gates takes the fused kernel only for chunk 64; for another chunk on sizes
 * the fused kernel would take, it runs the CUDA-core kernels and needs their larger workspace,
 * which mlstm_fwd_workspace_bytes(..., MLSTM_F32) returns (the layout does not depend on the
 * element type).  On the fused path, sizes whose grid would leave most SMs idle (long
 * sequences over few heads, see mlstm_fwd_segments) also get the sequence-parallel buffers:
 * per head and segment one float32 state C, n, m for the segment's own map and one for its
 * entering state (the long-context layer, B=1 NH=8 S=16384 d=256, about 18 MB in all).
 * bf16 heads with d_qk = 512 over at most 64 chunks of 64 tokens (and no sequence segments)
 * also get the buffers of the forward in five kernels: per token beta q and w k in fp16 (2 x
 * d_qk halves), a row of P in fp16 (64 halves) and eight floats, per chunk the n increment
 * (d_qk floats) and eight floats -- about 74 MB for the 1.3B-style layer (B=4 NH=4 S=2048).
 * With them the forward runs as: per head the gate prefix sums, stabiliser chain and token
 * factors; per (head, chunk) Q K^T on tensor cores with P, its row sums, beta q, w k and the n
 * increment (section 3 "The Parallel Dual Form": the in-chunk matrix and the chunk's state
 * update operands, which every d_v tile of a head shares); n entering each chunk; every
 * token's 1/den; then the state walk with the products U, X and P V only.  The result is the
 * same function up to rounding (the same state recurrence: C, n, m agree with the single
 * fused kernel to fp32 rounding). */
size_t mlstm_fwd_workspace_bytes(int B, int NH, int S, int DQK, int DV, int chunk,
                                 mlstm_dtype dt);

/* The least workspace mlstm_fwd_chunkwise accepts for these sizes (0 if unsupported): that of
 * mlstm_fwd_workspace_bytes without the sequence-parallel buffers or the five-kernel
 * forward's buffers.  A workspace below mlstm_fwd_workspace_bytes runs the forward over whole
 * sequences in the single fused kernel, one head at a time per CTA (or CTA pair). */
size_t mlstm_fwd_workspace_min_bytes(int B, int NH, int S, int DQK, int DV, int chunk,
                                     mlstm_dtype dt);

/* How many segments of each head's sequence mlstm_fwd_chunkwise runs in parallel for these
 * sizes with a workspace of `ws_bytes` (an addition of this library for long sequences over
 * few heads; the pages' chunkwise form walks each sequence in one pass).  The segments'
 * maps compose exactly -- section 3 "The Parallel Dual Form" (the state after a stretch of
 * tokens is the sum of its tokens' decayed contributions, so stretches compose by an
 * associative scan) and section 2 (the stabiliser recurrence is max-plus linear in m): a first
 * pass runs every segment from the zero state with m = -inf (segment 0 from the caller's
 * initial state), a scan forms the entering state of every segment and the final state, and
 * a second pass reruns segments 1..G-1 from their entering states.  The result is the same
 * function up to rounding.  Returns G = 1 (no split: the CUDA-core path, raw-gate-free
 * mlstm_fwd_from_gates, grids that already fill the GPU, or a workspace without the buffers),
 * a power of two G > 1 with S divisible by 64 G and at least 256 tokens per segment, or -1 for
 * unsupported sizes or dtype.  The choice depends on the device's SM count. */
int mlstm_fwd_segments(int B, int NH, int S, int DQK, int DV, int chunk, mlstm_dtype dt,
                       size_t ws_bytes);

/* Chunkwise forward of the mLSTM cell over a whole sequence (section 3 "The Parallel Dual
 * Form", chunked; section 2 stabiliser).
 *   q, k     [B, NH, S, DQK]  (dt)          v        [B, NH, S, DV]   (dt)
 *   igate_pre, fgate_pre  [B, NH, S] float32: the gate pre-activations i~_t and f~_t
 *   C_init [B,NH,DV,DQK], n_init [B,NH,DQK], m_init [B,NH] float32: the state the
 *       sequence continues from; all three NULL = the zero state with m_0 = 0 (either
 *       all NULL or none).
 *   h      [B, NH, S, DV]  (h_dt) output: h~_t for every token
 *   C_last [B,NH,DV,DQK], n_last [B,NH,DQK], m_last [B,NH] float32 outputs: the state
 *       after the last token (may alias C_init/n_init/m_init for an in-place update).
 *   workspace: at least mlstm_fwd_workspace_min_bytes(...) bytes of device memory;
 *       mlstm_fwd_workspace_bytes(...) bytes enable the sequence-parallel forward where it
 *       applies (mlstm_fwd_segments) and the five-kernel forward of d_qk = 512 heads (see
 *       mlstm_fwd_workspace_bytes).
 * S == 0 copies the initial state to the outputs. */
mlstm_status mlstm_fwd_chunkwise(const void *q, const void *k, const void *v,
                                 const float *igate_pre, const float *fgate_pre, int B, int NH,
                                 int S, int DQK, int DV, int chunk, mlstm_dtype dt,
                                 const float *C_init, const float *n_init, const float *m_init,
                                 void *h, mlstm_dtype h_dt, float *C_last, float *n_last,
                                 float *m_last, void *workspace, size_t ws_bytes, void *stream);

/* The two stages of mlstm_fwd_chunkwise, for callers that time or schedule them apart:
 * mlstm_fwd_gates (below) runs the gate preprocessing into `workspace`; then
 * mlstm_fwd_from_gates runs everything after it (state passing and output) on that
 * workspace.  Both calls must use the same sizes, chunk, workspace and m_init, in stream
 * order; C_init and n_init (both NULL or both given) belong to this second call.  Arguments
 * and outputs are those of mlstm_fwd_chunkwise. */
mlstm_status mlstm_fwd_from_gates(const void *q, const void *k, const void *v, int B, int NH,
                                  int S, int DQK, int DV, int chunk, mlstm_dtype dt,
                                  const float *C_init, const float *n_init, void *h,
                                  mlstm_dtype h_dt, float *C_last, float *n_last, float *m_last,
                                  void *workspace, size_t ws_bytes, void *stream);

/* The inter-chunk recurrence alone (gate preprocessing + state passing), materialising
 * the state at every chunk boundary:
 *   C_states [B, NH, NC+1, DV, DQK], n_states [B, NH, NC+1, DQK], m_states [B, NH, NC+1]
 * with NC = S / chunk; entry j is the state after j*chunk tokens (entry 0 = the initial
 * state, entry NC = the final state).  Other arguments as for mlstm_fwd_chunkwise. */
mlstm_status mlstm_fwd_chunk_states(const void *k, const void *v, const float *igate_pre,
                                    const float *fgate_pre, int B, int NH, int S, int DQK,
                                    int DV, int chunk, mlstm_dtype dt, const float *C_init,
                                    const float *n_init, const float *m_init, float *C_states,
                                    float *n_states, float *m_states, void *workspace,
                                    size_t ws_bytes, void *stream);

/* Gate preprocessing alone (kernel a): fills `workspace` with the per-token gate prefix
 * quantities and the per-chunk stabiliser (the input of mlstm_fwd_from_gates), and writes
 * the stabiliser m_t of every token, m_tok [B, NH, S], and of every chunk boundary,
 * m_states [B, NH, NC+1] (entry 0 = m_init or 0).  Either output may be NULL.  The
 * workspace must hold at least mlstm_fwd_workspace_bytes(B, NH, S, 32, 32, chunk, dt). */
mlstm_status mlstm_fwd_gates(const float *igate_pre, const float *fgate_pre, int B, int NH,
                             int S, int chunk, const float *m_init, float *m_tok,
                             float *m_states, void *workspace, size_t ws_bytes, void *stream);

/* Synchronises `stream` and reports whether the last forward that used `workspace` completed
 * every bounded device-side wait: MLSTM_OK, or MLSTM_ERR_TIMEOUT when a kernel gave up waiting
 * (mlstm_last_cuda_error() then returns the kernel's wait code).  The word it reads sits at
 * offset 0 of every forward workspace and every forward clears it before its kernels run, so
 * the answer concerns the last forward whatever its path or chunk; the size arguments are only
 * validated, and ws_bytes must be at least 256. */
mlstm_status mlstm_fwd_check(const void *workspace, size_t ws_bytes, int B, int NH, int S, int DQK,
                             int DV, int chunk, mlstm_dtype dt, void *stream);

/* Exercises the failure path of the bounded device-side waits (no counterpart on the pages; a
 * test hook for the fault handling): launches one CTA that runs the fused forward's wait on a
 * barrier nothing ever completes.  After about a second the wait gives up and records
 * MLSTM_SELFTEST_WAIT_CODE in the error word (offset 0) of `workspace`, exactly as a forward's
 * wait would; mlstm_fwd_check on the same workspace then returns MLSTM_ERR_TIMEOUT and
 * mlstm_last_cuda_error() the code.  Nothing faults, traps or hangs, and the device stays
 * usable.  Do not run it while a forward uses the same workspace.  ws_bytes >= 256. */
#define MLSTM_SELFTEST_WAIT_CODE 90
mlstm_status mlstm_wait_selftest(void *workspace, size_t ws_bytes, int B, int NH, int S, int DQK, int DV,
                                 int chunk, mlstm_dtype dt, void *stream);

/* One recurrent decode step for every (batch, head), in place (section 5 "Inference
 * Memory and Throughput Trade-Offs"; section 2 stabiliser; section 3 updates):
 *   q, k [B, NH, DQK] (dt), v [B, NH, DV] (dt), ig, fg [B, NH] float32 pre-activations
 *   C [B, NH, DV, DQK], n [B, NH, DQK], m [B, NH] float32: read, then overwritten with
 *       the state after this token
 *   h [B, NH, DV] (h_dt) output. */
mlstm_status mlstm_step(const void *q, const void *k, const void *v, const float *ig,
                        const float *fg, float *C, float *n, float *m, void *h, int B, int NH,
                        int DQK, int DV, mlstm_dtype dt, mlstm_dtype h_dt, void *stream);

/* T consecutive decode steps in one launch, in place (section 5 "Inference Memory and Throughput
 * Trade-Offs"; section 2 stabiliser; section 3 updates): exactly the results of T calls to
 * mlstm_step on tokens t = 0..T-1 in order, but the state C is read and written once for the T
 * tokens instead of T times (for speculative decoding or short prompt extensions).
 *   q, k [B, NH, T, DQK] (dt), v [B, NH, T, DV] (dt), ig, fg [B, NH, T] float32
 *   C [B, NH, DV, DQK], n [B, NH, DQK], m [B, NH] float32: read, then overwritten with the
 *       state after the T-th token
 *   h [B, NH, T, DV] (h_dt) output: h for every token.
 * 1 <= T <= 16; other sizes as for mlstm_step. */
mlstm_status mlstm_step_multi(const void *q, const void *k, const void *v, const float *ig,
                              const float *fg, float *C, float *n, float *m, void *h, int B, int NH,
                              int T, int DQK, int DV, mlstm_dtype dt, mlstm_dtype h_dt, void *stream);

/* The mLSTM block's step after the cell (section 4 "xLSTM Block Architecture and Residual
 * Stacking", the mLSTM block's item 5 "Group Normalization and Output Gating"; section 3
 * "Associative Matrix Cell State": h_t = o_t (.) h~_t).  For every (batch, head, token) row of
 * DV channels, with the head as the normalisation group:
 *   mu = mean_c h~_c, var = mean_c (h~_c - mu)^2 (biased),
 *   y_c = sigmoid(o~_c) * (gamma_c (h~_c - mu) / sqrt(var + eps) + beta_c)
 *   h  [B, NH, S, DV] (h_dt): the cell output h~, e.g. mlstm_fwd_chunkwise's h
 *   o_pre [B, NH, S, DV] (o_dt): the output-gate pre-activations o~
 *   gamma, beta [NH, DV] float32: per-channel scale and shift
 *   y  [B, NH, S, DV] (y_dt) output; y may be h itself when y_dt == h_dt (each row is read
 *      completely before it is written).
 * eps > 0.  DV a multiple of 32 in [32, 512]; S >= 0 (S = 0 launches nothing).  The pages do
 * not fix the gate's form or the epsilon: the sigmoid output gate of the LSTM and the caller's
 * eps are used.  Memory bound: one read of h and o_pre and one write of y. */
mlstm_status mlstm_groupnorm_gate(const void *h, const void *o_pre, const float *gamma, const float *beta,
                                  float eps, void *y, int B, int NH, int S, int DV, mlstm_dtype h_dt,
                                  mlstm_dtype o_dt, mlstm_dtype y_dt, void *stream);

/* Backward of mlstm_fwd_chunkwise (section 3 "The Parallel Dual Form": the parallel form is the
 * one trained; "Associative Matrix Cell State" for the updates and the retrieval; section 2 for
 * the stabiliser, which rescales C and n by exp(-m_t) and changes no value of h, so the
 * gradients are those of the unstabilised cell).  For L = sum_t dh_t . h_t with h from
 * mlstm_fwd_chunkwise on the same inputs:
 *   dq, dk [B,NH,S,DQK], dv [B,NH,S,DV] (dt) outputs: dL/dq, dL/dk (k as passed, unscaled),
 *       dL/dv;
 *   dig, dfg [B,NH,S] float32 outputs: dL/di~ and dL/df~ (through log sigmoid(f~), or f~ itself
 *       with MLSTM_FORGET_EXP OR-ed into dt);
 *   dC_init [B,NH,DV,DQK], dn_init [B,NH,DQK], dm_init [B,NH] float32 outputs (all three or
 *       none): dL/d of the initial state as the forward takes it (C_init, n_init relative to
 *       m_init; dm_init = <dC_init, C_init> + dn_init . n_init, zero without an initial state).
 *   dh [B,NH,S,DV] (dt): dL/dh.  Other inputs as for mlstm_fwd_chunkwise (same chunk rules).
 * Where |n_t . q_t| equals exp(-m_t) exactly, h has a kink; the derivative taken there treats
 * the floor as the active branch.  The forward is recomputed inside (gate preprocessing,
 * boundary states, per-token denominators), so no forward output is needed.  For bf16 inputs
 * with chunk 64 or 128, d_qk in {64, 128, 256, 512} and d_v a multiple of 128, the boundary and
 * adjoint state walks run on tensor cores (fp16 operands, fp32 accumulation) and, with d_qk a
 * multiple of 128 too, so do the products of the tokens with those states (tf32); the chunk-local
 * L x L work runs on CUDA cores in fp32, as does everything for other sizes.  The tensor-core
 * kernels' bounded device-side waits record into the error word at offset 0 of the workspace,
 * which mlstm_fwd_check reads (pass the backward's workspace and sizes).
 * workspace: at least mlstm_bwd_workspace_bytes(...) bytes. */
size_t mlstm_bwd_workspace_bytes(int B, int NH, int S, int DQK, int DV, int chunk, mlstm_dtype dt);
mlstm_status mlstm_bwd_chunkwise(const void *q, const void *k, const void *v,
                                 const float *igate_pre, const float *fgate_pre, const void *dh,
                                 int B, int NH, int S, int DQK, int DV, int chunk, mlstm_dtype dt,
                                 const float *C_init, const float *n_init, const float *m_init,
                                 void *dq, void *dk, void *dv, float *dig, float *dfg,
                                 float *dC_init, float *dn_init, float *dm_init, void *workspace,
                                 size_t ws_bytes, void *stream);

/* Forward without any device allocation (no counterpart on the source pages: an interface
 * addition of this library).
 *
 * Some callers cannot allocate device memory for a workspace: a plugin running inside a host
 * application that owns all device memory through its own pool (an extra cudaMalloc would
 * fail or fragment it), or a latency-critical serving loop where cudaMalloc/cudaFree may
 * synchronise the device.  This entry point takes the same arguments as mlstm_fwd_chunkwise
 * minus the workspace, and computes exactly the same outputs; its scratch is a fixed array
 * of MLSTM_NOALLOC_SCRATCH_BYTES bytes inside the library's device image, which every GPU
 * that loads the library holds until the process exits.  Nothing is allocated by the call:
 * no cudaMalloc, no cudaFree, no allocating library routine.
 *   - Sizes whose mlstm_fwd_workspace_min_bytes(...) exceeds MLSTM_NOALLOC_SCRATCH_BYTES are
 *     rejected with MLSTM_ERR_WORKSPACE before anything is launched.  That is the workspace of
 *     the path the forward takes: the 1.3B-style layer (B=4 NH=4 S=2048 d=512 bf16 chunk 64)
 *     needs about 0.43 MB and the long-context layer (B=1 NH=8 S=16384 d=256 bf16 chunk 128)
 *     about 1.6 MB; sizes that take the CUDA-core path materialise boundary states and fit
 *     only when small.  The array is passed on as a workspace of MLSTM_NOALLOC_SCRATCH_BYTES
 *     bytes, so the sequence-parallel forward runs where its buffers fit in it
 *     (mlstm_fwd_segments with that size says which) and the outputs are those of
 *     mlstm_fwd_chunkwise with a workspace of that size.
 *   - A bounded device-side wait that gave up inside this forward is reported, as for the
 *     workspace forward, by mlstm_fwd_check_noalloc (below).
 *   - The first call on a device resolves the array's device address on that device (with
 *     it current, cudaGetSymbolAddress); make that first call before any stream capture.
 *   - Every call in the process shares the one array: calls whose work may overlap on the
 *     GPU (different streams, or different host threads, without ordering) race on it and
 *     must be serialised by the caller.  Stale contents left by an earlier call are harmless:
 *     the forward rewrites all it reads and clears what must start at zero.
 * Other arguments, outputs and errors as for mlstm_fwd_chunkwise. */
#define MLSTM_NOALLOC_SCRATCH_BYTES (8u << 20)
mlstm_status mlstm_fwd_chunkwise_noalloc(const void *q, const void *k, const void *v,
                                         const float *igate_pre, const float *fgate_pre, int B,
                                         int NH, int S, int DQK, int DV, int chunk,
                                         mlstm_dtype dt, const float *C_init,
                                         const float *n_init, const float *m_init, void *h,
                                         mlstm_dtype h_dt, float *C_last, float *n_last,
                                         float *m_last, void *stream);

/* mlstm_fwd_check for the forward without allocation (no counterpart on the pages): synchronises
 * `stream` and reports whether the last mlstm_fwd_chunkwise_noalloc on the current device
 * completed every bounded device-side wait (MLSTM_OK or MLSTM_ERR_TIMEOUT, as mlstm_fwd_check).
 * It reads the error word of the library's fixed scratch array and allocates nothing. */
mlstm_status mlstm_fwd_check_noalloc(void *stream);

/* The device address (and, if `bytes` is not NULL, the size, MLSTM_NOALLOC_SCRATCH_BYTES) of
 * the fixed scratch array behind mlstm_fwd_chunkwise_noalloc on the current device (no
 * counterpart on the pages).  The first query on a device resolves the address, with that
 * device current, as the first forward call would.  The array belongs to the library: a caller
 * may read it (or point mlstm_wait_selftest at it to exercise mlstm_fwd_check_noalloc), but
 * anything it writes there may be overwritten by the next forward without allocation. */
mlstm_status mlstm_noalloc_scratch(void **ptr, size_t *bytes);

#ifdef __cplusplus
}
#endif

#endif /* MLSTM_B300_H */
