// states_tc.cu -- chunk-boundary states of a decayed rank-L recurrence on tensor cores.
//
// Page "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural Networks"
// (llms.blog), section 3 "Associative Matrix Cell State" (C_t = f_t C_{t-1} + i_t v_t k_t^T,
// n_t = f_t n_{t-1} + i_t k_t) unrolled over a chunk as in "The Parallel Dual Form", with the
// section 2 stabiliser.  Over chunks of L tokens, in either direction along the sequence:
//   T <- alpha_k T + X_k^T diag(omega) Y_k,     n <- alpha_k n + Y_k^T omega'
// where X is [S, DV] and Y is [S, DQK] (bf16, token-major) and omega, omega' are per-token
// weights.  Walked forwards with X = v, Y = k and the forward's state-update weights this is the
// inter-chunk recurrence (the boundary states C^(k), n^(k)); walked backwards with X = dh, Y = q
// and the backward's weights it is the adjoint recurrence (G^(k), N^(k)).
//
// One CTA per (128 rows of DV, half of DQK when DQK >= 128, head): T lives in tensor memory
// (128 lanes x the CTA's DQK fp32 columns, twice where it fits),
// each 64-token slab of X and Y arrives by TMA, is converted in place to fp16 (X scaled by its
// token's weight) and enters T with four K = 16 tcgen05 MMAs per 128 x min(DQK, 256) block.
// At every chunk boundary the epilogue warps read T, store the boundary state and write back
// T scaled for the next chunk.  fp16 has a narrow range, so each chunk's weights are divided by
// a power of two s_k >= their maximum (exact) and T is carried divided by the current chunk's
// s_k: the epilogue multiplies by alpha_k s_{k-1} / s_k when it rescales.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.cuh"
#include "sm100.cuh"
#include "tmap.cuh"

namespace mlstm {

namespace {
using namespace sm100;

constexpr int kSub = 64;      // tokens per slab (one TMA stage)
constexpr int kTileM = 128;   // rows of DV per CTA (tensor-memory lanes)
// slabs in flight: four (two chunks of 128 tokens) where shared memory allows, else two
template <int NQ>
__host__ __device__ constexpr int stages_for() { return NQ <= 4 ? 4 : 2; }
constexpr int kEpiT = 256;   // epilogue threads (warps 2-9)
constexpr int kConvT = 128;  // conversion threads (warps 10-13)
constexpr int kThreadsT = 64 + kEpiT + kConvT;
// warp 0: TMA loads; warp 1: tensor-memory allocation and MMA issue; warps 2-9: epilogue (warp
// w reads tensor-memory lanes 32 (w % 4) .. + 31, warps w and w + 4 taking alternate 32-column
// blocks, so that two warps share each quarter's state stores); warps 10-13: conversion and n.

template <int NQ>  // the CTA's columns of d_qk / 64
struct alignas(1024) StatesSmem {
  static constexpr int ST = stages_for<NQ>();
  unsigned char tile[ST][(2 + NQ) * 8192];  // X boxes 0, 1 then NQ Y boxes, 64 x 128 B each
  uint64_t full[ST], conv[ST], empty[ST];
  uint64_t mma_done, epi_ready, fin;
  float wx[ST][64];  // the slab's X weights
  float wn[ST][64];  // the slab's n weights
  uint32_t tmem_base;
  int abort_flag;
  int conv_fail;  // written by the conversion warps only, read by them after a barrier
  int epi_fail;   // the epilogue warps' first failed chunk (-1: none), read by them after a barrier
};

__device__ __forceinline__ bool st_aborted(const int *f) { return *(const volatile int *)f != 0; }
__device__ __forceinline__ void st_set_abort(int *f) { *(volatile int *)f = 1; }

template <int NQ>
__global__ void __launch_bounds__(kThreadsT, 1) states_tc_kernel(
    const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapY, const float *__restrict__ wx,
    const float *__restrict__ wn, const float *__restrict__ alpha, const float *__restrict__ sc, int S, int L,
    int DV, int reverse, const float *__restrict__ C0, const float *__restrict__ n0, float *__restrict__ states,
    float *__restrict__ nstates, float *__restrict__ C_fin, float *__restrict__ n_fin, int *__restrict__ err,
    float *__restrict__ states_t, int DQKt, int CS) {
  constexpr int DQK = 64 * NQ;  // this CTA's columns: [cb, cb + DQK) of the state's DQKt
  constexpr int NN = DQK > 256 ? 2 : 1;  // MMAs per K step (N <= 256 each)
  constexpr int NB = DQK / NN;           // N of each
  // two state buffers where tensor memory has room (d_qk <= 256): the products of chunk k then
  // accumulate into one while the epilogue stores the state held in the other
  constexpr bool PP = 2 * DQK <= 512;
  constexpr uint32_t kCols = PP ? 2 * DQK : DQK;
  constexpr int ST = stages_for<NQ>();
  extern __shared__ unsigned char st_raw[];
  StatesSmem<NQ> &sm = *reinterpret_cast<StatesSmem<NQ> *>(
      (reinterpret_cast<uintptr_t>(st_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA = (128 rows of DV, one of CS column blocks, head)
  const int p = blockIdx.y, a0 = (blockIdx.x / CS) * kTileM, cb = (blockIdx.x % CS) * DQK;
  const int NC = S / L, SUB = L / kSub, NS = S / kSub;
  // without per-chunk factors the walk keeps only the final state: the weights already carry
  // each token's decay to the end of the sequence (no rescaling between chunks, no stores)
  const bool final_only = alpha == nullptr;
  int *abort_ptr = &sm.abort_flag;
  // slab j (in walking order) is slab sub(j) of the sequence; chunk i of the walk is chunk kc(i)
  auto kc_of = [&](int i) { return reverse ? NC - 1 - i : i; };
  auto sub_of = [&](int j) {
    const int i = j / SUB, r = j % SUB;
    return kc_of(i) * SUB + r;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.conv[s], kConvT);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.mma_done, 1);
    mbar_init(&sm.epi_ready, kEpiT);
    mbar_init(&sm.fin, 1);
    sm.abort_flag = 0;
    sm.conv_fail = 0;
    sm.epi_fail = -1;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = sm.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA loads
    if (lane == 0) {
      prefetch_tensormap(&mapX);
      prefetch_tensormap(&mapY);
      int issued = 0;
      for (int j = 0; j < NS; ++j) {
        const int s = j % ST;
        if (j >= ST && !mbar_wait(&sm.empty[s], ((j / ST) - 1) & 1, err, 41, abort_ptr)) break;
        if (st_aborted(abort_ptr)) break;
        const int row = p * S + sub_of(j) * kSub;
        mbar_arrive_expect_tx(&sm.full[s], (uint32_t)(2 + NQ) * 8192u);
        tma_load_2d(sm.tile[s], &mapX, a0, row, &sm.full[s]);
        tma_load_2d(sm.tile[s] + 8192, &mapX, a0 + 64, row, &sm.full[s]);
        for (int q = 0; q < NQ; ++q)
          tma_load_2d(sm.tile[s] + (2 + q) * 8192, &mapY, cb + 64 * q, row, &sm.full[s]);
        issued = j + 1;
      }
      // nothing may leave while loads it issued are still landing
      for (int j = issued > ST ? issued - ST : 0; j < issued; ++j)
        mbar_wait(&sm.full[j % ST], (j / ST) & 1, err, 49);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t id = idesc_f16(kTileM, NB, /*f16*/ 0, /*a MN-major*/ 1, /*b MN-major*/ 1);
      int j = 0;
      bool ok = true;
      for (int i = 0; i < NC && ok; ++i) {
        if (!final_only && !mbar_wait(&sm.epi_ready, i & 1, err, 42, abort_ptr)) {
          ok = false;
          break;
        }
        for (int r = 0; r < SUB; ++r, ++j) {
          const int s = j % ST;
          if (!mbar_wait(&sm.conv[s], (j / ST) & 1, err, 43, abort_ptr)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dx = smem_desc(smem_u32(sm.tile[s]), 8192, 1024, kSwizzle128B);
          const uint64_t dy = smem_desc(smem_u32(sm.tile[s] + 2 * 8192), 8192, 1024, kSwizzle128B);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
#pragma unroll
            for (int h = 0; h < NN; ++h)
              mma_f16_ss(tm + (PP && !final_only ? (uint32_t)(((i + 1) & 1) * DQK) : 0u) + h * NB,
                         dx + (uint64_t)(ks * 2048 >> 4),
                         dy + (uint64_t)((ks * 2048 + h * (NB / 64) * 8192) >> 4), id,
                         final_only ? ((j | ks) != 0) : 1);
          mma_commit(&sm.empty[s]);
        }
        if (ok && !final_only) mma_commit(&sm.mma_done);
      }
      if (ok && final_only) mma_commit(&sm.mma_done);
      if (!ok) st_set_abort(abort_ptr);
      mma_commit(&sm.fin);  // completes once every MMA issued above has finished
      mbar_wait(&sm.fin, 0, err, 48);
    }
  } else if (warp < 2 + kEpiT / 32) {
    // ------------------------------------------------------------------ epilogue
    const int row = 32 * (warp & 3) + lane;  // the tensor-memory lane this thread may access
    const uint32_t trow = tm + ((uint32_t)(32 * (warp & 3)) << 16);
    const int cfirst = 32 * ((warp - 2) >> 2);  // this warp's first 32-column block; step 64
    float s_prev = 1.f;
    bool ok = true;
    if (final_only) {
      // one read of T after the last slab: the final state
      const bool got = __all_sync(0xffffffffu, mbar_wait(&sm.mma_done, 0, err, 44, abort_ptr));
      if (got) {
        tc_fence_after();
        for (int c0 = cfirst; c0 < DQK; c0 += 64) {
          uint32_t r[32];
          tmem_ld32(trow + c0, r);
          tmem_wait_ld();
          float *dst = C_fin + ((size_t)p * DV + a0 + row) * DQKt + cb + c0;
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4 *>(dst + e) = make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]),
                                                               __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
        }
      } else {
        ok = false;
      }
    }
    // the chunk's decay and scale, loaded one chunk ahead (they sit on the serial chain)
    float a_nxt = !final_only && NC > 0 ? alpha[(size_t)p * NC + kc_of(0)] : 0.f;
    float s_nxt = !final_only && NC > 0 ? sc[(size_t)p * NC + kc_of(0)] : 1.f;
    for (int i = 0; i <= NC && ok && !final_only; ++i) {
      const int b_in = reverse ? NC - i : i;  // boundary whose state T holds now
      const float s_cur = i < NC ? s_nxt : 1.f, a_cur = a_nxt;
      if (i + 1 < NC) {
        a_nxt = alpha[(size_t)p * NC + kc_of(i + 1)];
        s_nxt = sc[(size_t)p * NC + kc_of(i + 1)];
      }
      if (i > 0) {
        // all four warps take the same branch (they meet at named barriers below), each warp as a
        // whole before its collective tensor-memory loads
        const bool got = __all_sync(0xffffffffu, mbar_wait(&sm.mma_done, (i - 1) & 1, err, 44, abort_ptr));
        // (the chunk index, not a flag: a warp that fails at chunk i + 1 before a slower warp has
        // read the word for chunk i must not stop that warp one chunk early)
        if (!got) atomicCAS(&sm.epi_fail, -1, i);
        named_barrier_sync(2, kEpiT);
        const int failed = *(volatile int *)&sm.epi_fail;
        if (failed >= 0 && failed <= i) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      // buffers: the state entering chunk i sits in buffer i % 2, the products of chunk i go into
      // the other (one buffer without room for two)
      const uint32_t tcur = trow + (PP ? (uint32_t)((i & 1) * DQK) : 0u);
      const uint32_t tnxt = trow + (PP ? (uint32_t)(((i + 1) & 1) * DQK) : 0u);
      // the state at boundary b_in, 32 columns at a time (in its own stabiliser frame)
      auto state_piece = [&](int c0, float (&v)[32]) {
        if (i == 0) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            v[e] = C0 ? C0[((size_t)p * DV + a0 + row) * DQKt + cb + c0 + e] : 0.f;
        } else {
          uint32_t r[32];
          tmem_ld32(tcur + c0, r);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]) * s_prev;
        }
      };
      // T for the next chunk: alpha_k times the state, in units of s_k
      auto rescale_piece = [&](int c0, const float (&v)[32]) {
        uint32_t r[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(v[e] * (a_cur / s_cur));
        tmem_st16(tnxt + c0, *reinterpret_cast<uint32_t(*)[16]>(&r[0]));
        tmem_st16(tnxt + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&r[16]));
      };
      auto store_piece = [&](int c0, const float (&v)[32]) {
        if (states) {
          float *dst = states + ((size_t)(p * (NC + 1) + b_in) * DV + a0 + row) * DQKt + cb + c0;
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4 *>(dst + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
        if (i == NC && C_fin) {
          float *dst = C_fin + ((size_t)p * DV + a0 + row) * DQKt + cb + c0;
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4 *>(dst + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
        if (states_t) {
          // the transposed state [DQK][DV]: for each column the warp's 32 rows are contiguous
          float *dt = states_t + ((size_t)p * (NC + 1) + b_in) * (size_t)DQKt * DV + (size_t)(cb + c0) * DV + a0 + row;
#pragma unroll
          for (int e = 0; e < 32; ++e) dt[(size_t)e * DV] = v[e];
        }
      };
      if (PP) {
        // the next chunk's T first, so that its products start while this state is stored
        if (i < NC) {
          for (int c0 = cfirst; c0 < DQK; c0 += 64) {
            float v[32];
            state_piece(c0, v);
            rescale_piece(c0, v);
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&sm.epi_ready);
        }
        for (int c0 = cfirst; c0 < DQK; c0 += 64) {
          float v[32];
          state_piece(c0, v);
          store_piece(c0, v);
        }
      } else {
        for (int c0 = cfirst; c0 < DQK; c0 += 64) {
          float v[32];
          state_piece(c0, v);
          store_piece(c0, v);
          if (i < NC) rescale_piece(c0, v);
        }
      }
      if (i < NC) {
        if (!PP) {
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&sm.epi_ready);
        }
        s_prev = s_cur;
      }
    }
    if (!ok) st_set_abort(abort_ptr);
  } else {
    // ------------------------------------------------------------------ conversion and n
    const int ct = threadIdx.x - 64 - kEpiT;  // 0 .. kConvT - 1
    const bool do_n = blockIdx.x < CS && (nstates != nullptr || n_fin != nullptr);  // the first rows' CTAs
    constexpr int NPT = (DQK + kConvT - 1) / kConvT;  // n columns per thread
    float nacc[NPT];
#pragma unroll
    for (int u = 0; u < NPT; ++u) {
      const int c = ct + kConvT * u;
      nacc[u] = (n0 != nullptr && c < DQK) ? n0[(size_t)p * DQKt + cb + c] : 0.f;
    }
    auto store_n = [&](int b) {
      if (!do_n) return;
#pragma unroll
      for (int u = 0; u < NPT; ++u) {
        const int c = ct + kConvT * u;
        if (c < DQK) {
          if (nstates) nstates[((size_t)p * (NC + 1) + b) * DQKt + cb + c] = nacc[u];
        }
      }
    };
    int j = 0;
    bool ok = true;
    for (int i = 0; i < NC && ok; ++i) {
      const int kc = kc_of(i);
      store_n(reverse ? NC - i : i);
      const float al = final_only ? 1.f : alpha[(size_t)p * NC + kc];
#pragma unroll
      for (int u = 0; u < NPT; ++u) nacc[u] *= al;
      for (int r = 0; r < SUB; ++r, ++j) {
        const int s = j % ST;
        // every conversion thread passes each named barrier, so a wait that gives up in one of
        // them is shared through conv_fail before anyone acts on it
        const size_t tok0 = (size_t)p * S + (size_t)(kc * SUB + r) * kSub;
        // the slab's weights, staged once (both were read by the previous use of this stage
        // before the barriers of the slabs since)
        if (ct < kSub) sm.wx[s][ct] = wx[tok0 + ct];
        else if (do_n && ct < 2 * kSub) sm.wn[s][ct - kSub] = wn[tok0 + ct - kSub];
        if (!mbar_wait(&sm.full[s], (j / ST) & 1, err, 45, abort_ptr)) *(volatile int *)&sm.conv_fail = 1;
        named_barrier_sync(1, kConvT);
        if (*(volatile int *)&sm.conv_fail) {
          ok = false;
          break;
        }
        unsigned char *tile = sm.tile[s];
        if (do_n) {
          // n += sum_t omega'_t y_t, read from the bf16 slab before it is converted (eight
          // independent partial sums per column)
#pragma unroll
          for (int u = 0; u < NPT; ++u) {
            const int c = ct + kConvT * u;
            if (c < DQK) {
              const unsigned char *box = tile + (2 + c / 64) * 8192;
              const int ch = (c & 63) >> 3, el = c & 7;
              float acc[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
              for (int t0 = 0; t0 < kSub; t0 += 8)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const int t = t0 + e;  // t & 7 == e
                  const __nv_bfloat16 y =
                      *reinterpret_cast<const __nv_bfloat16 *>(box + t * 128 + ((ch ^ e) << 4) + 2 * el);
                  acc[e] = fmaf(sm.wn[s][t], __bfloat162float(y), acc[e]);
                }
              nacc[u] += ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
            }
          }
        }
        named_barrier_sync(1, kConvT);  // every read of the bf16 slab is done
        // X: 2 boxes x 64 rows x 8 pieces of 16 bytes; row = token, scaled by its weight
#pragma unroll
        for (int pc = ct; pc < 2 * 64 * 8; pc += kConvT) {
          const int t = (pc & 511) >> 3;
          uint4 *ptr = reinterpret_cast<uint4 *>(tile + pc * 16);
          const uint4 raw = *ptr;
          const float w = sm.wx[s][t];
          const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t out[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float lo = __uint_as_float(in[e] << 16) * w, hi = __uint_as_float(in[e] & 0xffff0000u) * w;
            const __half2 hv = __floats2half2_rn(lo, hi);
            out[e] = *reinterpret_cast<const uint32_t *>(&hv);
          }
          *ptr = make_uint4(out[0], out[1], out[2], out[3]);
        }
        // Y: NQ boxes, converted as they are
#pragma unroll
        for (int pc = ct; pc < NQ * 64 * 8; pc += kConvT) {
          uint4 *ptr = reinterpret_cast<uint4 *>(tile + 2 * 8192 + pc * 16);
          const uint4 raw = *ptr;
          const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t out[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __half2 hv = __floats2half2_rn(__uint_as_float(in[e] << 16), __uint_as_float(in[e] & 0xffff0000u));
            out[e] = *reinterpret_cast<const uint32_t *>(&hv);
          }
          *ptr = make_uint4(out[0], out[1], out[2], out[3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(&sm.conv[s]);
      }
    }
    if (ok && do_n) {
      store_n(reverse ? 0 : NC);
      if (n_fin) {
#pragma unroll
        for (int u = 0; u < NPT; ++u) {
          const int c = ct + kConvT * u;
          if (c < DQK) n_fin[(size_t)p * DQKt + cb + c] = nacc[u];
        }
      }
    }
    if (!ok) st_set_abort(abort_ptr);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tm, kCols);
  }
}

// Per-token weights and per-chunk factors of the state recurrences (one CTA per (chunk, head),
// one thread per token).  mode 2, the final forward state only: omega = omega' = the weight of
// token t in the final state, exp(i~_t + sum_{tau > t} log f_tau - m_S) / sqrt(d), and no
// per-chunk factors.  mode 0, the forward state C^(k): omega = omega' = w_t / sqrt(d) with
// the state-update weight w_t = exp(b_L + x_t - m^(k+1)); mode 1, the adjoint G^(k):
// omega = beta_t / D_t, omega' = beta_t c_t with beta_t = exp(m^(k) - max(m^(k), u_t)).  Both:
// alpha_k = exp(b_L + m^(k) - m^(k+1)); omega is stored divided by s_k, the power of two at or
// above the chunk's largest omega (1 when all are zero).
__global__ void state_weights_kernel(int mode, const float *__restrict__ gb, const float *__restrict__ gx,
                                     const float *__restrict__ gu, const float *__restrict__ cm,
                                     const float *__restrict__ invD, const float *__restrict__ cc, int S, int L,
                                     int DQK, float *__restrict__ wx, float *__restrict__ wn,
                                     float *__restrict__ alpha, float *__restrict__ sc) {
  __shared__ float smax[4];
  const int p = blockIdx.y, kc = blockIdx.x, t = threadIdx.x;
  const int NC = S / L;
  const size_t tb = (size_t)p * S + (size_t)kc * L;
  const float m_in = cm[(size_t)p * (NC + 1) + kc], m_out = cm[(size_t)p * (NC + 1) + kc + 1];
  const float bl = gb[tb + L - 1];
  float w, w2;
  if (mode == 2) {
    // the decay of every later chunk folded in: b from the end of this chunk to the end of the
    // sequence, against the final stabiliser (every weight <= 1, the largest exactly 1)
    __shared__ float s_after;
    if (t == 0) {
      float acc = 0.f;
      for (int j = kc + 1; j < NC; ++j) acc += gb[(size_t)p * S + (size_t)j * L + L - 1];
      s_after = acc;
    }
    __syncthreads();
    w = rsqrtf((float)DQK) * expf(bl + s_after + gx[tb + t] - cm[(size_t)p * (NC + 1) + NC]);
    wx[tb + t] = w;
    wn[tb + t] = w;
    return;
  }
  if (mode == 0) {
    w = rsqrtf((float)DQK) * expf(bl + gx[tb + t] - m_out);
    w2 = w;
  } else {
    const float beta = expf(m_in - fmaxf(m_in, gu[tb + t]));
    w = beta * invD[tb + t];
    w2 = beta * cc[tb + t];
  }
  float mx = fabsf(w);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((t & 31) == 0) smax[t >> 5] = mx;
  __syncthreads();
  mx = smax[0];
  for (int i = 1; i < L / 32; ++i) mx = fmaxf(mx, smax[i]);
  int e = 0;
  if (mx > 0.f) frexpf(mx, &e);  // mx = f 2^e with f in [0.5, 1): 2^e >= mx
  const float s = mx > 0.f ? ldexpf(1.f, e) : 1.f;
  wx[tb + t] = mx > 0.f ? ldexpf(w, -e) : 0.f;
  wn[tb + t] = w2;
  if (t == 0) {
    alpha[(size_t)p * NC + kc] = expf(bl + m_in - m_out);
    sc[(size_t)p * NC + kc] = s;
  }
}

template <int NQ>
cudaError_t states_tc_t(const CUtensorMap &mx, const CUtensorMap &my, const float *wx, const float *wn,
                        const float *alpha, const float *sc, int P, int S, int L, int DV, bool reverse,
                        const float *C0, const float *n0, float *states, float *nstates, float *C_fin, float *n_fin,
                        int *err, float *states_t, int DQKt, int CS, cudaStream_t stream) {
  auto kern = states_tc_kernel<NQ>;
  const size_t smem = sizeof(StatesSmem<NQ>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(DV / kTileM * CS, P), kThreadsT, smem, stream>>>(mx, my, wx, wn, alpha, sc, S, L, DV, reverse ? 1 : 0,
                                                               C0, n0, states, nstates, C_fin, n_fin, err, states_t,
                                                               DQKt, CS);
  return cudaGetLastError();
}

}  // namespace

bool states_tc_supported(int L, int DQK, int DV, bool bf16) {
  return bf16 && L % kSub == 0 && L <= 128 && (DQK == 64 || DQK == 128 || DQK == 256 || DQK == 512) &&
         DV % kTileM == 0;
}

cudaError_t launch_state_weights(int mode, const float *gb, const float *gx, const float *gu, const float *cm,
                                 const float *invD, const float *cc, int P, int S, int L, int DQK, float *wx,
                                 float *wn, float *alpha, float *sc, cudaStream_t stream) {
  if (P == 0 || S == 0) return cudaSuccess;
  state_weights_kernel<<<dim3(S / L, P), L, 0, stream>>>(mode, gb, gx, gu, cm, invD, cc, S, L, DQK, wx, wn, alpha,
                                                         sc);
  return cudaGetLastError();
}

cudaError_t launch_states_tc(const void *X, const void *Y, const float *wx, const float *wn, const float *alpha,
                             const float *sc, int P, int S, int L, int DQK, int DV, bool reverse, const float *C0,
                             const float *n0, float *states, float *nstates, float *C_fin, float *n_fin, int *err,
                             cudaStream_t stream, float *states_t) {
  if (P == 0 || S == 0) return cudaSuccess;  // no chunk: the caller's initial state is the only boundary
  CUtensorMap mx, my;
  const uint64_t rows = (uint64_t)P * S;
  if (!make_tmap_2d_b16(&mx, X, true, rows, DV, DV, 64, kSub)) return cudaErrorInvalidValue;
  if (!make_tmap_2d_b16(&my, Y, true, rows, DQK, DQK, 64, kSub)) return cudaErrorInvalidValue;
  // with every boundary stored, d_qk of 128 and more is split over two CTAs per 128 rows: twice
  // the SMs share the boundary states' stores, and each CTA holds two state buffers in tensor
  // memory (the final-state walk stores once and keeps its grid)
  const int CS = DQK >= 128 && alpha != nullptr ? 2 : 1;
  switch (DQK / CS) {
    case 64: return states_tc_t<1>(mx, my, wx, wn, alpha, sc, P, S, L, DV, reverse, C0, n0, states, nstates, C_fin, n_fin, err, states_t, DQK, CS, stream);
    case 128: return states_tc_t<2>(mx, my, wx, wn, alpha, sc, P, S, L, DV, reverse, C0, n0, states, nstates, C_fin, n_fin, err, states_t, DQK, CS, stream);
    case 256: return states_tc_t<4>(mx, my, wx, wn, alpha, sc, P, S, L, DV, reverse, C0, n0, states, nstates, C_fin, n_fin, err, states_t, DQK, CS, stream);
    case 512: return states_tc_t<8>(mx, my, wx, wn, alpha, sc, P, S, L, DV, reverse, C0, n0, states, nstates, C_fin, n_fin, err, states_t, DQK, CS, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace mlstm
