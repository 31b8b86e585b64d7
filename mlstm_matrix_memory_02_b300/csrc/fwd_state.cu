// fwd_state.cu -- the state walk of the three-kernel tensor-core forward: per (head, 128-row
// d_v tile, d_qk half) the matrix state stays in tensor memory for the whole sequence and each
// chunk costs three tensor-core products and one copy of the state.
//
// Page "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural Networks"
// (llms.blog): section 3 "The Parallel Dual Form" (H = ((Q K^T) o D) V inside a chunk, the state
// unrolled across chunks) and "Associative Matrix Cell State" (C_t = f_t C_{t-1} + i_t v_t k_t^T,
// h = C q / max(|n^T q|, .)).  With the chunk's operands prepared by the pre-pass (fwd_prep.cu:
// beta q and w k in fp16, P = (Q K^T / sqrt(d)) o D in fp16, 1/den per token), chunk k is
//   H^T = C16 (beta q)^T + V^T P^T           (X, then P V into the same accumulator)
//   T  += V^T (w k)                          (U: the state update, in the lazy frame C = e^sigma T)
//   h_r = H_r / den_r
// where C16 is the fp16 copy of the state entering the chunk.  The frame factors (e^sigma, the
// eager rescale) come from the pre-pass's per-chunk record, so nothing here depends on the gates.
//
// Work split as in the fused kernel: a cluster of two CTAs per 128-row d_v tile of a head, each
// holding half of d_qk (its half of T and of the C q sums); CTA rank rho finalises tokens
// [32 rho, 32 rho + 32) of each chunk, adding the partner's partial H^T columns received through
// distributed shared memory, and adds P V for those tokens only.
//
// Tensor memory: [0, DH) T (fp32), [DH, 3 DH / 2) C16 (fp16 pairs, the A operand of X),
// then two 64-column H^T buffers used by alternate chunks.
//
// Warp roles (512 threads; every hand-off an mbarrier, every wait bounded):
//   warp 0       TMA loads of the chunk's beta q and w k halves, v tile and own P rows (two stages)
//   warp 1       tensor-memory allocation; MMA issuer: U_k, X_k, P V_k, one commit
//   warps 4-7    the initial state; the copy T -> C16 before each chunk (lazy frame or eager
//                rescale); the final state
//   warps 8-11   epilogue: H^T from tensor memory, the partner's columns, 1/den, the h stores
//   warps 12-15  v of each stage: bf16 -> fp16 in place
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "f2math.cuh"
#include "kernels.cuh"
#include "sm100.cuh"
#include "tmap.cuh"

namespace mlstm {
namespace {

using namespace sm100;

constexpr int kLs = 64;       // chunk length
constexpr int kTileS = 128;   // d_v rows per CTA
constexpr int kStThreads = 512;
constexpr int kNR = 32;       // tokens finalised per CTA of the pair

struct StSmem {
  uint64_t full[2], empty[2], vready[2], done[2], hfree[2];
  uint64_t cready, hx_full, hx_free, fin, grp;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ bool st_aborted(const StSmem &sm) { return *(volatile const int *)&sm.abort_flag != 0; }
__device__ __forceinline__ void st_set_abort(StSmem &sm) { *(volatile int *)&sm.abort_flag = 1; }

template <int DH>
struct StLayout {
  static constexpr int QB = DH * 128;  // bytes of a [64 x DH] fp16 tile (DH / 64 swizzled blocks)
  static constexpr int OFF_K = QB, OFF_V = 2 * QB, OFF_P = 2 * QB + 16384;
  static constexpr int STAGE = 2 * QB + 16384 + kNR * 128;
  static constexpr int OFF_HX = 2 * STAGE;  // [128][32] fp32: the partner's H^T columns
  static constexpr size_t SMEM = (size_t)OFF_HX + 128 * 32 * 4 + 1024;
};

template <int DH, typename TO>
__global__ void __launch_bounds__(kStThreads, 1) fwd_state_kernel(
    const __grid_constant__ CUtensorMap mapQB, const __grid_constant__ CUtensorMap mapKW,
    const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapP,
    const __grid_constant__ CUtensorMap mapC, const float4 *__restrict__ cdat, const float *__restrict__ inv, int S,
    int DV, const float *__restrict__ C_init, TO *__restrict__ h, int *__restrict__ err) {
  using Lay = StLayout<DH>;
  constexpr int D = 2 * DH;
  constexpr uint32_t kColC16 = DH, kColH = DH + DH / 2;
  static_assert(DH == 256, "DH");
  static_assert(Lay::STAGE % 1024 == 0, "stage alignment");
  extern __shared__ uint8_t st_dyn[];
  __shared__ StSmem sm;
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(st_dyn) + 1023) & ~uintptr_t(1023));
  float *const HX = reinterpret_cast<float *>(base + Lay::OFF_HX);
#define SQ(s_) (base + (s_) * Lay::STAGE)
#define SK(s_) (base + (s_) * Lay::STAGE + Lay::OFF_K)
#define SV(s_) (base + (s_) * Lay::STAGE + Lay::OFF_V)
#define SP(s_) (base + (s_) * Lay::STAGE + Lay::OFF_P)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank(), prt = 1 - rank;
  const int a0 = (int)(blockIdx.x >> 1) * kTileS, c0 = rank * DH, p = blockIdx.y;
  const int NC = S / kLs, r_lo = kNR * rank;
  const int *abort_ptr = &sm.abort_flag;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
      mbar_init(&sm.vready[i], 128);
      mbar_init(&sm.done[i], 1);
      mbar_init(&sm.hfree[i], 128);
    }
    mbar_init(&sm.cready, 128);
    mbar_init(&sm.hx_full, 1);
    mbar_init(&sm.hx_free, 4);
    mbar_init(&sm.fin, 1);
    mbar_init(&sm.grp, 128);
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  pdl_wait();  // every operand comes from the previous kernels
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the partner's barriers are initialised before any remote access
  const uint32_t tm = sm.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA loads
    if (lane == 0) {
      prefetch_tensormap(&mapQB);
      prefetch_tensormap(&mapKW);
      prefetch_tensormap(&mapV);
      prefetch_tensormap(&mapP);
      int issued = 0;
      for (int k = 0; k < NC; ++k) {
        const int s = k & 1;
        // stage s is free once the products of chunk k-2 are done
        if (k >= 2 && !mbar_wait(&sm.empty[s], ((k >> 1) - 1) & 1, err, 111, abort_ptr)) {
          st_set_abort(sm);
          break;
        }
        if (st_aborted(sm)) break;
        const int row = p * S + k * kLs;
        mbar_arrive_expect_tx(&sm.full[s], (uint32_t)Lay::STAGE);
#pragma unroll 1
        for (int b = 0; b < DH / 64; ++b) {
          tma_load_2d(SQ(s) + b * 8192, &mapQB, c0 + b * 64, row, &sm.full[s]);
          tma_load_2d(SK(s) + b * 8192, &mapKW, c0 + b * 64, row, &sm.full[s]);
        }
        tma_load_2d(SV(s), &mapV, a0, row, &sm.full[s]);
        tma_load_2d(SV(s) + 8192, &mapV, a0 + 64, row, &sm.full[s]);
        tma_load_2d(SP(s), &mapP, 0, (p * NC + k) * kLs + r_lo, &sm.full[s]);
        issued = k + 1;
      }
      // nothing may leave while loads it issued are still landing
      for (int k = issued >= 2 ? issued - 2 : 0; k < issued; ++k) mbar_wait(&sm.full[k & 1], (k >> 1) & 1, err, 119);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_U = idesc_f16(kTileS, DH, 0, /*a MN-major*/ 1, /*b MN-major*/ 1);
      const uint32_t id_X = idesc_f16(kTileS, kLs, 0, 0, 0);
      const uint32_t id_P = idesc_f16(kTileS, kNR, 0, /*a MN-major*/ 1, 0);
      int k = 0;
      for (; k < NC; ++k) {
        const int s = k & 1;
        const uint32_t par = (k >> 1) & 1;
        const uint32_t colH = kColH + 64u * (uint32_t)(k & 1);
        if (!mbar_wait(&sm.full[s], par, err, 112, abort_ptr)) break;
        if (!mbar_wait(&sm.vready[s], par, err, 113, abort_ptr)) break;
        if (!mbar_wait(&sm.cready, k & 1, err, 114, abort_ptr)) break;  // C16 holds the state entering chunk k
        // the epilogue of chunk k-2 has read this H buffer
        if (k >= 2 && !mbar_wait(&sm.hfree[k & 1], ((k >> 1) - 1) & 1, err, 115, abort_ptr)) break;
        tc_fence_after();
        const uint64_t dv = smem_desc(smem_u32(SV(s)), 8192, 1024, kSwizzle128B);
        const uint64_t dkw = smem_desc(smem_u32(SK(s)), 8192, 1024, kSwizzle128B);
        const uint64_t dqb = smem_desc(smem_u32(SQ(s)), 16, 1024, kSwizzle128B);
        const uint64_t dp = smem_desc(smem_u32(SP(s)), 16, 1024, kSwizzle128B);
        // U: T += V^T (w k), one K = 16 step per block of 16 tokens (descriptors advance by adding
        // (byte offset >> 4) to the start-address field)
#pragma unroll
        for (int j = 0; j < kLs / 16; ++j)
          mma_f16_ss(tm, dv + (uint64_t)(j * 2048 >> 4), dkw + (uint64_t)(j * 2048 >> 4), id_U, 1);
        // X: H^T = C16 (beta q)^T over this CTA's d_qk half
#pragma unroll 4
        for (int kk = 0; kk < DH / 16; ++kk)
          mma_f16_ts(tm + colH, tm + kColC16 + kk * 8, dqb + (uint64_t)(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4),
                     id_X, kk > 0);
        // P V for the tokens finalised here, into the same accumulator after X
#pragma unroll
        for (int j = 0; j < kLs / 16; ++j)
          mma_f16_ss(tm + colH + r_lo, dv + (uint64_t)(j * 2048 >> 4), dp + (uint64_t)(j * 32 >> 4), id_P, 1);
        mma_commit(&sm.done[k & 1]);
        mma_commit(&sm.empty[s]);
      }
      if (k < NC) st_set_abort(sm);
      mma_commit(&sm.fin);  // completes once every MMA issued above has finished
      mbar_wait(&sm.fin, 0, err, 118);
    }
  } else if (warp < 4) {
    // warps 2 and 3 have no role
  } else if (warp < 8) {
    // ------------------------------------------------------------------ state copy, final state
    const int t = threadIdx.x - 128;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    uint32_t gph = 0;
    for (int c = 0; c < DH; c += 16) {
      uint32_t r[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        r[i] = __float_as_uint(C_init ? C_init[((size_t)p * DV + a0 + t) * D + c0 + c + i] : 0.f);
      tmem_st16(tm + lane_base + c, r);
    }
    tmem_wait_st();
    const float4 *cd = cdat + 2 * (size_t)p * NC;
    bool ok = true;
    for (int k = 0; k < NC; ++k) {
      // U_{k-1} has updated T and X_{k-1} has read C16
      if (k >= 1 && !mbar_wait(&sm.done[(k - 1) & 1], ((k - 1) >> 1) & 1, err, 120, abort_ptr)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float4 fr = cd[2 * k + 1];  // (exp(sigma), exp(sigma) alpha, lazy)
      const uint64_t frc2 = f2pack(fr.x, fr.x), frw2 = f2pack(fr.y, fr.y);
      if (fr.z != 0.f) {
        // C16 = fp16(exp(sigma) T): the next 32 columns load while the current ones convert
        uint32_t ua[32], ub[32];
        tmem_ld32(tm + lane_base, ua);
        tmem_wait_ld();
#pragma unroll 1
        for (int c = 0; c < DH; c += 64) {
          tmem_ld32(tm + lane_base + c + 32, ub);
          {
            uint32_t hv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              hv[i] = f2_to_h2(f2mul(f2pack(__uint_as_float(ua[2 * i]), __uint_as_float(ua[2 * i + 1])), frc2));
            tmem_st16(tm + lane_base + kColC16 + c / 2, hv);
          }
          tmem_wait_ld();
          if (c + 64 < DH) tmem_ld32(tm + lane_base + c + 64, ua);
          {
            uint32_t hv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              hv[i] = f2_to_h2(f2mul(f2pack(__uint_as_float(ub[2 * i]), __uint_as_float(ub[2 * i + 1])), frc2));
            tmem_st16(tm + lane_base + kColC16 + c / 2 + 16, hv);
          }
          if (c + 64 < DH) tmem_wait_ld();
        }
      } else {
        // eager: also write the decayed state back to frame 0
#pragma unroll 1
        for (int c = 0; c < DH; c += 32) {
          uint32_t u[32];
          tmem_ld32(tm + lane_base + c, u);
          tmem_wait_ld();
          uint32_t hv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint64_t x = f2pack(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1]));
            hv[i] = f2_to_h2(f2mul(x, frc2));
            float lo, hi;
            f2unpack(f2mul(x, frw2), lo, hi);
            u[2 * i] = __float_as_uint(lo);
            u[2 * i + 1] = __float_as_uint(hi);
          }
          tmem_st16(tm + lane_base + kColC16 + c / 2, hv);
          tmem_st16(tm + lane_base + c, *reinterpret_cast<const uint32_t(*)[16]>(&u[0]));
          tmem_st16(tm + lane_base + c + 16, *reinterpret_cast<const uint32_t(*)[16]>(&u[16]));
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&sm.cready);
    }
    // final state C_last = exp(frame) T once the last update is done; every stage is free by then
    if (ok && NC > 0 && !mbar_wait(&sm.done[(NC - 1) & 1], ((NC - 1) >> 1) & 1, err, 125, abort_ptr)) ok = false;
    if (ok) {
      tc_fence_after();
      const float frl = NC > 0 ? __expf(cd[2 * (NC - 1)].w) : 1.f;
      // 32 columns at a time through two swizzled staging tiles [128 rows x 128 bytes]; a bounded
      // barrier over the warpgroup orders the tile writes, the store and the tile's reuse
      auto group_sync = [&](int code) -> bool {
        mbar_arrive(&sm.grp);
        const bool r = mbar_wait(&sm.grp, gph & 1, err, code, abort_ptr);
        ++gph;
        return r;
      };
#pragma unroll 1
      for (int c = 0, slab = 0; c < DH; c += 32, ++slab) {
        uint8_t *tile = base + (slab & 1) * 16384;
        if (slab >= 2) {
          if (t == 0) bulk_wait_read<1>();  // the store that used this tile has read it
          if (!group_sync(126)) { ok = false; break; }
        }
        uint32_t u[32];
        tmem_ld32(tm + lane_base + c, u);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<float4 *>(tile + t * 128 + ((i ^ (t & 7)) << 4)) =
              make_float4(__uint_as_float(u[4 * i]) * frl, __uint_as_float(u[4 * i + 1]) * frl,
                          __uint_as_float(u[4 * i + 2]) * frl, __uint_as_float(u[4 * i + 3]) * frl);
        fence_proxy_async_smem();
        if (!group_sync(127)) { ok = false; break; }
        if (t == 0) {
          tma_store_2d(&mapC, c0 + c, p * DV + a0, tile);
          bulk_commit();
        }
      }
      if (t == 0) bulk_wait_all();
    }
    if (!ok) st_set_abort(sm);
  } else if (warp < 12) {
    // ------------------------------------------------------------------ epilogue
    const int t = threadIdx.x - 256;  // tensor-memory lane = d_v row within the tile
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    bool ok = true;
    for (int k = 0; k < NC; ++k) {
      const uint32_t colH = kColH + 64u * (uint32_t)(k & 1);
      if (!mbar_wait(&sm.done[k & 1], (k >> 1) & 1, err, 121, abort_ptr)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t u[2][32];
      tmem_ld32(tm + lane_base + colH + 32 * rank, u[0]);  // tokens finalised here
      tmem_ld32(tm + lane_base + colH + 32 * prt, u[1]);   // the partner's
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&sm.hfree[k & 1]);
      // the partner's partial sums for the tokens finalised here, and ours for its tokens
      if (k >= 1 && !mbar_wait_cluster(&sm.hx_free, (k - 1) & 1, err, 122, abort_ptr)) {
        ok = false;
        break;
      }
      const uint32_t rbar = mapa_shared(smem_u32(&sm.hx_full), prt);
      const uint32_t dst = mapa_shared(smem_u32(HX + t * 32), prt);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        st_async_v4(dst + ((i ^ (t & 7)) << 4), __uint_as_float(u[1][4 * i]), __uint_as_float(u[1][4 * i + 1]),
                    __uint_as_float(u[1][4 * i + 2]), __uint_as_float(u[1][4 * i + 3]), rbar);
      if (t == 0) mbar_arrive_expect_tx(&sm.hx_full, 128 * 32 * 4);
      if (!mbar_wait_cluster(&sm.hx_full, k & 1, err, 123, abort_ptr)) {
        ok = false;
        break;
      }
      const float *src = HX + t * 32;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 v4 = *reinterpret_cast<const float4 *>(src + 4 * (i ^ (t & 7)));
        u[0][4 * i] = __float_as_uint(__uint_as_float(u[0][4 * i]) + v4.x);
        u[0][4 * i + 1] = __float_as_uint(__uint_as_float(u[0][4 * i + 1]) + v4.y);
        u[0][4 * i + 2] = __float_as_uint(__uint_as_float(u[0][4 * i + 2]) + v4.z);
        u[0][4 * i + 3] = __float_as_uint(__uint_as_float(u[0][4 * i + 3]) + v4.w);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&sm.hx_free), prt));
      const size_t tok = (size_t)p * S + (size_t)k * kLs + r_lo;
      const float *iv = inv + tok;
      TO *hp = h + tok * DV + a0 + t;
#pragma unroll
      for (int i = 0; i < kNR; i += 4) {
        const float4 i4 = *reinterpret_cast<const float4 *>(iv + i);
        hp[(size_t)i * DV] = from_f32<TO>(__uint_as_float(u[0][i]) * i4.x);
        hp[(size_t)(i + 1) * DV] = from_f32<TO>(__uint_as_float(u[0][i + 1]) * i4.y);
        hp[(size_t)(i + 2) * DV] = from_f32<TO>(__uint_as_float(u[0][i + 2]) * i4.z);
        hp[(size_t)(i + 3) * DV] = from_f32<TO>(__uint_as_float(u[0][i + 3]) * i4.w);
      }
    }
    if (!ok) st_set_abort(sm);
  } else {
    // ------------------------------------------------------------------ v: bf16 -> fp16 in place
    const int t = threadIdx.x - 384;
    for (int k = 0; k < NC; ++k) {
      const int s = k & 1;
      if (!mbar_wait(&sm.full[s], (k >> 1) & 1, err, 124, abort_ptr)) {
        st_set_abort(sm);
        break;
      }
      uint4 *vp = reinterpret_cast<uint4 *>(SV(s));
      uint4 raw[8];
#pragma unroll
      for (int b = 0; b < 8; ++b) raw[b] = vp[t + 128 * b];
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        uint4 o4;
        o4.x = bf2_to_h2(raw[b].x);
        o4.y = bf2_to_h2(raw[b].y);
        o4.z = bf2_to_h2(raw[b].z);
        o4.w = bf2_to_h2(raw[b].w);
        vp[t + 128 * b] = o4;
      }
      fence_proxy_async_smem();
      mbar_arrive(&sm.vready[s]);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its partner may still access its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tm, 512);
  }
#undef SQ
#undef SK
#undef SV
#undef SP
}

template <int DH, typename TO>
cudaError_t launch_state_one(const PrepBuffers &b, const void *v, int P, int S, int DV, const float *C_init, void *h,
                             float *C_last, int *err, cudaStream_t stream) {
  constexpr int D = 2 * DH;
  CUtensorMap mq, mk, mv, mp, mc;
  if (!make_tmap_2d_b16(&mq, b.qb, false, (uint64_t)P * S, D, D, 64, kLs)) return cudaErrorInvalidValue;
  if (!make_tmap_2d_b16(&mk, b.kw, false, (uint64_t)P * S, D, D, 64, kLs)) return cudaErrorInvalidValue;
  if (!make_tmap_2d_b16(&mv, v, true, (uint64_t)P * S, DV, DV, 64, kLs)) return cudaErrorInvalidValue;
  if (!make_tmap_2d_b16(&mp, b.pm, false, (uint64_t)P * S, kLs, kLs, kLs, kNR)) return cudaErrorInvalidValue;
  if (!make_tmap_2d_f32(&mc, C_last, (uint64_t)P * DV, D, kTileS)) return cudaErrorInvalidValue;
  auto kern = fwd_state_kernel<DH, TO>;
  const size_t smem = StLayout<DH>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((DV / kTileS) * 2, P, 1);
  cfg.blockDim = dim3(kStThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may start while the previous kernel finishes (pdl_wait above orders the reads)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mp, mc, static_cast<const float4 *>(b.cdat),
                            static_cast<const float *>(b.inv), S, DV, C_init, static_cast<TO *>(h), err);
}

}  // namespace

cudaError_t launch_fwd_state(const PrepBuffers &b, const void *v, bool out_bf16, int P, int S, int D, int DV,
                             const float *C_init, void *h, float *C_last, int *err, cudaStream_t stream) {
  if (P == 0 || S == 0) return cudaSuccess;
  if (DV % kTileS != 0 || S % kLs != 0) return cudaErrorInvalidValue;
  if (D != 512) return cudaErrorInvalidValue;  // the sizes the pre-pass takes
  return out_bf16 ? launch_state_one<256, __nv_bfloat16>(b, v, P, S, DV, C_init, h, C_last, err, stream)
                  : launch_state_one<256, float>(b, v, P, S, DV, C_init, h, C_last, err, stream);
}

}  // namespace mlstm
