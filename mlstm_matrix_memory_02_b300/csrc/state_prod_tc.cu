// state_prod_tc.cu -- products of every chunk's tokens with a chunk-boundary state, on tensor
// cores (tf32).
//
// Page "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural Networks"
// (llms.blog), section 3 "Associative Matrix Cell State" (the retrieval C_t q_t) and "The Parallel
// Dual Form" (chunked: a chunk's tokens meet the state entering it through one product).  The
// backward needs four such products per chunk k of each head (C^(k) the boundary state entering
// chunk k, G^(k+1) the adjoint state entering it from the right):
//   C^(k) q_t,   C^(k)^T dh_t,   G^(k+1)^T v_t,   G^(k+1) k_t     (t in chunk k)
// each Out[t][r] = scale_t sum_c A[r][c] Y[t][c] with A a state in [rows][cols] layout (the state
// itself, or its transpose), Y the token rows (fp32 copies of the bf16 inputs) and scale_t an
// optional per-token factor.  fp32 operands enter the MMA as tf32: the states keep fp32's range
// (the adjoint state grows like dh / D) with 2^-11 relative rounding.
//
// CTA = (128 rows of A, 64-token slab, head): warp 0 loads 32-column slabs of the A tile [128 x 32] and of
// the token tile [64 x 32] by TMA (four slabs in flight), warp 1 allocates 64 tensor-memory
// columns and issues four K = 8 MMAs per slab (M = 128, N = 64, both operands K-major), warps 2-5
// read the 128 x 64 result and store Out[t][r]: for each token the 32 lanes of a warp write 32
// consecutive r (128-byte stores).
#include "common.cuh"
#include "kernels.cuh"
#include "sm100.cuh"
#include "tmap.cuh"

namespace mlstm {

namespace {
using namespace sm100;

constexpr int kRowsA = 128;  // rows of A per CTA (tensor-memory lanes)
constexpr int kTok = 64;     // tokens per chunk (N of the MMA)
constexpr int kSlabK = 32;   // fp32 columns per 128-byte swizzle atom
constexpr int kStagesP = 4;
constexpr int kThreadsP = 192;

struct alignas(1024) ProdSmem {
  unsigned char a[kStagesP][kRowsA * 128];  // 16 KB per slab
  unsigned char y[kStagesP][kTok * 128];    // 8 KB per slab
  uint64_t full[kStagesP], empty[kStagesP];
  uint64_t done, fin;
  uint32_t tmem_base;
  int abort_flag;
};

// Instruction descriptor of kind::tf32 with fp32 accumulation (the operand format field holds
// 2 for tf32; both operands K-major).
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// A: the states of all heads at the boundaries of chunks of L tokens, [P * (S / L + 1) * MA
// rows][K] (row i = row i % MA of boundary i / MA); the 64 tokens of slab j of a head use the
// state at boundary j / (L / 64) + bshift.  Y: tokens [P * S][K].  Out: [P * S][MA].
__global__ void __launch_bounds__(kThreadsP, 1) state_prod_kernel(
    const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapY, int S, int L, int MA, int K,
    int bshift, const float *__restrict__ tok_scale, float scale, float *__restrict__ out, int *__restrict__ err) {
  extern __shared__ unsigned char sp_raw[];
  ProdSmem &sm = *reinterpret_cast<ProdSmem *>((reinterpret_cast<uintptr_t>(sp_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * kRowsA, kc = blockIdx.y, p = blockIdx.z;  // kc: the 64-token slab
  const int NC = S / L, NK = K / kSlabK;
  int *abort_ptr = &sm.abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesP; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.done, 1);
    mbar_init(&sm.fin, 1);
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, kTok);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = sm.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tensormap(&mapA);
      prefetch_tensormap(&mapY);
      const int arow = ((p * (NC + 1) + kc / (L / kTok) + bshift) * MA) + r0;
      const int yrow = p * S + kc * kTok;
      int issued = 0;
      for (int j = 0; j < NK; ++j) {
        const int s = j % kStagesP;
        if (j >= kStagesP && !mbar_wait(&sm.empty[s], ((j / kStagesP) - 1) & 1, err, 51, abort_ptr)) break;
        mbar_arrive_expect_tx(&sm.full[s], (uint32_t)(kRowsA + kTok) * 128u);
        tma_load_2d(sm.a[s], &mapA, j * kSlabK, arow, &sm.full[s]);
        tma_load_2d(sm.y[s], &mapY, j * kSlabK, yrow, &sm.full[s]);
        issued = j + 1;
      }
      for (int j = issued > kStagesP ? issued - kStagesP : 0; j < issued; ++j)
        mbar_wait(&sm.full[j % kStagesP], (j / kStagesP) & 1, err, 59);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id = idesc_tf32(kRowsA, kTok);
      bool ok = true;
      for (int j = 0; j < NK; ++j) {
        const int s = j % kStagesP;
        if (!mbar_wait(&sm.full[s], (j / kStagesP) & 1, err, 52, abort_ptr)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t da = smem_desc(smem_u32(sm.a[s]), 16, 1024, kSwizzle128B);
        const uint64_t dy = smem_desc(smem_u32(sm.y[s]), 16, 1024, kSwizzle128B);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)  // K = 8 tf32 = 32 bytes per step
          mma_tf32_ss(tm, da + (uint64_t)(ks * 32 >> 4), dy + (uint64_t)(ks * 32 >> 4), id, (j | ks) != 0);
        mma_commit(&sm.empty[s]);
      }
      if (ok) mma_commit(&sm.done);
      else *(volatile int *)abort_ptr = 1;
      mma_commit(&sm.fin);  // completes once every MMA issued above has finished
      mbar_wait(&sm.fin, 0, err, 58);
    }
  } else {
    const int q = warp & 3;  // tensor-memory lanes 32 q .. 32 q + 31
    const int row = 32 * q + lane;
    const bool got = __all_sync(0xffffffffu, mbar_wait(&sm.done, 0, err, 53, abort_ptr));
    if (got) {
      tc_fence_after();
      const uint32_t trow = tm + ((uint32_t)(32 * q) << 16);
      float *o = out + ((size_t)p * S + (size_t)kc * kTok) * MA + r0 + row;
      for (int c0 = 0; c0 < kTok; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(trow + c0, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int t = c0 + e;
          const float f = tok_scale ? tok_scale[(size_t)p * S + (size_t)kc * kTok + t] * scale : scale;
          o[(size_t)t * MA] = __uint_as_float(r[e]) * f;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tm, kTok);
  }
}

}  // namespace

bool state_prod_supported(int L, int DQK, int DV) {
  return L % kTok == 0 && DQK % kRowsA == 0 && DV % kRowsA == 0;
}

cudaError_t launch_state_prod(const float *A, int MA, int K, int bshift, const float *Y, const float *tok_scale,
                              float scale, int P, int S, int L, float *out, int *err, cudaStream_t stream) {
  if (P == 0 || S == 0) return cudaSuccess;
  const int NC = S / L;
  CUtensorMap ma, my;
  if (!make_tmap_2d_f32(&ma, A, (uint64_t)P * (NC + 1) * MA, (uint64_t)K, kRowsA)) return cudaErrorInvalidValue;
  if (!make_tmap_2d_f32(&my, Y, (uint64_t)P * S, (uint64_t)K, kTok)) return cudaErrorInvalidValue;
  const size_t smem = sizeof(ProdSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(state_prod_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  state_prod_kernel<<<dim3(MA / kRowsA, S / kTok, P), kThreadsP, smem, stream>>>(ma, my, S, L, MA, K, bshift,
                                                                                   tok_scale, scale, out, err);
  return cudaGetLastError();
}

}  // namespace mlstm
