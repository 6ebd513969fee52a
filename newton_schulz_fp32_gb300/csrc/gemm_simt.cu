// CUDA-core matrix products of the Newton-Schulz iteration.
//
// This is the FP32-operand mode: FP32 inputs, FP32 fused multiply-adds,
// FP32 outputs, so the iteration keeps single-precision accuracy (plain TF32
// tensor-core products would not).  The same kernel also runs with BF16
// operands (FP32 accumulation, BF16 output rounded to nearest even) as an
// independent cross-check of the tensor-core path.
//
//   D = alpha * A op(B) + beta * E + gamma * I        (fp32 epilogue, in
//   that order: alpha*acc, + beta*E, + gamma on the diagonal)
//
// A 128 x 128 output tile per 256-thread block, 8 x 8 outputs per thread,
// K staged through shared memory 16 at a time.  Grouped: the block reads its
// (problem, tile) pair from a precomputed list covering every matrix of the
// phase.
#include <cuda_bf16.h>

#include "muon_internal.h"

namespace muon {
namespace {

constexpr int BM = kSimtTile, BN = kSimtTile, BK = 16, TM = 8, TN = 8;
constexpr int NT = (BM / TM) * (BN / TN);   // 256

template <int ES>
__device__ __forceinline__ float ld_el(const void* p, int64_t i) {
  if constexpr (ES == 2) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  else return reinterpret_cast<const float*>(p)[i];
}

__device__ __forceinline__ float ld_rt(const void* p, int es, int64_t i) {
  if (es == 2) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  return reinterpret_cast<const float*>(p)[i];
}

__device__ __forceinline__ void st_rt(void* p, int es, int64_t i, float v) {
  if (es == 2) reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  else reinterpret_cast<float*>(p)[i] = v;
}

template <int ES>
__global__ void __launch_bounds__(NT)
k_gemm_simt(const GemmProblem* __restrict__ probs, const GemmTile* __restrict__ tiles,
            const StepState* state) {
  if (state != nullptr && state->overflow) return;
  __shared__ __align__(16) float As[BK][BM + 4];
  __shared__ __align__(16) float Bs[BK][BN + 4];
  const GemmTile t = tiles[blockIdx.x];
  const GemmProblem p = probs[t.problem];
  const int m0 = t.tm * BM, n0 = t.tn * BN;
  const int tx = threadIdx.x % (BN / TN), ty = threadIdx.x / (BN / TN);
  float acc[TM][TN];
  #pragma unroll
  for (int i = 0; i < TM; ++i)
    #pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < p.K; k0 += BK) {
    for (int i = threadIdx.x; i < BM * BK; i += NT) {
      const int r = i / BK, kk = i % BK;
      const int gm = m0 + r, gk = k0 + kk;
      As[kk][r] = (gm < p.M && gk < p.K) ? ld_el<ES>(p.A, int64_t(gm) * p.lda + gk) : 0.f;
    }
    if (p.b_kmajor) {
      for (int i = threadIdx.x; i < BN * BK; i += NT) {
        const int c = i / BK, kk = i % BK;
        const int gn = n0 + c, gk = k0 + kk;
        Bs[kk][c] = (gn < p.N && gk < p.K) ? ld_el<ES>(p.B, int64_t(gn) * p.ldb + gk) : 0.f;
      }
    } else {
      for (int i = threadIdx.x; i < BN * BK; i += NT) {
        const int kk = i / BN, c = i % BN;
        const int gn = n0 + c, gk = k0 + kk;
        Bs[kk][c] = (gn < p.N && gk < p.K) ? ld_el<ES>(p.B, int64_t(gk) * p.ldb + gn) : 0.f;
      }
    }
    __syncthreads();
    #pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[TM], b[TN];
      #pragma unroll
      for (int i = 0; i < TM; i += 4) {
        const float4 v = *reinterpret_cast<const float4*>(&As[kk][ty * TM + i]);
        a[i] = v.x; a[i + 1] = v.y; a[i + 2] = v.z; a[i + 3] = v.w;
      }
      #pragma unroll
      for (int j = 0; j < TN; j += 4) {
        const float4 v = *reinterpret_cast<const float4*>(&Bs[kk][tx * TN + j]);
        b[j] = v.x; b[j + 1] = v.y; b[j + 2] = v.z; b[j + 3] = v.w;
      }
      #pragma unroll
      for (int i = 0; i < TM; ++i)
        #pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = __fmaf_rn(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }

  #pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int gm = m0 + ty * TM + i;
    if (gm >= p.M) continue;
    #pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int gn = n0 + tx * TN + j;
      if (gn >= p.N) continue;
      if (p.symmetric && gn < gm) continue;
      float v = __fmul_rn(p.alpha, acc[i][j]);
      if (p.E != nullptr) v = __fadd_rn(v, __fmul_rn(p.beta, ld_rt(p.E, p.e_es, int64_t(gm) * p.lde + gn)));
      if (p.gamma != 0.f && gm == gn) v = __fadd_rn(v, p.gamma);
      st_rt(p.D, p.d_es, int64_t(gm) * p.ldd + gn, v);
      if (p.symmetric && gn > gm) st_rt(p.D, p.d_es, int64_t(gn) * p.ldd + gm, v);
    }
  }
}

}  // namespace

void launch_gemm_simt(const GemmProblem* probs, const GemmTile* tiles, int ntiles, int ab_es,
                      const StepState* state, cudaStream_t s) {
  if (ntiles <= 0) return;
  if (ab_es == 2) k_gemm_simt<2><<<ntiles, NT, 0, s>>>(probs, tiles, state);
  else k_gemm_simt<4><<<ntiles, NT, 0, s>>>(probs, tiles, state);
}

namespace {
__global__ void k_convert_bf16(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst,
                               int64_t n, const StepState* state) {
  if (state != nullptr && state->overflow) return;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x)
    dst[i] = __float2bfloat16_rn(src[i]);
}
}  // namespace

void launch_convert_bf16(const float* src, void* dst, int64_t n, const StepState* state,
                         cudaStream_t s) {
  if (n <= 0) return;
  const int64_t blocks = (n + 255) / 256;
  k_convert_bf16<<<static_cast<int>(blocks < 4096 ? blocks : 4096), 256, 0, s>>>(
      src, static_cast<__nv_bfloat16*>(dst), n, state);
}

}  // namespace muon
