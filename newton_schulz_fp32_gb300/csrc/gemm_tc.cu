// Tensor-core matrix products of the Newton-Schulz iteration (BF16 operands,
// FP32 accumulation in tensor memory), written for sm_103a with tcgen05,
// TMA and mbarriers in inline PTX.
//
//   D = alpha * A op(B) + beta * E + gamma * I     (D, E bf16; epilogue fp32)
//
// One persistent CTA per SM walks a static list of (problem, 128 x 256 tile)
// pairs covering every matrix of one phase of the iteration (grouped GEMM).
// Warp roles:
//   warp 0      TMA producer: A tile 128 x 64 and B tile 256 x 64 per stage,
//               128-byte swizzle, 4-stage ring guarded by full/empty mbarriers
//   warp 1      allocates 512 TMEM columns (two 128 x 256 FP32 accumulators)
//               and issues tcgen05.mma (M=128, N=256, K=16) from one thread
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, alpha/beta/gamma in
//               FP32, round to BF16, store (and mirror for symmetric outputs)
// Double-buffered accumulators let the epilogue of tile i overlap the main
// loop of tile i+1.
//
// B comes either K-major (stored N x K: the Gram products X X^T, A A, R R,
// P R, T P) or MN-major (stored K x N: B X, P Q, Q X0), selected by the
// instruction descriptor's B-major bit and the matching shared-memory
// descriptor.
//
// Every wait is bounded: after ~2 s without progress the CTA records an
// error code, stops issuing work, frees its tensor memory and exits.
#include <cuda_bf16.h>

#include <cstring>

#include "tc_common.cuh"

namespace muon {
namespace {

using namespace tc;

constexpr int BM = kTcBM, BN = kTcBN, BK = kTcBK;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;          // 16 KB
constexpr int B_BYTES = BN * BK * 2;          // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 512;                // 2 accumulators x 256 fp32 columns
constexpr int EPI_WARPS = 8;                  // two per TMEM lane quarter, 4 chunks each
constexpr int NTHREADS = 64 + 32 * EPI_WARPS;
// Epilogue staging per epilogue warp: one 32 x 32 bf16 addend chunk (TMA
// load, 64-byte swizzle) and one output box of 64-byte rows (TMA store,
// 64-byte swizzle: 32 bf16 or 16 fp32 columns).  Buffers are 1 KB aligned.
constexpr int EPI_E_BYTES = 32 * 32 * 2;                                 // 2 KB
constexpr int EPI_D_BYTES = 32 * 64;                                     // 2 KB
constexpr int EPI_WARP_BYTES = EPI_E_BYTES + EPI_D_BYTES;                // 4 KB
constexpr int EPI_BYTES = EPI_WARPS * EPI_WARP_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 4 + EPI_WARPS;   // full, empty, tfull x2, tempty x2, E per epilogue warp
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + 1024 /*align*/ + 256 /*barriers*/;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
__global__ void __launch_bounds__(NTHREADS, 1)
k_gemm_tc(const GemmProblem* __restrict__ probs, const TcMaps* __restrict__ maps,
          const GemmTile* __restrict__ tiles, int ntiles, const StepState* state,
          int* err_flag) {
  if (state != nullptr && state->overflow) return;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;          // 1024-aligned stage ring
  uint8_t* base_ptr = smem_raw + (base - raw);
  uint8_t* epi_base = base_ptr + STAGES * STAGE_BYTES;    // per-warp epilogue staging
  const uint32_t bar_base = base + STAGES * STAGE_BYTES + EPI_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + STAGES * STAGE_BYTES + EPI_BYTES);
  // barrier layout: full[STAGES], empty[STAGES], tfull[2], tempty[2]
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto tfull_bar = [&](int i) { return bar_base + 8u * (2 * STAGES + i); };
  auto tempty_bar = [&](int i) { return bar_base + 8u * (2 * STAGES + 2 + i); };
  auto e_bar = [&](int w) { return bar_base + 8u * (2 * STAGES + 4 + w); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + NUM_BARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull_bar(i), 1);
      mbar_init(tempty_bar(i), EPI_WARPS);   // one arrival per epilogue warp
    }
    for (int w = 0; w < EPI_WARPS; ++w) mbar_init(e_bar(w), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int last_problem = -1;
      for (int ti = blockIdx.x; ti < ntiles && !*abort_flag; ti += gridDim.x) {
        const GemmTile t = tiles[ti];
        const GemmProblem& p = probs[t.problem];
        const TcMaps* mp = maps + t.problem;
        if (t.problem != last_problem) {
          asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mp->a)));
          asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mp->b)));
          last_problem = t.problem;
        }
        const int nk = (p.K + BK - 1) / BK;
        const bool b_k = p.b_kmajor != 0;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, err_flag, ERR_TIMEOUT_PRODUCER)) break;
          const uint32_t sa = base + s * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          mbar_expect_tx(full_bar(s), STAGE_BYTES);
          tma_load_2d(sa, &mp->a, kb * BK, t.tm * BM, full_bar(s));
          if (b_k) {
            tma_load_2d(sb, &mp->b, kb * BK, t.tn * BN, full_bar(s));
          } else {
            #pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_2d(sb + j * (64 * BK * 2), &mp->b, t.tn * BN + j * 64, kb * BK, full_bar(s));
          }
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t acc_ph = 0;
      for (int ti = blockIdx.x; ti < ntiles && !*abort_flag; ti += gridDim.x) {
        const GemmTile t = tiles[ti];
        const GemmProblem& p = probs[t.problem];
        const int nk = (p.K + BK - 1) / BK;
        const bool b_k = p.b_kmajor != 0;
        // MMA width: the tile's columns inside the matrix, rounded up to the
        // B operand's swizzle atom (32 rows K-major, 64 elements MN-major);
        // the epilogue reads no column beyond it
        const int n_rem = p.N - t.tn * BN;
        const int n_eff = min(BN, b_k ? (n_rem + 31) & ~31 : (n_rem + 63) & ~63);
        const uint32_t idesc = make_idesc(!b_k, BM, n_eff);
        if (!mbar_wait(tempty_bar(acc), acc_ph ^ 1u, abort_flag, err_flag, ERR_TIMEOUT_MMA)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(full_bar(s), ph, abort_flag, err_flag, ERR_TIMEOUT_MMA)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = base + s * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          #pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            // K-major, 128B swizzle: the 16-element K slice starts 32 bytes in
            const uint64_t ad = make_desc(sa + k * 32, 16, 1024, kSwizzle128);
            // K-major B: same; MN-major B: 16 K-rows of 128 bytes further,
            // 64-element MN chunks 8 KB apart (LBO), 8-row K groups 1 KB (SBO)
            const uint64_t bd = b_k ? make_desc(sb + k * 32, 16, 1024, kSwizzle128)
                                    : make_desc(sb + k * 16 * 128, 64 * BK * 2, 1024, kSwizzle128);
            umma_bf16(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(empty_bar(s));      // frees this stage when the MMAs finish
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));      // accumulator ready for the epilogue
        acc ^= 1;
        if (acc == 0) acc_ph ^= 1u;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                       // TMEM lane quarter this warp may read
    const int ew = warp - 2;                      // epilogue warp 0..7
    // the two warps of a lane quarter take alternate 32-column chunks, so the
    // upper-triangle chunks of a diagonal tile are shared evenly
    const int c_par = ew >> 2;
    uint8_t* ebuf = epi_base + ew * EPI_WARP_BYTES;
    uint8_t* dbuf = ebuf + EPI_E_BYTES;
    const uint32_t ebuf_s = smem_u32(ebuf);
    const uint32_t dbuf_s = smem_u32(dbuf);
    uint32_t eph = 0u;
    bool ebuf_mirrored = false;   // the last tile staged mirror chunks in ebuf
    int acc = 0;
    uint32_t acc_ph = 0;
    bool ok = true;
    for (int ti = blockIdx.x; ti < ntiles && ok && !*abort_flag; ti += gridDim.x) {
      const GemmTile t = tiles[ti];
      const GemmProblem& p = probs[t.problem];     // read through L1, not held in registers
      const TcMaps* mp = maps + t.problem;
      const int gm0 = t.tm * BM + q * 32;          // first row of this warp's 32-row slab
      // chunks this warp writes: inside the matrix, and for symmetric
      // products not strictly below the diagonal (32-aligned both ways)
      uint32_t todo = 0;
      if (gm0 < p.M)
        for (int c = c_par; c < BN / 32; c += 2) {
          const int gn0 = t.tn * BN + c * 32;
          if (gn0 < p.N && !(p.symmetric && gn0 < gm0)) todo |= 1u << c;
        }
      const bool has_e = p.E != nullptr;
      if (has_e && todo && lane == 0) {   // prefetch the first addend chunk
        if (ebuf_mirrored) tma_store_wait_read();   // a mirror store may still read ebuf
        mbar_expect_tx(e_bar(ew), EPI_E_BYTES);
        tma_load_2d(ebuf_s, &mp->e, t.tn * BN + (__ffs(todo) - 1) * 32, gm0, e_bar(ew));
      }
      if (!mbar_wait(tfull_bar(acc), acc_ph, abort_flag, err_flag, ERR_TIMEOUT_EPILOGUE)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float ssq = 0.f;   // this warp's sum of squares of the tile (last product only)
      uint32_t rest = todo;
      while (rest) {
        const int c = __ffs(rest) - 1;
        rest &= rest - 1;
        const int gn0 = t.tn * BN + c * 32;
        float x[32];
        tmem_ld32(tmem_base + static_cast<uint32_t>(acc * BN + c * 32) +
                      (static_cast<uint32_t>(q * 32) << 16),
                  x);
        #pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = __fmul_rn(p.alpha, x[j]);
        if (p.blk != 0 && gm0 / p.blk != gn0 / p.blk) {   // across stacked blocks
          #pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = 0.f;
        }
        if (has_e) {
          if (!mbar_wait(e_bar(ew), eph, abort_flag, err_flag, ERR_TIMEOUT_EPILOGUE)) {
            ok = false;
            break;
          }
          eph ^= 1u;
          #pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint4 w = *reinterpret_cast<const uint4*>(ebuf + sw64(lane, g));
            const __nv_bfloat162* hh = reinterpret_cast<const __nv_bfloat162*>(&w);
            #pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float2 f = __bfloat1622float2(hh[u]);
              x[g * 8 + 2 * u] = __fadd_rn(x[g * 8 + 2 * u], __fmul_rn(p.beta, f.x));
              x[g * 8 + 2 * u + 1] = __fadd_rn(x[g * 8 + 2 * u + 1], __fmul_rn(p.beta, f.y));
            }
          }
          __syncwarp();   // every lane has read the addend: the buffer may be refilled
          if (rest && lane == 0) {
            mbar_expect_tx(e_bar(ew), EPI_E_BYTES);
            tma_load_2d(ebuf_s, &mp->e, t.tn * BN + (__ffs(rest) - 1) * 32, gm0, e_bar(ew));
          }
        }
        if (p.gamma != 0.f) {
          #pragma unroll
          for (int j = 0; j < 32; ++j)
            if (gm0 + lane == gn0 + j) x[j] = __fadd_rn(x[j], p.gamma);
        }
        if (p.ssq != nullptr) ssq = chunk_sumsq(x, p.d_es, ssq);
        // without an addend the E buffer doubles as the mirror's staging box
        store_chunk(p, mp, x, gm0, gn0, lane, p.symmetric && gn0 == gm0, dbuf, dbuf_s,
                    has_e ? nullptr : ebuf, ebuf_s);
        __syncwarp();
      }
      ebuf_mirrored = !has_e && p.symmetric;
      if (p.ssq != nullptr)
        warp_sumsq_store(p.ssq + (int64_t(t.tm) * ((p.N + BN - 1) / BN) + t.tn) * kSsqSlots + ew, ssq,
                         lane);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1u;
    }
    if (lane == 0) tma_store_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

int g_num_sms = 0;

}  // namespace

bool tc_encode_maps(const GemmProblem& p, TcMaps* out) {
  std::memset(out, 0, sizeof(TcMaps));
  bool ok = encode_2d(&out->a, p.A, 2, p.K, p.M, p.lda, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (p.b_kmajor)
    ok = ok && encode_2d(&out->b, p.B, 2, p.K, p.N, p.ldb, BK, BN, CU_TENSOR_MAP_SWIZZLE_128B);
  else
    ok = ok && encode_2d(&out->b, p.B, 2, p.N, p.K, p.ldb, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B);
  if (p.E != nullptr)
    ok = ok && p.e_es == 2 &&
         encode_2d(&out->e, p.E, 2, p.N, p.M, p.lde, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
  if (p.d_es == 6)
    ok = ok && encode_2d(&out->d, p.D, 2, p.N, p.M, p.ldd, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B, 3, p.d_ps);
  else
    ok = ok && encode_2d(&out->d, p.D, p.d_es, p.N, p.M, p.ldd, p.d_es == 2 ? 32 : 16, 32,
                         CU_TENSOR_MAP_SWIZZLE_64B);
  return ok;
}

bool tc_available() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  return major == 10 && minor == 3;
}

int launch_gemm_tc(const GemmProblem* probs, const TcMaps* maps, const GemmTile* tiles,
                   int ntiles, const StepState* state, int* err_flag, cudaStream_t s) {
  if (ntiles <= 0) return 0;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(k_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
      return -1;
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    attr_set = true;
  }
  const int grid = ntiles < g_num_sms ? ntiles : g_num_sms;
  k_gemm_tc<<<grid, NTHREADS, SMEM_BYTES, s>>>(probs, maps, tiles, ntiles, state, err_flag);
  return 0;
}

}  // namespace muon
