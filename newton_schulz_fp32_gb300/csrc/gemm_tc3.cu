// FP32-accurate matrix products on the BF16 tensor cores (tcgen05).
//
// Every FP32 matrix of the FP32-operand mode (and of the gram recurrence) is
// stored as three bfloat16 planes whose sum is the value exactly:
//   x = hi + mid + lo,  hi = bf16(x), mid = bf16(x - hi), lo = x - hi - mid.
// A product A B expands into nine plane products; the six whose magnitude is
// above 2^-24 of the result (hi*hi, hi*mid, mid*hi, hi*lo, lo*hi, mid*mid)
// are accumulated in FP32 in tensor memory, which keeps single-precision
// accuracy at six BF16 MMAs per product (the BF16 rate is twice the TF32
// rate, so this matches three-pass TF32 in speed, with exact operand splits).
//
//   D = alpha * A op(B) + beta * E + gamma * I
//
// Layout: 128 x 128 output tiles, K steps of 32 (64-byte rows, 64-byte
// swizzle), 4-stage ring of 3 A planes + 3 B planes (48 KB per stage).
// Warp 0: TMA producer; warp 1: TMEM allocation and MMA issue; warps 2-5:
// epilogue (32 rows each): sums the addend's three planes, adds alpha*acc,
// gamma on the diagonal, and writes D as three planes (or bf16 / fp32),
// mirroring symmetric products.  All waits are bounded.
#include <cuda_bf16.h>

#include <cstring>

#include "tc_common.cuh"

namespace muon {
namespace {

using namespace tc;

constexpr int BM = 128, BN = 128, BK = 32;
constexpr int STAGES = 4;
constexpr int PLANE_A = BM * BK * 2;        // 8 KB
constexpr int PLANE_B = BN * BK * 2;        // 8 KB
constexpr int STAGE_BYTES = 3 * PLANE_A + 3 * PLANE_B;
// Accumulation: four fp32 accumulators of 128 columns (all 512 TMEM
// columns); K-block kb accumulates into slot kb % 4 and the epilogue adds the
// slots with round-to-nearest fp32 additions.  The tensor cores' fp32
// accumulation truncates at every MMA, and the error of a chain grows with
// its length, so four interleaved chains keep FP32-level accuracy on long K.
// One tile is in flight at a time (no room left for a second buffer).
constexpr int KSPLIT = 4;
constexpr int TMEM_COLS = KSPLIT * BN;
constexpr int EPI_WARPS = 4;
constexpr int NTHREADS = 64 + 32 * EPI_WARPS;
constexpr int EPI_E_BYTES = 3 * 32 * 32 * 2;   // three bf16 addend planes of a 32 x 32 chunk
constexpr int EPI_D_BYTES = 32 * 64;           // one 64-byte-row output box
constexpr int EPI_WARP_BYTES = EPI_E_BYTES + EPI_D_BYTES;
constexpr int EPI_BYTES = EPI_WARPS * EPI_WARP_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 4 + EPI_WARPS;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + 1024 + 256;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");


__global__ void __launch_bounds__(NTHREADS, 1)
k_gemm_x3(const GemmProblem* __restrict__ probs, const TcMaps* __restrict__ maps,
          const GemmTile* __restrict__ tiles, int ntiles, const StepState* state, int* err_flag) {
  if (state != nullptr && state->overflow) return;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  uint8_t* epi_base = base_ptr + STAGES * STAGE_BYTES;
  const uint32_t bar_base = base + STAGES * STAGE_BYTES + EPI_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + STAGES * STAGE_BYTES + EPI_BYTES);
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
      mbar_init(tempty_bar(i), EPI_WARPS);
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
      for (int ti = blockIdx.x; ti < ntiles && !*abort_flag; ti += gridDim.x) {
        const GemmTile t = tiles[ti];
        const GemmProblem& p = probs[t.problem];
        const TcMaps* mp = maps + t.problem;
        const int nk = (p.K + BK - 1) / BK;
        const bool b_k = p.b_kmajor != 0;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, err_flag, ERR_TIMEOUT_PRODUCER)) break;
          const uint32_t sa = base + s * STAGE_BYTES;
          const uint32_t sb = sa + 3 * PLANE_A;
          mbar_expect_tx(full_bar(s), STAGE_BYTES);
          #pragma unroll
          for (int pl = 0; pl < 3; ++pl) {
            tma_load_3d(sa + pl * PLANE_A, &mp->a, kb * BK, t.tm * BM, pl, full_bar(s));
            if (b_k) {
              tma_load_3d(sb + pl * PLANE_B, &mp->b, kb * BK, t.tn * BN, pl, full_bar(s));
            } else {
              #pragma unroll
              for (int j = 0; j < BN / 32; ++j)
                tma_load_3d(sb + pl * PLANE_B + j * (32 * BK * 2), &mp->b, t.tn * BN + j * 32,
                            kb * BK, pl, full_bar(s));
            }
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
      uint32_t acc_ph = 0;
      for (int ti = blockIdx.x; ti < ntiles && !*abort_flag; ti += gridDim.x) {
        const GemmTile t = tiles[ti];
        const GemmProblem& p = probs[t.problem];
        const int nk = (p.K + BK - 1) / BK;
        const bool b_k = p.b_kmajor != 0;
        const uint32_t idesc = make_idesc(!b_k, BM, BN);
        if (!mbar_wait(tempty_bar(0), acc_ph ^ 1u, abort_flag, err_flag, ERR_TIMEOUT_MMA)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(full_bar(s), ph, abort_flag, err_flag, ERR_TIMEOUT_MMA)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = base + s * STAGE_BYTES;
          const uint32_t sb = sa + 3 * PLANE_A;
          #pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {
            // the six plane products, smallest first: lo*hi, hi*lo, mid*mid,
            // mid*hi, hi*mid, hi*hi
            constexpr int kPA[6] = {2, 0, 1, 1, 0, 0};
            constexpr int kPB[6] = {0, 2, 1, 0, 1, 0};
            #pragma unroll
            for (int q = 0; q < 6; ++q) {
              const int pa = kPA[q], pb = kPB[q];
              // K-major, 64-byte swizzle: the 16-element K slice starts 32 B in
              const uint64_t ad = make_desc(sa + pa * PLANE_A + ks * 32, 16, 512, kSwizzle64);
              // MN-major B: 16 K-rows of 64 B further; 32-element MN chunks
              // 2 KB apart (LBO), 8-row K groups 512 B apart (SBO)
              const uint64_t bd = b_k ? make_desc(sb + pb * PLANE_B + ks * 32, 16, 512, kSwizzle64)
                                      : make_desc(sb + pb * PLANE_B + ks * 16 * 64, 32 * BK * 2, 512,
                                                  kSwizzle64);
              // slot kb % KSPLIT; the first MMA into a slot overwrites it
              const bool first = kb < KSPLIT && ks == 0 && q == 0;
              umma_bf16(d_tmem + static_cast<uint32_t>((kb % KSPLIT) * BN), ad, bd, idesc,
                        first ? 0u : 1u);
            }
          }
          umma_commit(empty_bar(s));
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        umma_commit(tfull_bar(0));
        acc_ph ^= 1u;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int ew = warp - 2;
    uint8_t* ebuf = epi_base + ew * EPI_WARP_BYTES;
    uint8_t* dbuf = ebuf + EPI_E_BYTES;
    const uint32_t ebuf_s = smem_u32(ebuf);
    const uint32_t dbuf_s = smem_u32(dbuf);
    uint32_t eph = 0u;
    uint32_t acc_ph = 0;
    bool ok = true;
    for (int ti = blockIdx.x; ti < ntiles && ok && !*abort_flag; ti += gridDim.x) {
      const GemmTile t = tiles[ti];
      const GemmProblem& p = probs[t.problem];
      const TcMaps* mp = maps + t.problem;
      const int gm0 = t.tm * BM + q * 32;
      uint32_t todo = 0;
      if (gm0 < p.M)
        for (int c = 0; c < BN / 32; ++c) {
          const int gn0 = t.tn * BN + c * 32;
          if (gn0 < p.N && !(p.symmetric && gn0 < gm0)) todo |= 1u << c;
        }
      const bool has_e = p.E != nullptr;
      auto load_e = [&](int c) {
        mbar_expect_tx(e_bar(ew), EPI_E_BYTES);
        #pragma unroll
        for (int pl = 0; pl < 3; ++pl)
          tma_load_3d(ebuf_s + pl * 2048, &mp->e, t.tn * BN + c * 32, gm0, pl, e_bar(ew));
      };
      if (has_e && todo && lane == 0) load_e(__ffs(todo) - 1);
      if (!mbar_wait(tfull_bar(0), acc_ph, abort_flag, err_flag, ERR_TIMEOUT_EPILOGUE)) {
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
        const uint32_t tcol = tmem_base + static_cast<uint32_t>(c * 32) +
                              (static_cast<uint32_t>(q * 32) << 16);
        tmem_ld32(tcol, x);
        const int used = min(KSPLIT, (p.K + BK - 1) / BK);   // slots that were written
        for (int sl = 1; sl < used; ++sl) {
          float y[32];
          tmem_ld32(tcol + sl * BN, y);
          #pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = __fadd_rn(x[j], y[j]);
        }
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
            const uint4 w0 = *reinterpret_cast<const uint4*>(ebuf + sw64(lane, g));
            const uint4 w1 = *reinterpret_cast<const uint4*>(ebuf + 2048 + sw64(lane, g));
            const uint4 w2 = *reinterpret_cast<const uint4*>(ebuf + 4096 + sw64(lane, g));
            const __nv_bfloat16* h0 = reinterpret_cast<const __nv_bfloat16*>(&w0);
            const __nv_bfloat16* h1 = reinterpret_cast<const __nv_bfloat16*>(&w1);
            const __nv_bfloat16* h2 = reinterpret_cast<const __nv_bfloat16*>(&w2);
            #pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float e = __fadd_rn(__fadd_rn(__bfloat162float(h0[u]), __bfloat162float(h1[u])),
                                        __bfloat162float(h2[u]));
              x[g * 8 + u] = __fadd_rn(x[g * 8 + u], __fmul_rn(p.beta, e));
            }
          }
          __syncwarp();
          if (rest && lane == 0) load_e(__ffs(rest) - 1);
        }
        if (p.gamma != 0.f) {
          #pragma unroll
          for (int j = 0; j < 32; ++j)
            if (gm0 + lane == gn0 + j) x[j] = __fadd_rn(x[j], p.gamma);
        }
        if (p.ssq != nullptr) ssq = chunk_sumsq(x, p.d_es, ssq);
        store_chunk(p, mp, x, gm0, gn0, lane, p.symmetric && gn0 == gm0, dbuf, dbuf_s);
        __syncwarp();
      }
      if (p.ssq != nullptr)
        warp_sumsq_store(p.ssq + (int64_t(t.tm) * ((p.N + BN - 1) / BN) + t.tn) * kSsqSlots + ew, ssq,
                         lane);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(0));
      acc_ph ^= 1u;
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

int g_sms = 0;

}  // namespace

bool x3_encode_maps(const GemmProblem& p, TcMaps* out) {
  std::memset(out, 0, sizeof(TcMaps));
  bool ok = encode_2d(&out->a, p.A, 2, p.K, p.M, p.lda, BK, BM, CU_TENSOR_MAP_SWIZZLE_64B, 3, p.a_ps);
  if (p.b_kmajor)
    ok = ok && encode_2d(&out->b, p.B, 2, p.K, p.N, p.ldb, BK, BN, CU_TENSOR_MAP_SWIZZLE_64B, 3, p.b_ps);
  else
    ok = ok && encode_2d(&out->b, p.B, 2, p.N, p.K, p.ldb, 32, BK, CU_TENSOR_MAP_SWIZZLE_64B, 3, p.b_ps);
  if (p.E != nullptr)
    ok = ok && p.e_es == 6 &&
         encode_2d(&out->e, p.E, 2, p.N, p.M, p.lde, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B, 3, p.e_ps);
  if (p.d_es == 6)
    ok = ok && encode_2d(&out->d, p.D, 2, p.N, p.M, p.ldd, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B, 3, p.d_ps);
  else
    ok = ok && encode_2d(&out->d, p.D, p.d_es, p.N, p.M, p.ldd, p.d_es == 2 ? 32 : 16, 32,
                         CU_TENSOR_MAP_SWIZZLE_64B);
  return ok;
}

int launch_gemm_x3(const GemmProblem* probs, const TcMaps* maps, const GemmTile* tiles, int ntiles,
                   const StepState* state, int* err_flag, cudaStream_t s) {
  if (ntiles <= 0) return 0;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(k_gemm_x3, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
        cudaSuccess)
      return -1;
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
    attr_set = true;
  }
  const int grid = ntiles < g_sms ? ntiles : g_sms;
  k_gemm_x3<<<grid, NTHREADS, SMEM_BYTES, s>>>(probs, maps, tiles, ntiles, state, err_flag);
  return 0;
}

}  // namespace muon
