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

#include "muon_internal.h"

namespace muon {
namespace {

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
constexpr unsigned long long kTimeoutNs = 2000000000ull;

enum : int { ERR_TIMEOUT_PRODUCER = 1, ERR_TIMEOUT_MMA = 2, ERR_TIMEOUT_EPILOGUE = 3 };

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait; returns false (and raises the abort flag) on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* err_flag, int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kTimeoutNs) {
      *abort_flag = 1;
      if (err_flag) atomicExch(err_flag, code);
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void tma_store_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Byte offset of 16-byte granule `granule` of row `row` in a box of 64-byte
// rows under the 64-byte swizzle (granule index XOR bits 7-8 of the offset).
__device__ __forceinline__ uint32_t sw64(int row, int granule) {
  return uint32_t(row) * 64u + (uint32_t(granule ^ ((row >> 1) & 3)) << 4);
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (16-byte units), fixed version bits 46-47 = 1,
// swizzle mode 2 (128-byte) in bits 61-63.
__device__ __forceinline__ uint64_t make_desc(uint32_t saddr, uint32_t lbo_bytes,
                                              uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, A K-major,
// B K-major or MN-major, N = 256, M = 128.
__host__ __device__ constexpr uint32_t make_idesc(bool b_mn_major) {
  return (1u << 4)                 // D format: f32
         | (1u << 7)               // A format: bf16
         | (1u << 10)              // B format: bf16
         | (0u << 15)              // A K-major
         | ((b_mn_major ? 1u : 0u) << 16)
         | (static_cast<uint32_t>(BN >> 3) << 17)
         | (static_cast<uint32_t>(BM >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 columns of fp32 from tensor memory; thread i gets row
// (lane base + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  #pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Writes one 32 x 32 output chunk held by one warp (lane = row, x = the
// finished fp32 values).  Off the diagonal the chunk is staged in `dbuf` in
// the 64-byte-swizzled layout and written by TMA stores (which clip rows >= M
// and columns >= N): one box for bf16, two 16-column boxes for fp32.  A
// chunk above the diagonal of a symmetric product is also written transposed
// to its mirror position with direct stores (lanes hold consecutive rows, so
// each store instruction covers 64 or 128 contiguous bytes).  A chunk on the
// diagonal is written directly: its upper triangle (with the diagonal) by
// rows and its strictly upper part again as the mirror, so the lower
// triangle is an exact copy of the upper.
__device__ __forceinline__ void store_chunk(const GemmProblem& p, const TcMaps* mp, const float* x,
                                            int gm0, int gn0, int lane, bool diag, uint8_t* dbuf,
                                            uint32_t dbuf_s) {
  const int gm = gm0 + lane;
  const bool f32 = p.d_es == 4;
  if (diag) {
    if (gm >= p.M) return;
    #pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int gn = gn0 + j;
      if (gn >= p.N || j < lane) continue;
      if (f32) {
        float* D = reinterpret_cast<float*>(p.D);
        D[int64_t(gm) * p.ldd + gn] = x[j];
        if (j > lane) D[int64_t(gn) * p.ldd + gm] = x[j];
      } else {
        __nv_bfloat16* D = reinterpret_cast<__nv_bfloat16*>(p.D);
        const __nv_bfloat16 o = __float2bfloat16_rn(x[j]);
        D[int64_t(gm) * p.ldd + gn] = o;
        if (j > lane) D[int64_t(gn) * p.ldd + gm] = o;
      }
    }
    return;
  }
  #pragma unroll
  for (int h = 0; h < 2; ++h) {
    const bool live = (h == 0) || (f32 && gn0 + 16 < p.N);   // warp-uniform
    if (!live) continue;
    if (lane == 0) tma_store_wait_read();   // the previous store has read dbuf
    __syncwarp();
    #pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint4 w;
      if (f32) {
        const float* xs = x + 16 * h + 4 * g;
        w = make_uint4(__float_as_uint(xs[0]), __float_as_uint(xs[1]), __float_as_uint(xs[2]),
                       __float_as_uint(xs[3]));
      } else {
        __nv_bfloat162 hh[4];
        #pragma unroll
        for (int u = 0; u < 4; ++u) hh[u] = __floats2bfloat162_rn(x[8 * g + 2 * u], x[8 * g + 2 * u + 1]);
        w = *reinterpret_cast<const uint4*>(hh);
      }
      *reinterpret_cast<uint4*>(dbuf + sw64(lane, g)) = w;
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) tma_store_2d(&mp->d, gn0 + 16 * h, gm0, dbuf_s);
  }
  if (p.symmetric && gm < p.M) {
    if (f32) {
      float* D = reinterpret_cast<float*>(p.D);
      #pragma unroll
      for (int j = 0; j < 32; ++j)
        if (gn0 + j < p.N) D[int64_t(gn0 + j) * p.ldd + gm] = x[j];
    } else {
      __nv_bfloat16* D = reinterpret_cast<__nv_bfloat16*>(p.D);
      #pragma unroll
      for (int j = 0; j < 32; ++j)
        if (gn0 + j < p.N) D[int64_t(gn0 + j) * p.ldd + gm] = __float2bfloat16_rn(x[j]);
    }
  }
}

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
        const uint32_t idesc = make_idesc(!b_k);
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
            const uint64_t ad = make_desc(sa + k * 32, 16, 1024);
            // K-major B: same; MN-major B: 16 K-rows of 128 bytes further,
            // 64-element MN chunks 8 KB apart (LBO), 8-row K groups 1 KB (SBO)
            const uint64_t bd = b_k ? make_desc(sb + k * 32, 16, 1024)
                                    : make_desc(sb + k * 16 * 128, 64 * BK * 2, 1024);
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
    const int c_lo = (ew >> 2) * 4;               // its chunks: columns [32 c_lo, 32 c_lo + 128)
    uint8_t* ebuf = epi_base + ew * EPI_WARP_BYTES;
    uint8_t* dbuf = ebuf + EPI_E_BYTES;
    const uint32_t ebuf_s = smem_u32(ebuf);
    const uint32_t dbuf_s = smem_u32(dbuf);
    uint32_t eph = 0u;
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
        for (int c = c_lo; c < c_lo + 4; ++c) {
          const int gn0 = t.tn * BN + c * 32;
          if (gn0 < p.N && !(p.symmetric && gn0 < gm0)) todo |= 1u << c;
        }
      const bool has_e = p.E != nullptr;
      if (has_e && todo && lane == 0) {   // prefetch the first addend chunk
        mbar_expect_tx(e_bar(ew), EPI_E_BYTES);
        tma_load_2d(ebuf_s, &mp->e, t.tn * BN + (__ffs(todo) - 1) * 32, gm0, e_bar(ew));
      }
      if (!mbar_wait(tfull_bar(acc), acc_ph, abort_flag, err_flag, ERR_TIMEOUT_EPILOGUE)) {
        ok = false;
        break;
      }
      tc_fence_after();
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
        store_chunk(p, mp, x, gm0, gn0, lane, p.symmetric && gn0 == gm0, dbuf, dbuf_s);
        __syncwarp();
      }
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

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2-D map over a row-major matrix: `inner` elements per row, `outer` rows,
// row stride `ld` elements.
bool encode_2d(CUtensorMap* m, const void* base, int es, int64_t inner, int64_t outer, int64_t ld,
               uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * es)};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, es == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

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
