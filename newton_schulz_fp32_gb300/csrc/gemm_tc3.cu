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
// swizzle), 3-stage ring of 3 A planes + 3 B planes (48 KB per stage).
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
constexpr int STAGES = 3;
constexpr int PLANE_A = BM * BK * 2;        // 8 KB
constexpr int PLANE_B = BN * BK * 2;        // 8 KB
constexpr int STAGE_BYTES = 3 * PLANE_A + 3 * PLANE_B;
// Accumulation: the tensor cores' fp32 accumulation truncates at every MMA
// and the error of a chain grows with its length, so a tile accumulates in
// several interleaved chains (K block kb into chain kb % chains) that the
// epilogue adds with round-to-nearest fp32 additions.  TMEM holds two
// buffers of 256 columns (two 128-column chains each).  Tiles with at most
// kNarrowNk K blocks use two chains in one buffer, so the next tile's MMAs
// overlap this tile's epilogue; longer tiles use four chains over both.
constexpr int BUF_COLS = 2 * BN;
constexpr int TMEM_COLS = 2 * BUF_COLS;
constexpr int kNarrowNk = 16;
constexpr int EPI_WARPS = 4;
constexpr int NTHREADS = 64 + 32 * EPI_WARPS;
// Per epilogue warp: an addend buffer, an output box and a mirror box, each
// a 32 x 32 chunk of three bf16 planes (2 KB each; a bf16 output uses the
// first plane, an fp32 output two 16-column boxes).
constexpr int CHUNK_BYTES = 3 * 32 * 32 * 2;
constexpr int EPI_WARP_BYTES = 3 * CHUNK_BYTES;
constexpr int EPI_BYTES = EPI_WARPS * EPI_WARP_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 4 + EPI_WARPS;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + 1024 + 256;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// Two floats to a packed bf16 pair, each rounded to nearest even (PTX
// cvt.rn.bf16x2.f32; the first argument lands in the low half).
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// split3 of 32 values, two at a time: pk[b][u] holds plane b (hi, mid, lo)
// of x[2u] (low half) and x[2u + 1] (high half).  Bit for bit the planes
// split3 gives, with one conversion per plane and pair.
__device__ __forceinline__ void split3_pack(const float* x, uint32_t (&pk)[3][16]) {
  #pragma unroll
  for (int u = 0; u < 16; ++u) {
    const float x0 = x[2 * u], x1 = x[2 * u + 1];
    const uint32_t h = bf16x2_rn(x0, x1);
    const float r0 = __fsub_rn(x0, __uint_as_float(h << 16));
    const float r1 = __fsub_rn(x1, __uint_as_float(h & 0xFFFF0000u));
    const uint32_t m = bf16x2_rn(r0, r1);
    const float l0 = __fsub_rn(r0, __uint_as_float(m << 16));
    const float l1 = __fsub_rn(r1, __uint_as_float(m & 0xFFFF0000u));
    pk[0][u] = h;
    pk[1][u] = m;
    pk[2][u] = bf16x2_rn(l0, l1);
  }
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            int w, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

// MN-major B whose columns come in whole groups of 32 is read through a
// 4-D view (32 columns, K rows, column groups, planes), so one copy moves a
// stage's whole B tile (4 groups x 3 planes); other MN-major B tiles are
// copied one 32-column group and plane at a time.
__host__ __device__ inline bool b_grouped(const GemmProblem& p) {
  return p.b_kmajor == 0 && p.N % 32 == 0;
}

// TMEM column of accumulation chain c of a tile whose first buffer is buf.
__device__ __forceinline__ uint32_t chain_col(int buf, int c) {
  return static_cast<uint32_t>(((buf + (c >> 1)) & 1) * BUF_COLS + (c & 1) * BN);
}

// The chunk's values (lane = row, x[j] = column j) in the output format:
// des 6: pk[b][u] holds plane b of columns 2u, 2u+1; des 2: pk[0] the bf16
// values; des 4: the fp32 values are taken from x.
__device__ __forceinline__ void pack_chunk(const float* x, int des, uint32_t (&pk)[3][16]) {
  if (des == 6) {
    split3_pack(x, pk);
  } else if (des == 2) {
    #pragma unroll
    for (int u = 0; u < 16; ++u) pk[0][u] = bf16x2_rn(x[2 * u], x[2 * u + 1]);
  }
}

// Stages the chunk by rows: box row `lane` = the lane's 32 values.
__device__ __forceinline__ void stage_rows(uint8_t* buf, const float* x, const uint32_t (&pk)[3][16],
                                           int lane, int des) {
  if (des == 4) {
    #pragma unroll
    for (int b = 0; b < 2; ++b)
      #pragma unroll
      for (int g = 0; g < 4; ++g) {
        const float* xs = x + 16 * b + 4 * g;
        *reinterpret_cast<uint4*>(buf + b * 2048 + sw64(lane, g)) =
            make_uint4(__float_as_uint(xs[0]), __float_as_uint(xs[1]), __float_as_uint(xs[2]),
                       __float_as_uint(xs[3]));
      }
    return;
  }
  const int planes = des == 6 ? 3 : 1;
  #pragma unroll
  for (int b = 0; b < 3; ++b) {
    if (b >= planes) break;
    #pragma unroll
    for (int g = 0; g < 4; ++g)
      *reinterpret_cast<uint4*>(buf + b * 2048 + sw64(lane, g)) =
          make_uint4(pk[b][4 * g], pk[b][4 * g + 1], pk[b][4 * g + 2], pk[b][4 * g + 3]);
  }
}

// Stages the chunk transposed: box row r, column `lane` = x[r], for rows
// r > lane only when lower_only (the mirror half of a diagonal chunk).
__device__ __forceinline__ void stage_cols(uint8_t* buf, const float* x, const uint32_t (&pk)[3][16],
                                           int lane, int des, bool lower_only) {
  if (des == 4) {
    uint8_t* bb = buf + (lane >> 4) * 2048;
    const int cl = lane & 15;
    #pragma unroll
    for (int r = 0; r < 32; ++r)
      if (!lower_only || r > lane)
        *reinterpret_cast<float*>(bb + sw64(r, cl >> 2) + (cl & 3) * 4) = x[r];
    return;
  }
  const int planes = des == 6 ? 3 : 1;
  #pragma unroll
  for (int b = 0; b < 3; ++b) {
    if (b >= planes) break;
    #pragma unroll
    for (int r = 0; r < 32; ++r)
      if (!lower_only || r > lane)
        *reinterpret_cast<uint16_t*>(buf + b * 2048 + sw64(r, lane >> 3) + (lane & 7) * 2) =
            static_cast<uint16_t>((r & 1) ? (pk[b][r >> 1] >> 16) : (pk[b][r >> 1] & 0xFFFFu));
  }
}

// Issues the TMA store(s) of one staged box at (column x0, row y0) of D and
// returns the number of bulk groups committed (one per store).  An fp32
// chunk is two 16-column boxes; the second is skipped when it starts past
// the last column.
__device__ __forceinline__ int issue_box(const TcMaps* mp, uint32_t buf_s, int x0, int y0, int des,
                                         int ncols) {
  if (des == 6) {
    tma_store_3d(&mp->d, x0, y0, 0, buf_s);
    return 1;
  }
  if (des == 2) {
    tma_store_2d(&mp->d, x0, y0, buf_s);
    return 1;
  }
  tma_store_2d(&mp->d, x0, y0, buf_s);
  if (x0 + 16 >= ncols) return 1;
  tma_store_2d(&mp->d, x0 + 16, y0, buf_s + 2048);
  return 2;
}

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
        const bool b_g = b_grouped(p);
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, err_flag, ERR_TIMEOUT_PRODUCER)) break;
          const uint32_t sa = base + s * STAGE_BYTES;
          const uint32_t sb = sa + 3 * PLANE_A;
          mbar_expect_tx(full_bar(s), STAGE_BYTES);
          // A and K-major B: one box of all three planes each
          tma_load_3d(sa, &mp->a, kb * BK, t.tm * BM, 0, full_bar(s));
          if (b_k) {
            tma_load_3d(sb, &mp->b, kb * BK, t.tn * BN, 0, full_bar(s));
          } else if (b_g) {
            tma_load_4d(sb, &mp->b, 0, kb * BK, t.tn * (BN / 32), 0, full_bar(s));
          } else {
            #pragma unroll
            for (int pl = 0; pl < 3; ++pl)
              #pragma unroll
              for (int j = 0; j < BN / 32; ++j)
                tma_load_3d(sb + pl * PLANE_B + j * (32 * BK * 2), &mp->b, t.tn * BN + j * 32,
                            kb * BK, pl, full_bar(s));
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
      int buf = 0;        // first TMEM buffer of the next tile
      uint32_t bph = 0;   // bit b: use parity of buffer b
      for (int ti = blockIdx.x; ti < ntiles && !*abort_flag; ti += gridDim.x) {
        const GemmTile t = tiles[ti];
        const GemmProblem& p = probs[t.problem];
        const int nk = (p.K + BK - 1) / BK;
        const int chains = nk <= kNarrowNk ? 2 : 4;
        const int nbuf = chains / 2;
        const bool b_k = p.b_kmajor != 0;
        // MMA width: the tile's columns inside the matrix, rounded up to 32
        // (the epilogue reads no column beyond it)
        const int n_eff = min(BN, (p.N - t.tn * BN + 31) & ~31);
        const uint32_t idesc = make_idesc(!b_k, BM, n_eff);
        bool ok = true;
        for (int i = 0; i < nbuf && ok; ++i) {
          const int b = (buf + i) & 1;
          ok = mbar_wait(tempty_bar(b), ((bph >> b) & 1u) ^ 1u, abort_flag, err_flag, ERR_TIMEOUT_MMA);
        }
        if (!ok) break;
        tc_fence_after();
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(full_bar(s), ph, abort_flag, err_flag, ERR_TIMEOUT_MMA)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = base + s * STAGE_BYTES;
          const uint32_t sb = sa + 3 * PLANE_A;
          const int c = kb % chains;
          const uint32_t d_tmem = tmem_base + chain_col(buf, c);
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
              // the first MMA into a chain overwrites it
              const bool first = kb < chains && ks == 0 && q == 0;
              umma_bf16(d_tmem, ad, bd, idesc, first ? 0u : 1u);
            }
          }
          umma_commit(empty_bar(s));
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        for (int i = 0; i < nbuf; ++i) {
          const int b = (buf + i) & 1;
          umma_commit(tfull_bar(b));
          bph ^= 1u << b;
        }
        buf = (buf + nbuf) & 1;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int ew = warp - 2;
    uint8_t* ebuf = epi_base + ew * EPI_WARP_BYTES;
    uint8_t* dbuf = ebuf + CHUNK_BYTES;
    uint8_t* mbuf = dbuf + CHUNK_BYTES;
    const uint32_t ebuf_s = smem_u32(ebuf);
    const uint32_t dbuf_s = smem_u32(dbuf);
    const uint32_t mbuf_s = smem_u32(mbuf);
    uint32_t eph = 0u;
    int buf = 0;
    uint32_t bph = 0;
    // bulk groups committed by lane 0 so far, and the count right after the
    // last store from the output box and from the mirror box
    int groups = 0, g_d = 0, g_m = 0;
    bool ok = true;
    for (int ti = blockIdx.x; ti < ntiles && ok && !*abort_flag; ti += gridDim.x) {
      const GemmTile t = tiles[ti];
      const GemmProblem& p = probs[t.problem];
      const TcMaps* mp = maps + t.problem;
      const int nk = (p.K + BK - 1) / BK;
      const int chains = nk <= kNarrowNk ? 2 : 4;
      const int nbuf = chains / 2;
      const int used = min(chains, nk);   // chains that were written
      const int gm0 = t.tm * BM + q * 32;
      uint32_t todo = 0;
      if (gm0 < p.M)
        for (int c = 0; c < BN / 32; ++c) {
          const int gn0 = t.tn * BN + c * 32;
          if (gn0 < p.N && !(p.symmetric && gn0 < gm0)) todo |= 1u << c;
        }
      const bool has_e = p.E != nullptr;
      auto load_e = [&](int c) {
        mbar_expect_tx(e_bar(ew), CHUNK_BYTES);
        tma_load_3d(ebuf_s, &mp->e, t.tn * BN + c * 32, gm0, 0, e_bar(ew));
      };
      if (has_e && todo && lane == 0) load_e(__ffs(todo) - 1);
      for (int i = 0; i < nbuf && ok; ++i) {
        const int b = (buf + i) & 1;
        ok = mbar_wait(tfull_bar(b), (bph >> b) & 1u, abort_flag, err_flag, ERR_TIMEOUT_EPILOGUE);
      }
      if (!ok) break;
      tc_fence_after();
      const int des = p.d_es;
      const bool sym = p.symmetric != 0;
      float ssq = 0.f;   // this warp's sum of squares of the tile (last product only)
      uint32_t rest = todo;
      while (rest) {
        const int c = __ffs(rest) - 1;
        rest &= rest - 1;
        const int gn0 = t.tn * BN + c * 32;
        float x[32];
        const uint32_t lanes = static_cast<uint32_t>(q * 32) << 16;
        tmem_ld32(tmem_base + chain_col(buf, 0) + static_cast<uint32_t>(c * 32) + lanes, x);
        for (int ch = 1; ch < used; ++ch) {
          float y[32];
          tmem_ld32(tmem_base + chain_col(buf, ch) + static_cast<uint32_t>(c * 32) + lanes, y);
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
        if (p.ssq != nullptr) ssq = chunk_sumsq(x, des, ssq);
        uint32_t pk[3][16];
        pack_chunk(x, des, pk);
        // the output box: rows of this chunk; a diagonal chunk of a
        // symmetric product takes its strictly lower half from the upper
        // half (transposed), so D is exactly symmetric
        const bool diag = sym && gn0 == gm0;
        if (lane == 0) bulk_wait_read_n(groups - g_d);
        __syncwarp();
        stage_rows(dbuf, x, pk, lane, des);
        if (diag) {
          __syncwarp();
          stage_cols(dbuf, x, pk, lane, des, true);
        }
        fence_async_smem();
        __syncwarp();
        groups += lane == 0 ? issue_box(mp, dbuf_s, gn0, gm0, des, p.N) : (des == 4 && gn0 + 16 < p.N ? 2 : 1);
        g_d = groups;
        if (sym && !diag) {   // the mirror chunk at (gn0, gm0)
          if (lane == 0) bulk_wait_read_n(groups - g_m);
          __syncwarp();
          stage_cols(mbuf, x, pk, lane, des, false);
          fence_async_smem();
          __syncwarp();
          groups += lane == 0 ? issue_box(mp, mbuf_s, gm0, gn0, des, p.M) : (des == 4 && gm0 + 16 < p.M ? 2 : 1);
          g_m = groups;
        }
      }
      if (p.ssq != nullptr)
        warp_sumsq_store(p.ssq + (int64_t(t.tm) * ((p.N + BN - 1) / BN) + t.tn) * kSsqSlots + ew, ssq,
                         lane);
      tc_fence_before();
      __syncwarp();
      for (int i = 0; i < nbuf; ++i) {
        const int b = (buf + i) & 1;
        if (lane == 0) mbar_arrive(tempty_bar(b));
        bph ^= 1u << b;
      }
      buf = (buf + nbuf) & 1;
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

namespace {
// 4-D view of an MN-major split-3 B (K rows of N columns, N % 32 == 0):
// (32 columns, K rows, N / 32 column groups, 3 planes); a box of
// (32, BK, BN / 32, 3) lands in shared memory as [plane][group][row][32].
bool encode_b_grouped(CUtensorMap* m, const GemmProblem& p) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {32, static_cast<cuuint64_t>(p.K), static_cast<cuuint64_t>(p.N / 32), 3};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(p.ldb * 2), 64,
                           static_cast<cuuint64_t>(p.b_ps * 2)};
  cuuint32_t box[4] = {32, BK, BN / 32, 3};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(p.B), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A map over three bf16 planes `pstride` elements apart whose box spans all
// three: one TMA copy moves a whole split-3 box (an operand tile of one
// K step, or a 32 x 32 addend or output chunk).
bool encode_planes_box(CUtensorMap* m, const void* base, int64_t inner, int64_t outer, int64_t ld,
                       int64_t pstride, uint32_t box_inner = 32, uint32_t box_outer = 32) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer), 3};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * 2), static_cast<cuuint64_t>(pstride * 2)};
  cuuint32_t box[3] = {box_inner, box_outer, 3};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

bool x3_encode_maps(const GemmProblem& p, TcMaps* out) {
  std::memset(out, 0, sizeof(TcMaps));
  // A and K-major B: boxes of all three planes (one copy per stage each)
  bool ok = encode_planes_box(&out->a, p.A, p.K, p.M, p.lda, p.a_ps, BK, BM);
  if (p.b_kmajor)
    ok = ok && encode_planes_box(&out->b, p.B, p.K, p.N, p.ldb, p.b_ps, BK, BN);
  else if (b_grouped(p))
    ok = ok && encode_b_grouped(&out->b, p);
  else
    ok = ok && encode_2d(&out->b, p.B, 2, p.N, p.K, p.ldb, 32, BK, CU_TENSOR_MAP_SWIZZLE_64B, 3, p.b_ps);
  // addend and split-3 output boxes carry all three planes of a 32 x 32 chunk
  if (p.E != nullptr)
    ok = ok && p.e_es == 6 && encode_planes_box(&out->e, p.E, p.N, p.M, p.lde, p.e_ps);
  if (p.d_es == 6)
    ok = ok && encode_planes_box(&out->d, p.D, p.N, p.M, p.ldd, p.d_ps);
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
