// Tensor-core matrix products on SM pairs: tcgen05.mma.cta_group::2 with
// 256 x 256 output tiles, BF16 operands, FP32 accumulation in the tensor
// memory of both SMs.
//
//   D = alpha * A op(B) + beta * E + gamma * I     (D, E bf16; epilogue fp32)
//
// One persistent cluster of two CTAs per SM pair takes tasks -- (problem,
// 256 x 256 tile) -- from a task list in order through a global counter.
// A task may name a dependency: a counter that the tiles of an earlier
// product of the same Newton-Schulz problem raise when their outputs are
// in memory; the task's operands are loaded only once it has reached its
// target.  All products of an iteration can so run in one launch (a
// dataflow over the problems): a problem's next product starts as soon as
// its previous one is complete, whatever the other problems are doing,
// instead of waiting at a launch boundary for every problem's previous
// product.  Tasks depend only on earlier tasks and every cluster is
// resident, so the earliest unfinished task can always progress.
//
// Per K block of 64, CTA r loads rows [128 r, 128 r + 128) of the A tile and
// columns [128 r, 128 r + 128) of the B tile into its own shared memory; the
// even CTA's single MMA thread issues M=256, N=256 MMAs that read both
// halves, and each CTA ends up holding its 128 rows x 256 columns of the
// tile in its tensor memory.  Per K block an SM loads 32 KB for a
// 128 x 256 x 64 product (a single-SM 128 x 256 tile needs 48 KB).
//
// Warp roles per CTA:
//   warp 0      TMA producer (both CTAs), 5-stage ring of 32 KB stages; the
//               loads of both CTAs complete on the even CTA's full barrier.
//               In the even CTA it also fetches the tasks, waits for their
//               dependencies and publishes them to both CTAs through a
//               4-slot task ring.
//   warp 1      TMEM allocation for the pair (512 columns: two 128 x 256
//               FP32 accumulators per CTA); in the even CTA also the MMA
//               issuer, whose commits release both CTAs' stages and
//               accumulators
//   warps 2-9   epilogue of this CTA's 128 rows: addend chunks by TMA,
//               FP32 alpha/beta/gamma, BF16 TMA stores through two
//               alternating boxes, a box of its own for the transposed chunk
//               of symmetric products; then, for
//               tasks that others depend on, the warps wait for their stores
//               to complete and one raises the task's counter (release, GPU
//               scope): a tile is complete at 2 arrivals, one per CTA.
//
// Every wait is bounded: after ~2 s without progress a CTA records an error
// code, stops issuing work, lets its copies in flight land, frees its
// tensor memory and exits.
#include <cuda_bf16.h>

#include <cstring>

#include "tc_common.cuh"

namespace muon {
namespace {

using namespace tc;

constexpr int BM = 256, BMC = 128, BN = 256, BK = 64;   // pair tile, rows per CTA
constexpr int STAGES = 5;
constexpr int A_BYTES = BMC * BK * 2;         // 16 KB
constexpr int B_BYTES = (BN / 2) * BK * 2;    // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int EPI_WARPS = 8;
constexpr int NTHREADS = 64 + 32 * EPI_WARPS;
constexpr int EPI_E_BYTES = 32 * 32 * 2;
constexpr int EPI_D_BYTES = 32 * 64;
constexpr int EPI_M_BYTES = 32 * 64;                 // mirrored chunk of a symmetric product
constexpr int EPI_WARP_BYTES = EPI_E_BYTES + 2 * EPI_D_BYTES + EPI_M_BYTES;   // two output boxes
constexpr int EPI_BYTES = EPI_WARPS * EPI_WARP_BYTES;
constexpr int TASK_SLOTS = 4;
constexpr int SLOT_INTS = 6;   // task ring entry: index, problem, tm, tn, nk | b_kmajor << 16, done
// full, empty per stage; tfull, tempty per accumulator; E per epilogue
// warp; task full, task empty per task slot
constexpr int NUM_BARS = 2 * STAGES + 4 + EPI_WARPS + 2 * TASK_SLOTS;
constexpr int kEpiBarrier = 1;   // named barrier of the epilogue warps
constexpr int TASK_CONSUMERS = 2 + 2 * EPI_WARPS;     // peer producer, MMA, epilogue warps of both
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + 1024 + 512;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(NUM_BARS * 8 + 8 + 4 * SLOT_INTS * TASK_SLOTS <= 512, "barrier and task-ring area");
static_assert(kTcPairBM == BM && kTcPairBN == BN && kTcBK == BK, "tile shape shared with the planner");
constexpr int ERR_TIMEOUT_DEP = 4;

// A task as published in the ring: everything the MMA issuer needs, so it
// issues without dependent global loads.
struct TaskInfo {
  int ti, problem, tm, tn, nk, bk, done;
};

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait for a dependency counter to reach `target`.
__device__ __forceinline__ bool wait_counter(const int* ctr, int target, volatile int* abort_flag,
                                             int* err_flag) {
  if (ld_acquire(ctr) >= target) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    __nanosleep(64);
    if (ld_acquire(ctr) >= target) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kTimeoutNs) {
      *abort_flag = 1;
      if (err_flag) atomicExch(err_flag, ERR_TIMEOUT_DEP);
      return false;
    }
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
k_gemm_tc2(const GemmProblem* __restrict__ probs, const TcMaps* __restrict__ maps,
           const PairTask* __restrict__ tasks, int ntasks, int* counters, const StepState* state,
           int* err_flag) {
  // uniform over the pair: both CTAs leave together
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
  auto qfull_bar = [&](int i) { return bar_base + 8u * (2 * STAGES + 4 + EPI_WARPS + i); };
  auto qempty_bar = [&](int i) {
    return bar_base + 8u * (2 * STAGES + 4 + EPI_WARPS + TASK_SLOTS + i);
  };

  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + NUM_BARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS) + 1;
  int* task_slot = reinterpret_cast<int*>(bars + NUM_BARS) + 2;    // TASK_SLOTS x SLOT_INTS
  const uint32_t task_slot_s = smem_u32(task_slot);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();      // 0: fetches tasks and issues the MMAs

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);                 // the even CTA's arrive + both CTAs' bytes
      mbar_init(empty_bar(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull_bar(i), 1);
      mbar_init(tempty_bar(i), 2 * EPI_WARPS);   // epilogue warps of both CTAs
    }
    for (int w = 0; w < EPI_WARPS; ++w) mbar_init(e_bar(w), 1);
    for (int i = 0; i < TASK_SLOTS; ++i) {
      mbar_init(qfull_bar(i), 1);                // the even CTA's producer publishes
      mbar_init(qempty_bar(i), TASK_CONSUMERS);  // used in the even CTA
    }

    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    // one warp of each CTA of the pair allocates, collectively
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  __syncwarp();
  tc_fence_before();
  cluster_sync();   // barriers of both CTAs initialised, tensor memory allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Task ring, consumer side: the next task (ti = -1: no more); the slot is
  // then handed back to the even CTA's producer.
  // In the even CTA the producer and the consumers share the CTA, so
  // CTA-scope acquire / release suffice; the odd CTA synchronises with the
  // even CTA's producer at cluster scope.
  auto take_task = [&](int& slot, uint32_t& qph) -> TaskInfo {
    TaskInfo r{-1, 0, 0, 0, 0, 0, -1};
    const bool got = rank == 0
        ? mbar_wait(qfull_bar(slot), qph, abort_flag, err_flag, ERR_TIMEOUT_MMA)
        : mbar_wait_cluster(qfull_bar(slot), qph, abort_flag, err_flag, ERR_TIMEOUT_MMA);
    if (!got) return r;
    const volatile int* e = task_slot + slot * SLOT_INTS;
    r.ti = e[0];
    r.problem = e[1];
    r.tm = e[2];
    r.tn = e[3];
    r.nk = e[4] & 0xffff;
    r.bk = e[4] >> 16;
    r.done = e[5];
    if (rank == 0) mbar_arrive(qempty_bar(slot));
    else mbar_arrive_cluster(mapa_shared(qempty_bar(slot), 0));
    if (++slot == TASK_SLOTS) { slot = 0; qph ^= 1u; }
    return r;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int qs = 0;
      uint32_t qph = 0;
      int last_problem = -1;
      // the even CTA fetches one task ahead, so the atomic's round trip
      // overlaps the loads of the task before
      int next = rank == 0 ? atomicAdd(counters, 1) : -1;
      while (!*abort_flag) {
        TaskInfo t{-1, 0, 0, 0, 0, 0, -1};
        if (rank == 0) {
          // take the fetched task, wait for its dependency, publish it
          if (!mbar_wait_cluster(qempty_bar(qs), qph ^ 1u, abort_flag, err_flag, ERR_TIMEOUT_PRODUCER))
            break;
          const int ti = next < ntasks ? next : -1;
          if (ti >= 0) {
            next = atomicAdd(counters, 1);
            const PairTask pt = tasks[ti];
            t = TaskInfo{ti, pt.problem, pt.tm, pt.tn, pt.nk, pt.b_kmajor != 0 ? 1 : 0, pt.done};
            if (pt.dep >= 0 && !wait_counter(counters + pt.dep, pt.dep_target, abort_flag, err_flag))
              break;
          }
          const int e[SLOT_INTS] = {t.ti, t.problem, t.tm, t.tn, t.nk | (t.bk << 16), t.done};
          const uint32_t remote = mapa_shared(task_slot_s + 4u * SLOT_INTS * qs, 1);
          #pragma unroll
          for (int i = 0; i < SLOT_INTS; ++i) {
            task_slot[qs * SLOT_INTS + i] = e[i];
            asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote + 4u * i), "r"(e[i]) : "memory");
          }
          mbar_arrive(qfull_bar(qs));
          mbar_arrive_cluster(mapa_shared(qfull_bar(qs), 1));
          if (++qs == TASK_SLOTS) { qs = 0; qph ^= 1u; }
        } else {
          t = take_task(qs, qph);
        }
        if (t.ti < 0) break;
        // the operands were written by other SMs (generic release / acquire
        // above); order the TMA reads after that
        asm volatile("fence.proxy.async.global;" ::: "memory");
        const TcMaps* mp = maps + t.problem;
        if (t.problem != last_problem) {
          asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mp->a)));
          asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mp->b)));
          last_problem = t.problem;
        }
        const int nk = t.nk;
        const bool b_k = t.bk != 0;
        const int row0 = t.tm * BM + static_cast<int>(rank) * BMC;        // this CTA's A rows
        const int col0 = t.tn * BN + static_cast<int>(rank) * (BN / 2);   // this CTA's B columns
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, err_flag, ERR_TIMEOUT_PRODUCER)) break;
          const uint32_t sa = base + s * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          const uint32_t fb = mapa_shared(full_bar(s), 0);
          if (rank == 0) mbar_expect_tx(full_bar(s), 2 * STAGE_BYTES);
          tma_load_2d_pair(sa, &mp->a, kb * BK, row0, fb);
          if (b_k) {
            tma_load_2d_pair(sb, &mp->b, kb * BK, col0, fb);
          } else {
            #pragma unroll
            for (int j = 0; j < (BN / 2) / 64; ++j)
              tma_load_2d_pair(sb + j * (64 * BK * 2), &mp->b, col0 + j * 64, kb * BK, fb);
          }
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      int s = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t acc_ph = 0;
      int qs = 0;
      uint32_t qph = 0;
      while (!*abort_flag) {
        const TaskInfo t = take_task(qs, qph);
        if (t.ti < 0) break;
        const int nk = t.nk;
        const bool b_k = t.bk != 0;
        const uint32_t idesc = make_idesc(!b_k, BM, BN);
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
            const uint64_t ad = make_desc(sa + k * 32, 16, 1024, kSwizzle128);
            const uint64_t bd = b_k ? make_desc(sb + k * 32, 16, 1024, kSwizzle128)
                                    : make_desc(sb + k * 16 * 128, 64 * BK * 2, 1024, kSwizzle128);
            umma_bf16_pair(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit_pair(empty_bar(s), 0x3);   // frees this stage in both CTAs
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        umma_commit_pair(tfull_bar(acc), 0x3);   // both CTAs' accumulators ready
        acc ^= 1;
        if (acc == 0) acc_ph ^= 1u;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int ew = warp - 2;
    // the two warps of a lane quarter take alternate 32-column chunks, so
    // the upper-triangle chunks of a diagonal tile (and their mirrors) are
    // shared evenly between them
    const int c_par = ew >> 2;
    uint8_t* ebuf = epi_base + ew * EPI_WARP_BYTES;
    uint8_t* dbuf = ebuf + EPI_E_BYTES;
    uint8_t* mbuf = dbuf + 2 * EPI_D_BYTES;
    // bulk groups committed by lane 0, and the count right after the last
    // store out of each box: a box may be refilled once at most (groups -
    // that count) newer groups still read their sources
    int groups = 0, g_d[2] = {0, 0}, g_m = 0, dsel = 0;
    const uint32_t ebuf_s = smem_u32(ebuf);
    const uint32_t dbuf_s = smem_u32(dbuf);
    const uint32_t mbuf_s = smem_u32(mbuf);
    uint32_t eph = 0u;
    int acc = 0;
    uint32_t acc_ph = 0;
    int qs = 0;
    uint32_t qph = 0;
    bool ok = true;
    bool finished = false;   // left the loop on the end-of-tasks marker
    while (ok && !*abort_flag) {
      // lane 0 takes the task for the warp and hands the slot back
      TaskInfo t{-1, 0, 0, 0, 0, 0, -1};
      if (lane == 0) {
        t = take_task(qs, qph);
      } else if (++qs == TASK_SLOTS) {
        qs = 0;
        qph ^= 1u;
      }
      t.ti = __shfl_sync(0xffffffffu, t.ti, 0);
      if (t.ti < 0) {
        finished = !*abort_flag;
        break;
      }
      t.problem = __shfl_sync(0xffffffffu, t.problem, 0);
      t.tm = __shfl_sync(0xffffffffu, t.tm, 0);
      t.tn = __shfl_sync(0xffffffffu, t.tn, 0);
      t.done = __shfl_sync(0xffffffffu, t.done, 0);
      const GemmProblem& p = probs[t.problem];
      if (p.E != nullptr && lane == 0)   // addends come from other SMs
        asm volatile("fence.proxy.async.global;" ::: "memory");
      const TcMaps* mp = maps + t.problem;
      const int gm0 = t.tm * BM + static_cast<int>(rank) * BMC + q * 32;
      uint32_t todo = 0;
      if (gm0 < p.M)
        for (int c = c_par; c < BN / 32; c += 2) {
          const int gn0 = t.tn * BN + c * 32;
          if (gn0 < p.N && !(p.symmetric && gn0 < gm0)) todo |= 1u << c;
        }
      const bool has_e = p.E != nullptr;
      // addend chunks arrive by TMA one chunk ahead
      auto load_e = [&](int c) {   // lane 0
        mbar_expect_tx(e_bar(ew), EPI_E_BYTES);
        tma_load_2d(ebuf_s, &mp->e, t.tn * BN + c * 32, gm0, e_bar(ew));
      };
      if (has_e && todo && lane == 0) load_e(__ffs(todo) - 1);
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
          const uint8_t* eb = ebuf;
          #pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint4 w = *reinterpret_cast<const uint4*>(eb + sw64(lane, g));
            const __nv_bfloat162* hh = reinterpret_cast<const __nv_bfloat162*>(&w);
            #pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float2 f = __bfloat1622float2(hh[u]);
              x[g * 8 + 2 * u] = __fadd_rn(x[g * 8 + 2 * u], __fmul_rn(p.beta, f.x));
              x[g * 8 + 2 * u + 1] = __fadd_rn(x[g * 8 + 2 * u + 1], __fmul_rn(p.beta, f.y));
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
        const bool diag = p.symmetric && gn0 == gm0;
        if (p.d_es == 2 && !diag) {
          // BF16 box through alternating staging boxes, then the mirror
          const int b = dsel;
          dsel ^= 1;
          uint8_t* db = dbuf + b * EPI_D_BYTES;
          if (lane == 0) bulk_wait_read_n(groups - g_d[b]);
          __syncwarp();
          #pragma unroll
          for (int g = 0; g < 4; ++g) {
            __nv_bfloat162 h[4];
            #pragma unroll
            for (int u = 0; u < 4; ++u)
              h[u] = __floats2bfloat162_rn(x[8 * g + 2 * u], x[8 * g + 2 * u + 1]);
            *reinterpret_cast<uint4*>(db + sw64(lane, g)) = *reinterpret_cast<const uint4*>(h);
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) tma_store_2d(&mp->d, gn0, gm0, dbuf_s + b * EPI_D_BYTES);
          g_d[b] = ++groups;
          if (p.symmetric) {
            if (lane == 0) bulk_wait_read_n(groups - g_m);
            __syncwarp();
            #pragma unroll
            for (int r = 0; r < 32; ++r)
              *reinterpret_cast<__nv_bfloat16*>(mbuf + sw64(r, lane >> 3) + (lane & 7) * 2) =
                  __float2bfloat16_rn(x[r]);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) tma_store_2d(&mp->d, gm0, gn0, mbuf_s);
            g_m = ++groups;
          }
        } else {
          // diagonal chunks (direct stores) and FP32 / split-3 outputs: the
          // general writer, which first waits for every earlier store to
          // have read its box
          store_chunk(p, mp, x, gm0, gn0, lane, diag, dbuf, dbuf_s);
          if (!diag) groups += p.d_es == 6 ? 3 : (gn0 + 16 < p.N ? 2 : 1);
          g_d[0] = g_d[1] = g_m = groups;
        }
        __syncwarp();
      }
      if (!ok) break;
      if (p.ssq != nullptr)
        warp_sumsq_store(p.ssq + (int64_t(t.tm) * ((p.N + BN - 1) / BN) + t.tn) * kSsqSlots +
                             static_cast<int>(rank) * 8 + ew,
                         ssq, lane);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1u;
      if (t.done >= 0) {
        // Later tasks read this tile: once every epilogue warp's stores are
        // complete in memory, raise the counter with release semantics (one
        // arrival per CTA).
        if (lane == 0) tma_store_wait_all();
        __syncwarp();
        asm volatile("bar.sync %0, %1;" ::"n"(kEpiBarrier), "n"(32 * EPI_WARPS) : "memory");
        if (ew == 0 && lane == 0) {
          asm volatile("fence.proxy.async.global;" ::: "memory");
          asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(counters + t.done) : "memory");
        }
      }
    }
    if (!finished) {
      // A warp that gives up owes at most the one epilogue barrier the others
      // may be waiting in (none can pass it without this warp); arriving
      // there lets them reach the loop top and see the abort.
      __syncwarp();
      asm volatile("bar.arrive %0, %1;" ::"n"(kEpiBarrier), "n"(32 * EPI_WARPS) : "memory");
    }
    if (lane == 0) tma_store_wait_all();
    __syncwarp();
  }

  if (*abort_flag) {
    // an aborted pair may leave loads in flight that target this CTA's (or
    // the peer's) barriers: let them land before either CTA exits
    const unsigned long long t0 = globaltimer();
    while (globaltimer() - t0 < 20000000ull) __nanosleep(100000);
  }
  __syncwarp();      // the aligned cluster barrier wants converged warps
  tc_fence_before();
  cluster_sync();   // no MMA, load or arrive of the pair is outstanding
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

int g_sms2 = 0;

}  // namespace

bool tc2_encode_maps(const GemmProblem& p, TcMaps* out) {
  std::memset(out, 0, sizeof(TcMaps));
  bool ok = encode_2d(&out->a, p.A, 2, p.K, p.M, p.lda, BK, BMC, CU_TENSOR_MAP_SWIZZLE_128B);
  if (p.b_kmajor)
    ok = ok && encode_2d(&out->b, p.B, 2, p.K, p.N, p.ldb, BK, BN / 2, CU_TENSOR_MAP_SWIZZLE_128B);
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

int tc2_pairs() {
  if (g_sms2 == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms2, cudaDevAttrMultiProcessorCount, dev);
  }
  return g_sms2 / 2 > 0 ? g_sms2 / 2 : 1;
}

int launch_gemm_tc2(const GemmProblem* probs, const TcMaps* maps, const PairTask* tasks,
                    int ntasks, int* counters, int ncounters, const StepState* state,
                    int* err_flag, cudaStream_t s) {
  if (ntasks <= 0) return 0;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(k_gemm_tc2, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
      return -1;
    attr_set = true;
  }
  // task counter and dependency counters start from zero on every launch
  if (cudaMemsetAsync(counters, 0, sizeof(int) * ncounters, s) != cudaSuccess) return -1;
  const int pairs = ntasks < tc2_pairs() ? ntasks : tc2_pairs();
  k_gemm_tc2<<<2 * pairs, NTHREADS, SMEM_BYTES, s>>>(probs, maps, tasks, ntasks, counters, state,
                                                     err_flag);
  return 0;
}

}  // namespace muon
