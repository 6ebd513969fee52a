// PTX wrappers shared by the tensor-core GEMM kernels (tcgen05, TMA,
// mbarrier) and the host-side TMA descriptor encoder.  Included by the
// kernel translation units only.
#pragma once

#include <cuda_bf16.h>

#include "muon_internal.h"

namespace muon {
namespace tc {

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

// ---- thread-block clusters and CTA pairs (tcgen05 cta_group::2)

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared::cluster address of the same shared-memory location in CTA
// `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Every thread of every CTA of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Arrive on an mbarrier given by its shared::cluster address (possibly in
// another CTA of the cluster).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

// Bounded wait with cluster-scope acquire: for barriers that other CTAs of
// the cluster arrive on to hand over data they wrote.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag, int* err_flag, int code) {
  auto try_once = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
  };
  if (try_once()) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (try_once()) return true;
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
// Waits until at most n of this thread's bulk async-groups still read
// their shared-memory sources (n clamped to 7; waiting for fewer pending
// groups is only stricter).
__device__ __forceinline__ void bulk_wait_read_n(int n) {
  switch (n < 0 ? 0 : (n > 7 ? 7 : n)) {
    case 0: asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.bulk.wait_group.read 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.bulk.wait_group.read 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.bulk.wait_group.read 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.bulk.wait_group.read 6;" ::: "memory"); break;
    default: asm volatile("cp.async.bulk.wait_group.read 7;" ::: "memory"); break;
  }
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
// swizzle mode in bits 61-63 (2 = 128-byte, 4 = 64-byte).
constexpr uint32_t kSwizzle128 = 2, kSwizzle64 = 4;
__device__ __forceinline__ uint64_t make_desc(uint32_t saddr, uint32_t lbo_bytes,
                                              uint32_t sbo_bytes, uint32_t swizzle) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(swizzle) << 61;
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, A K-major,
// B K-major or MN-major, the given M and N.
__host__ __device__ constexpr uint32_t make_idesc(bool b_mn_major, int M, int N) {
  return (1u << 4)                 // D format: f32
         | (1u << 7)               // A format: bf16
         | (1u << 10)              // B format: bf16
         | (0u << 15)              // A K-major
         | ((b_mn_major ? 1u : 0u) << 16)
         | (static_cast<uint32_t>(N >> 3) << 17)
         | (static_cast<uint32_t>(M >> 4) << 24);
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

// Pair MMA: issued by one thread of the even CTA, A rows and B columns
// split across the two CTAs' shared memory, D in both CTAs' tensor memory.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives, when the pair's earlier MMAs finish, on the mbarrier at this
// shared-memory offset in every CTA of `mask`.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar), "h"(mask)
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

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, int x, int y, int z,
                                             uint32_t src) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z), "r"(src)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Exact three-way split of a float into bfloat16 parts, v = hi + mid + lo:
// hi = bf16(v), mid = bf16(v - hi), lo = v - hi - mid (fits bfloat16).
__device__ __forceinline__ void split3(float v, __nv_bfloat16& hi, __nv_bfloat16& mid,
                                       __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(v);
  const float r1 = __fsub_rn(v, __bfloat162float(hi));
  mid = __float2bfloat16_rn(r1);
  lo = __float2bfloat16_rn(__fsub_rn(r1, __bfloat162float(mid)));
}

// Epilogue output: one 32 x 32 chunk per warp, staged through a 2 KB buffer
// of 64-byte rows (64-byte swizzle) and written by TMA stores.
// Writes one output element: fp32, bf16 or three split-3 planes `ps` apart.
__device__ __forceinline__ void put_plane(void* D, int64_t idx, int64_t ps, int d_es, float v) {
  if (d_es == 4) {
    reinterpret_cast<float*>(D)[idx] = v;
  } else if (d_es == 2) {
    reinterpret_cast<__nv_bfloat16*>(D)[idx] = __float2bfloat16_rn(v);
  } else {
    __nv_bfloat16 h, m, l;
    split3(v, h, m, l);
    __nv_bfloat16* d = reinterpret_cast<__nv_bfloat16*>(D);
    d[idx] = h;
    d[idx + ps] = m;
    d[idx + 2 * ps] = l;
  }
}

// Writes one 32 x 32 chunk (lane = row).  Off the diagonal each plane (or
// the bf16 / two fp32 boxes) goes through the swizzled staging buffer and a
// TMA store; diagonal chunks of symmetric products are written directly
// (upper triangle by rows, strictly upper again as the mirror); chunks above
// the diagonal are also mirrored with direct, coalesced stores.
// Stages one 64-byte-row box (lane = row) and issues its TMA store.
template <class Fill>
__device__ __forceinline__ void stage_and_store(uint8_t* dbuf, int lane, Fill fill) {
  if (lane == 0) tma_store_wait_read();   // the previous store has read dbuf
  __syncwarp();
  #pragma unroll
  for (int g = 0; g < 4; ++g) *reinterpret_cast<uint4*>(dbuf + sw64(lane, g)) = fill(g);
  fence_async_smem();
  __syncwarp();
}

// mbuf (bf16 outputs, optional): a second 2 KB box buffer; chunks above the
// diagonal of a symmetric product are then mirrored by staging the
// transposed chunk there and storing it with TMA as well.
__device__ __forceinline__ void store_chunk(const GemmProblem& p, const TcMaps* mp, const float* x,
                                            int gm0, int gn0, int lane, bool diag, uint8_t* dbuf,
                                            uint32_t dbuf_s, uint8_t* mbuf = nullptr,
                                            uint32_t mbuf_s = 0) {
  // fields read once: later stores to D would force reloads through p
  const int M = p.M, N = p.N, des = p.d_es;
  const bool sym = p.symmetric != 0;
  const int64_t ldd = p.ldd, dps = p.d_ps;
  void* D = p.D;
  const int gm = gm0 + lane;
  if (diag) {
    if (gm >= M) return;
    #pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int gn = gn0 + j;
      if (gn >= N || j < lane) continue;
      put_plane(D, int64_t(gm) * ldd + gn, dps, des, x[j]);
      if (j > lane) put_plane(D, int64_t(gn) * ldd + gm, dps, des, x[j]);
    }
    return;
  }
  if (des == 2) {
    stage_and_store(dbuf, lane, [&](int g) {
      __nv_bfloat162 h[4];
      #pragma unroll
      for (int u = 0; u < 4; ++u) h[u] = __floats2bfloat162_rn(x[8 * g + 2 * u], x[8 * g + 2 * u + 1]);
      return *reinterpret_cast<const uint4*>(h);
    });
    if (lane == 0) tma_store_2d(&mp->d, gn0, gm0, dbuf_s);
  } else if (des == 4) {
    #pragma unroll
    for (int b = 0; b < 2; ++b) {
      if (b == 1 && gn0 + 16 >= N) break;   // warp-uniform
      stage_and_store(dbuf, lane, [&](int g) {
        const float* xs = x + 16 * b + 4 * g;
        return make_uint4(__float_as_uint(xs[0]), __float_as_uint(xs[1]), __float_as_uint(xs[2]),
                          __float_as_uint(xs[3]));
      });
      if (lane == 0) tma_store_2d(&mp->d, gn0 + 16 * b, gm0, dbuf_s);
    }
  } else {
    #pragma unroll
    for (int b = 0; b < 3; ++b) {
      stage_and_store(dbuf, lane, [&](int g) {
        __nv_bfloat16 h[8];
        #pragma unroll
        for (int u = 0; u < 8; ++u) {
          __nv_bfloat16 hi, mid, lo;
          split3(x[8 * g + u], hi, mid, lo);
          h[u] = b == 0 ? hi : (b == 1 ? mid : lo);
        }
        return *reinterpret_cast<const uint4*>(h);
      });
      if (lane == 0) tma_store_3d(&mp->d, gn0, gm0, b, dbuf_s);
    }
  }
  if (sym && des == 2 && mbuf != nullptr) {
    // The store above waited for every earlier store to read its buffer, so
    // mbuf is free.  Box row r = output row gn0 + r, box column = lane
    // (output column gm0 + lane); TMA clips what falls outside the matrix.
    #pragma unroll
    for (int r = 0; r < 32; ++r)
      *reinterpret_cast<__nv_bfloat16*>(mbuf + sw64(r, lane >> 3) + (lane & 7) * 2) =
          __float2bfloat16_rn(x[r]);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) tma_store_2d(&mp->d, gm0, gn0, mbuf_s);
    return;
  }
  if (sym && gm < M) {
    if (des == 2) {
      __nv_bfloat16* Db = reinterpret_cast<__nv_bfloat16*>(D);
      #pragma unroll
      for (int j = 0; j < 32; ++j)
        if (gn0 + j < N) Db[int64_t(gn0 + j) * ldd + gm] = __float2bfloat16_rn(x[j]);
    } else {
      #pragma unroll
      for (int j = 0; j < 32; ++j)
        if (gn0 + j < N) put_plane(D, int64_t(gn0 + j) * ldd + gm, dps, des, x[j]);
    }
  }
}

// Sum of squares of one chunk's values as stored (bf16-rounded for bf16
// outputs; FP32 and split-3 outputs hold the value exactly), accumulated in
// FP32 in column order.
__device__ __forceinline__ float chunk_sumsq(const float* x, int d_es, float acc) {
  #pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float v = d_es == 2 ? __bfloat162float(__float2bfloat16_rn(x[j])) : x[j];
    acc = __fmaf_rn(v, v, acc);
  }
  return acc;
}

// A warp's per-lane sums, added in a fixed shuffle order in double; lane 0
// writes the total.
__device__ __forceinline__ void warp_sumsq_store(double* dst, float acc, int lane) {
  double d = acc;
  #pragma unroll
  for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
  if (lane == 0) *dst = d;
}

// ------------------------------------------------------------------ host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
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
// Map over a row-major matrix: `inner` elements per row, `outer` rows, row
// stride `ld` elements; `planes` > 1 adds a third dimension of `planes`
// matrices `pstride` elements apart (the split-3 planes).
inline bool encode_2d(CUtensorMap* m, const void* base, int es, int64_t inner, int64_t outer,
                      int64_t ld, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw,
                      int planes = 1, int64_t pstride = 0) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer),
                        static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * es), static_cast<cuuint64_t>(pstride * es)};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, es == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
            planes > 1 ? 3 : 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


}  // namespace tc
}  // namespace muon
