// Streaming (HBM-bound) kernels of the Muon step:
//   S1  accumulate              accum += scale * bf16 grad
//   S2  reduce (pass 1)         overflow check + per-tile sums of squares of
//                               m' = beta*m + g (Muon) or g (auxiliary)
//       owner_norm              per-block divisor ||m'||_F + 1e-7
//       gather (pass 2)         momentum <- m', X0 = m' / divisor in the
//                               canonical (rows <= cols) orientation
//   S4  update_sumsq            per-tile sums of squares of the NS result
//       finalize                global norm, clip coefficient, result struct
//       scatter                 owned-slice write-back of coef*u (Muon) and
//                               coef*g (auxiliary), master -= lr*coef*u
// Step order and semantics follow "Run Muon once per optimizer step under
// ZeRO-3, not once per micro-batch" ("The change": overflow check, then
// Muon, then the gradient norm over the Muon updates, then clipping) and
// "Support Muon in BF16_Optimizer with FP32 gradient accumulation" (PR
// description: FP32 accumulation, full-matrix Muon, owned intersections,
// padding excluded).
//
// Every reduction has a fixed shape that depends only on an owner's element
// index, never on where partition boundaries fall, so results are bitwise
// independent of the partition table.
#include <cuda_bf16.h>

#include "tc_common.cuh"

namespace muon {

namespace {

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Workspace elements: esize 2 = bf16, 4 = fp32, 6 = split-3 (three bf16
// planes `ps` elements apart whose sum is the fp32 value exactly).
__device__ __forceinline__ int ebytes(int esize) { return esize == 6 ? 2 : esize; }

__device__ __forceinline__ float load_ws(const void* base, int esize, int64_t i, int64_t ps = 0) {
  if (esize == 2) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[i]);
  if (esize == 6) {
    const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(base);
    return __fadd_rn(__fadd_rn(__bfloat162float(b[i]), __bfloat162float(b[i + ps])),
                     __bfloat162float(b[i + 2 * ps]));
  }
  return reinterpret_cast<const float*>(base)[i];
}

__device__ __forceinline__ void store_ws(void* base, int esize, int64_t i, float v, int64_t ps = 0) {
  if (esize == 2) {
    reinterpret_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
  } else if (esize == 6) {
    __nv_bfloat16* b = reinterpret_cast<__nv_bfloat16*>(base);
    tc::split3(v, b[i], b[i + ps], b[i + 2 * ps]);
  } else {
    reinterpret_cast<float*>(base)[i] = v;
  }
}

// Last segment whose rel_begin <= rel.
__device__ __forceinline__ int find_seg(const Segment* s, int n, int64_t rel) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (s[mid].rel_begin <= rel) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Fixed-shape block reduction of one double per thread; result valid in
// thread 0.
template <int NT>
__device__ __forceinline__ double block_sum(double v) {
  __shared__ double red[NT / 32];
  #pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  double r = 0.0;
  if (w == 0) {
    r = (l < NT / 32) ? red[l] : 0.0;
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  }
  __syncthreads();
  return r;
}

__device__ __forceinline__ float momentum_of(float beta, float m, float g) {
  return __fadd_rn(__fmul_rn(beta, m), g);
}

// The gradient the step uses: accum * grad_scale (a loss scale undone).
__device__ __forceinline__ float grad_in(const StreamLaunchArgs& a, float g) {
  return a.grad_scale == 1.f ? g : __fmul_rn(a.grad_scale, g);
}

// The gradient fed to the momentum: grad_in, times the clip coefficient
// when gradients are clipped before Muon (cpre = 1 otherwise).
__device__ __forceinline__ float grad_m(const StreamLaunchArgs& a, float cpre, float g) {
  const float gs = grad_in(a, g);
  return a.clip_mode == 1 ? __fmul_rn(cpre, gs) : gs;
}

// Adam on one auxiliary element (clipped gradient g), in the oracle's
// operation order: m, v and w in, updated m, v and w out.
__device__ __forceinline__ void adam_el(const StreamLaunchArgs& a, float g, float& m, float& v, float& w) {
  m = __fadd_rn(__fmul_rn(a.adam_b1, m), __fmul_rn(a.adam_omb1, g));
  v = __fadd_rn(__fmul_rn(a.adam_b2, v), __fmul_rn(__fmul_rn(a.adam_omb2, g), g));
  const float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), a.adam_sqrt_bc2), a.adam_eps);
  w = __fadd_rn(w, __fmul_rn(a.adam_neg_step, __fdiv_rn(m, denom)));
}

__device__ __forceinline__ void adam_one(const StreamLaunchArgs& a, int64_t st, float g) {
  float m = a.exp_avg[st], v = a.exp_avg_sq[st], w = a.master[st];
  adam_el(a, g, m, v, w);
  a.exp_avg[st] = m;
  a.exp_avg_sq[st] = v;
  a.master[st] = w;
}

// Adam on four consecutive auxiliary elements starting at a 16-byte aligned
// storage index.
__device__ __forceinline__ void adam_four(const StreamLaunchArgs& a, int64_t st, float4 g) {
  float4 m = *reinterpret_cast<const float4*>(a.exp_avg + st);
  float4 v = *reinterpret_cast<const float4*>(a.exp_avg_sq + st);
  float4 w = *reinterpret_cast<const float4*>(a.master + st);
  adam_el(a, g.x, m.x, v.x, w.x);
  adam_el(a, g.y, m.y, v.y, w.y);
  adam_el(a, g.z, m.z, v.z, w.z);
  adam_el(a, g.w, m.w, v.w, w.w);
  *reinterpret_cast<float4*>(a.exp_avg + st) = m;
  *reinterpret_cast<float4*>(a.exp_avg_sq + st) = v;
  *reinterpret_cast<float4*>(a.master + st) = w;
}

// ------------------------------------------------------------------ S1

__device__ __forceinline__ float acc_one(float a, float g, float scale, int overwrite) {
  const float sg = __fmul_rn(scale, g);
  return overwrite ? sg : __fadd_rn(a, sg);
}

__device__ __forceinline__ float4 acc_four(float4 a, uint2 b, float scale, int overwrite) {
  return make_float4(acc_one(a.x, __uint_as_float(b.x << 16), scale, overwrite),
                     acc_one(a.y, __uint_as_float(b.x & 0xffff0000u), scale, overwrite),
                     acc_one(a.z, __uint_as_float(b.y << 16), scale, overwrite),
                     acc_one(a.w, __uint_as_float(b.y & 0xffff0000u), scale, overwrite));
}

// Where the step's gradient comes from, fixed per launch (the launchers pick
// the instantiation, so the loads of the 16-byte paths carry no branch):
// kind 0 reads accum; kind 1 folds last_grad in; kind 2 folds prev_grad and
// then last_grad in.  old: accum's old value is read (false when a folded
// micro-batch overwrites it).
//
// When a folded micro-batch overwrites accum's old value, forming the
// gradient reads as many bytes as reading accum would, so the first pass does
// not write it: every pass that reads the gradient forms it again with
// muon_accumulate's arithmetic (all of them see the same bits), and accum is
// written once, by the write-back (or by k_fold_commit when the step is
// skipped).  Otherwise (old) the first pass writes the formed gradient into
// accum and the later passes read accum (the host launches them with kind 0):
// forming it again there would add bytes and read streams to the gather,
// which measured slower.  (Writing it in the first pass for the transposed
// blocks alone measured slower on the Llama-3-8B step too: 2 ms less in the
// gather, 3 ms more in the first pass.)
template <int K, bool OLD>
struct Fold {
  static constexpr int kind = K;
  static constexpr bool old = OLD;
};

template <class F>
__device__ __forceinline__ float grad_at(const StreamLaunchArgs& a, int64_t st) {
  float g = F::old ? a.accum[st] : 0.f;
  if (F::kind == 2) g = acc_one(g, bf16_bits_to_float(a.prev_grad[st]), a.prev_scale, a.prev_overwrite);
  if (F::kind >= 1) g = acc_one(g, bf16_bits_to_float(a.last_grad[st]), a.last_scale, a.last_overwrite);
  return g;
}

// grad_at of the four elements st .. st+3 (st a multiple of 4): one 16-byte
// accum load and one 8-byte load per folded micro-batch
template <class F>
__device__ __forceinline__ float4 grad_at4(const StreamLaunchArgs& a, int64_t st) {
  float4 g = F::old ? *reinterpret_cast<const float4*>(a.accum + st) : make_float4(0.f, 0.f, 0.f, 0.f);
  if (F::kind == 2)
    g = acc_four(g, *reinterpret_cast<const uint2*>(a.prev_grad + st), a.prev_scale, a.prev_overwrite);
  if (F::kind >= 1)
    g = acc_four(g, *reinterpret_cast<const uint2*>(a.last_grad + st), a.last_scale, a.last_overwrite);
  return g;
}

// grad_at of the eight elements st .. st+7 (st a multiple of 8, the folded
// micro-batches 16-byte aligned): 16-byte loads of each bf16 micro-batch
template <class F>
__device__ __forceinline__ void grad_at8(const StreamLaunchArgs& a, int64_t st, float4& lo, float4& hi) {
  lo = F::old ? *reinterpret_cast<const float4*>(a.accum + st) : make_float4(0.f, 0.f, 0.f, 0.f);
  hi = F::old ? *reinterpret_cast<const float4*>(a.accum + st + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
  if (F::kind == 2) {
    const uint4 p = *reinterpret_cast<const uint4*>(a.prev_grad + st);
    lo = acc_four(lo, make_uint2(p.x, p.y), a.prev_scale, a.prev_overwrite);
    hi = acc_four(hi, make_uint2(p.z, p.w), a.prev_scale, a.prev_overwrite);
  }
  if (F::kind >= 1) {
    const uint4 l = *reinterpret_cast<const uint4*>(a.last_grad + st);
    lo = acc_four(lo, make_uint2(l.x, l.y), a.last_scale, a.last_overwrite);
    hi = acc_four(hi, make_uint2(l.z, l.w), a.last_scale, a.last_overwrite);
  }
}

// ------------------------------------------------------------------ debug bounds checks
// Debug builds (MUON_DEBUG) check, before a block touches memory, that its
// tile stays inside the extents the tables describe: the storage range of
// its elements (its own range on the 16-byte path, every segment of its
// owner otherwise) and its owner's X region.  A tile that would leave them
// records kErrBounds (read by muon_device_error) and touches nothing.  The
// check is per block, so every thread of the block takes the same branch.
#ifdef MUON_DEBUG
__device__ __forceinline__ bool dbg_in(int64_t lo, int64_t hi, int64_t extent) {
  return lo >= 0 && lo <= hi && hi <= extent;
}
__device__ bool dbg_tile_ok(const StreamLaunchArgs& a, const Owner& o, bool fast, int64_t sdelta,
                            int64_t rel_lo, int64_t rel_hi, bool uses_x) {
  if (fast) {
    if (!dbg_in(sdelta + rel_lo, sdelta + rel_hi, a.dbg_storage_extent)) return false;
  } else {
    for (int k = 0; k < o.seg_count; ++k) {
      const Segment sg = a.segs[o.seg_begin + k];
      if (!dbg_in(sg.storage_begin, sg.storage_begin + sg.len, a.dbg_storage_extent)) return false;
    }
  }
  if (uses_x && !dbg_in(o.x_off, o.x_off + int64_t(o.m) * o.ldx, a.dbg_x_extent)) return false;
  return true;
}
// The owner-relative element range of a gather / scatter tile.
__device__ __forceinline__ void dbg_etile_range(const ETile& t, const Owner& o, int64_t& lo,
                                                int64_t& hi) {
  if (t.kind == 0) {
    lo = int64_t(t.r0) * o.cols;
    hi = int64_t(t.r0 + t.nr) * o.cols;
  } else if (t.kind == 1 || t.kind == 3) {
    const int re = min(t.r0 + kTT, o.rows), ce = min(t.c0 + (t.kind == 3 ? 2 * kTT : kTT), o.cols);
    lo = int64_t(t.r0) * o.cols + t.c0;
    hi = int64_t(re - 1) * o.cols + ce;
  } else {
    lo = t.rel_begin;
    hi = t.rel_begin + t.len;
  }
}
#define MUON_DBG_CHECK(ok_expr, flag)                        \
  do {                                                       \
    if (!(ok_expr)) {                                        \
      if (threadIdx.x == 0 && (flag)) atomicExch((flag), kErrBounds); \
      return;                                                \
    }                                                        \
  } while (0)
#else
#define MUON_DBG_CHECK(ok_expr, flag) \
  do {                                \
  } while (0)
#endif

__global__ void __launch_bounds__(kStreamThreads)
k_accumulate(float* __restrict__ accum, const uint16_t* __restrict__ grad,
             const Run* __restrict__ runs, float scale, int overwrite, int64_t dbg_extent,
             int* dbg_flag) {
  const Run r = runs[blockIdx.x];
  MUON_DBG_CHECK(dbg_in(r.begin, r.begin + r.len, dbg_extent), dbg_flag);
  const int64_t b = r.begin, e = r.begin + r.len;
  int64_t vb = (b + 3) & ~int64_t(3);
  if (vb > e) vb = e;
  const int64_t ve = vb + ((e - vb) & ~int64_t(3));
  for (int64_t i = b + threadIdx.x; i < vb; i += blockDim.x)
    accum[i] = acc_one(accum[i], bf16_bits_to_float(grad[i]), scale, overwrite);
  constexpr int U = 4;
  const int64_t step = int64_t(4) * blockDim.x;
  int64_t i = vb + int64_t(4) * threadIdx.x;
  for (; i + (U - 1) * step < ve; i += U * step) {
    float4 a[U];
    uint2 g[U];
    #pragma unroll
    for (int u = 0; u < U; ++u) {
      g[u] = *reinterpret_cast<const uint2*>(grad + i + u * step);
      if (!overwrite) a[u] = *reinterpret_cast<const float4*>(accum + i + u * step);
      else a[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    #pragma unroll
    for (int u = 0; u < U; ++u) {
      float4 o;
      o.x = acc_one(a[u].x, __uint_as_float(g[u].x << 16), scale, overwrite);
      o.y = acc_one(a[u].y, __uint_as_float(g[u].x & 0xffff0000u), scale, overwrite);
      o.z = acc_one(a[u].z, __uint_as_float(g[u].y << 16), scale, overwrite);
      o.w = acc_one(a[u].w, __uint_as_float(g[u].y & 0xffff0000u), scale, overwrite);
      *reinterpret_cast<float4*>(accum + i + u * step) = o;
    }
  }
  for (; i < ve; i += step) {
    const float4 a = overwrite ? make_float4(0.f, 0.f, 0.f, 0.f)
                               : *reinterpret_cast<const float4*>(accum + i);
    const uint2 g = *reinterpret_cast<const uint2*>(grad + i);
    float4 o;
    o.x = acc_one(a.x, __uint_as_float(g.x << 16), scale, overwrite);
    o.y = acc_one(a.y, __uint_as_float(g.x & 0xffff0000u), scale, overwrite);
    o.z = acc_one(a.z, __uint_as_float(g.y << 16), scale, overwrite);
    o.w = acc_one(a.w, __uint_as_float(g.y & 0xffff0000u), scale, overwrite);
    *reinterpret_cast<float4*>(accum + i) = o;
  }
  for (int64_t j = ve + threadIdx.x; j < e; j += blockDim.x)
    accum[j] = acc_one(accum[j], bf16_bits_to_float(grad[j]), scale, overwrite);
}

// C micro-batches in one pass: element by element the arithmetic of C
// k_accumulate launches in order (the first with `overwrite`), accum read at
// most once and written once.  Same runs and vector layout as k_accumulate.
template <int C>
__device__ __forceinline__ float acc_set(const GradSet& gs, float a, int64_t i, int overwrite) {
  #pragma unroll
  for (int j = 0; j < C; ++j)
    a = acc_one(a, bf16_bits_to_float(gs.grad[j][i]), gs.scale[j], j == 0 ? overwrite : 0);
  return a;
}

template <int C>
__global__ void __launch_bounds__(kStreamThreads)
k_accumulate_n(float* __restrict__ accum, const GradSet gs, const Run* __restrict__ runs,
               int overwrite, int64_t dbg_extent, int* dbg_flag) {
  const Run r = runs[blockIdx.x];
  MUON_DBG_CHECK(dbg_in(r.begin, r.begin + r.len, dbg_extent), dbg_flag);
  const int64_t b = r.begin, e = r.begin + r.len;
  int64_t vb = (b + 3) & ~int64_t(3);
  if (vb > e) vb = e;
  const int64_t ve = vb + ((e - vb) & ~int64_t(3));
  for (int64_t i = b + threadIdx.x; i < vb; i += blockDim.x)
    accum[i] = acc_set<C>(gs, overwrite ? 0.f : accum[i], i, overwrite);
  constexpr int U = C <= 2 ? 4 : 2;
  const int64_t step = int64_t(4) * blockDim.x;
  int64_t i = vb + int64_t(4) * threadIdx.x;
  for (; i + (U - 1) * step < ve; i += U * step) {
    float4 a[U];
    uint2 g[U][C];
    #pragma unroll
    for (int u = 0; u < U; ++u) {
      #pragma unroll
      for (int j = 0; j < C; ++j) g[u][j] = *reinterpret_cast<const uint2*>(gs.grad[j] + i + u * step);
      a[u] = overwrite ? make_float4(0.f, 0.f, 0.f, 0.f)
                       : *reinterpret_cast<const float4*>(accum + i + u * step);
    }
    #pragma unroll
    for (int u = 0; u < U; ++u) {
      float4 o = a[u];
      #pragma unroll
      for (int j = 0; j < C; ++j) o = acc_four(o, g[u][j], gs.scale[j], j == 0 ? overwrite : 0);
      *reinterpret_cast<float4*>(accum + i + u * step) = o;
    }
  }
  for (; i < ve; i += step) {
    float4 o = overwrite ? make_float4(0.f, 0.f, 0.f, 0.f) : *reinterpret_cast<const float4*>(accum + i);
    #pragma unroll
    for (int j = 0; j < C; ++j)
      o = acc_four(o, *reinterpret_cast<const uint2*>(gs.grad[j] + i), gs.scale[j], j == 0 ? overwrite : 0);
    *reinterpret_cast<float4*>(accum + i) = o;
  }
  for (int64_t j = ve + threadIdx.x; j < e; j += blockDim.x)
    accum[j] = acc_set<C>(gs, overwrite ? 0.f : accum[j], j, overwrite);
}

// ------------------------------------------------------------------ S2 pass 1

// One element of pass 1: the sum of squares of what the mode needs and the
// overflow check on the gradient the step uses.
__device__ __forceinline__ void reduce_one(const StreamLaunchArgs& a, float graw, float m, bool use_m,
                                           float c, float& acc, bool& bad) {
  const float gs = grad_in(a, graw);
  bad |= !isfinite(gs);
  const float ge = c == 1.f ? gs : __fmul_rn(c, gs);
  const float v = use_m ? momentum_of(a.beta, m, ge) : ge;
  acc = __fmaf_rn(v, v, acc);
}

// One pass-1 tile, the gradient read through F (and written into accum when
// F reads accum's old value).
template <class F>
__device__ __forceinline__ void reduce_tile(const StreamLaunchArgs& a, const RTile& t, const Owner& o,
                                            bool use_m, float c, float& acc, bool& bad) {
  constexpr int NT = kStreamThreads;
  const int64_t tb = t.rel_begin, te = t.rel_begin + t.len;
  const int ngroups = (t.len + 3) / 4;
  if (t.fast) {
    const int64_t base = t.sdelta + tb;
    const float* M = a.momentum + base;
    constexpr int U = 4;   // 8 or 16 groups in flight per thread measured 1.8x / 3.4x slower
    for (int g0 = threadIdx.x; g0 < ngroups; g0 += NT * U) {
      float4 gv[U], mv[U];
      #pragma unroll
      for (int u = 0; u < U; ++u) {
        const int g = g0 + u * NT;
        if (g < ngroups) {
          gv[u] = grad_at4<F>(a, base + 4 * g);
          if (F::kind > 0 && F::old) *reinterpret_cast<float4*>(a.accum + base + 4 * g) = gv[u];
          mv[u] = use_m ? *reinterpret_cast<const float4*>(M + 4 * g) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      #pragma unroll
      for (int u = 0; u < U; ++u) {
        if (g0 + u * NT < ngroups) {
          reduce_one(a, gv[u].x, mv[u].x, use_m, c, acc, bad);
          reduce_one(a, gv[u].y, mv[u].y, use_m, c, acc, bad);
          reduce_one(a, gv[u].z, mv[u].z, use_m, c, acc, bad);
          reduce_one(a, gv[u].w, mv[u].w, use_m, c, acc, bad);
        }
      }
    }
  } else {
    const Segment* segs = a.segs + o.seg_begin;
    int si = -1;
    for (int g = threadIdx.x; g < ngroups; g += NT) {
      for (int j = 0; j < 4; ++j) {
        const int64_t rel = tb + 4 * int64_t(g) + j;
        if (rel >= te) break;
        if (si < 0) si = find_seg(segs, o.seg_count, rel);
        while (rel >= segs[si].rel_begin + segs[si].len) ++si;
        const int64_t st = segs[si].storage_begin + (rel - segs[si].rel_begin);
        const float gr = grad_at<F>(a, st);
        if (F::kind > 0 && F::old) a.accum[st] = gr;
        reduce_one(a, gr, use_m ? a.momentum[st] : 0.f, use_m, c, acc, bad);
      }
    }
  }
}

// Thread t of the tile sums the 4-element groups t, t + NT, t + 2 NT, ...
// (elements in order within a group), whatever segments they fall in: the
// sum order depends only on the owner-relative index.  Tiles inside one
// aligned segment read float4s; others resolve each element's segment.
// reduce_mode 0: Muon tiles sum (beta m + g)^2, auxiliary tiles g^2;
//             1: every tile sums g^2 (the gradient norm, clip-before-Muon);
//             2: Muon tiles sum (beta m + coef g)^2 after the gradient clip.
template <class F>
__global__ void __launch_bounds__(kStreamThreads)
k_reduce(StreamLaunchArgs a) {
  constexpr int NT = kStreamThreads;
  const RTile t = a.rtiles[blockIdx.x];
  const Owner o = a.owners[t.owner];
  if (a.reduce_mode == 2 && (!o.is_muon || a.state->overflow)) return;
  MUON_DBG_CHECK(dbg_tile_ok(a, o, t.fast, t.sdelta, t.rel_begin, t.rel_begin + t.len, false),
                 a.dbg_flag);
  const bool use_m = a.reduce_mode == 1 ? false : (o.is_muon != 0);
  const float c = a.reduce_mode == 2 ? a.state->coef : 1.f;
  float acc = 0.f;
  bool bad = false;
  reduce_tile<F>(a, t, o, use_m, c, acc, bad);
  if (__syncthreads_or(bad) && threadIdx.x == 0 && a.reduce_mode != 2) atomicOr(&a.state->overflow, 1);
  const double s = block_sum<NT>(static_cast<double>(acc));
  if (threadIdx.x == 0) a.rtile_sum[blockIdx.x] = s;
}

// A skipped step with folded micro-batches: accum takes the gradient the
// step formed (grad_at), the state muon_accumulate on those micro-batches
// would have left; padding stays untouched.  The tiles of k_reduce, strided
// over a grid of a few CTAs per SM, so an applied step costs one flag read
// per CTA.
template <class F>
__global__ void __launch_bounds__(kStreamThreads)
k_fold_commit(StreamLaunchArgs a) {
  if (!a.state->overflow) return;
  for (int k = blockIdx.x; k < a.n_rtiles; k += gridDim.x) {
    const RTile t = a.rtiles[k];
    const Owner o = a.owners[t.owner];
    MUON_DBG_CHECK(dbg_tile_ok(a, o, t.fast, t.sdelta, t.rel_begin, t.rel_begin + t.len, false),
                   a.dbg_flag);
    const int64_t tb = t.rel_begin, te = t.rel_begin + t.len;
    if (t.fast) {
      const int64_t base = t.sdelta + tb;
      for (int g = threadIdx.x; g < t.len / 4; g += kStreamThreads)
        *reinterpret_cast<float4*>(a.accum + base + 4 * g) = grad_at4<F>(a, base + 4 * g);
      continue;
    }
    const Segment* segs = a.segs + o.seg_begin;
    for (int si = find_seg(segs, o.seg_count, tb); si < o.seg_count && segs[si].rel_begin < te; ++si) {
      const Segment sg = segs[si];
      const int64_t lo = sg.rel_begin > tb ? sg.rel_begin : tb;
      const int64_t hi = (sg.rel_begin + sg.len) < te ? (sg.rel_begin + sg.len) : te;
      const int64_t base = sg.storage_begin - sg.rel_begin;
      for (int64_t rel = lo + threadIdx.x; rel < hi; rel += kStreamThreads)
        a.accum[base + rel] = grad_at<F>(a, base + rel);
    }
  }
}

__global__ void k_owner_norm(StreamLaunchArgs a) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.n_owners) return;
  const Owner o = a.owners[i];
  if (!o.is_muon) return;
  double s = 0.0;
  for (int k = 0; k < o.rtile_count; ++k) s += a.rtile_sum[o.rtile_begin + k];
  a.owner_div[i] = static_cast<float>(sqrt(s) + kNormEps);
}

// ------------------------------------------------------------------ S2 pass 2

// Calls f(rel, storage_index) for the elements [lo, hi) of one owner row,
// lane-strided across a warp, resolving partition segments.
template <class F>
__device__ __forceinline__ void for_row(const Segment* segs, int nseg, int64_t lo, int64_t hi,
                                        int lane, F&& f) {
  int si = find_seg(segs, nseg, lo);
  for (; si < nseg && segs[si].rel_begin < hi; ++si) {
    const Segment sg = segs[si];
    const int64_t plo = sg.rel_begin > lo ? sg.rel_begin : lo;
    const int64_t phi = (sg.rel_begin + sg.len) < hi ? (sg.rel_begin + sg.len) : hi;
    const int64_t base = sg.storage_begin - sg.rel_begin;
    for (int64_t rel = plo + lane; rel < phi; rel += 32) f(rel, base + rel);
  }
}

// ---- 16-byte fast paths (tile in one segment, aligned; see ETile::fast).
// All loads of a batch are issued before any store, so a thread keeps
// several 16-byte requests in flight.

__device__ __forceinline__ uint2 pack4_bf16(float a, float b, float c, float d) {
  __nv_bfloat162 h[2] = {__floats2bfloat162_rn(a, b), __floats2bfloat162_rn(c, d)};
  return *reinterpret_cast<const uint2*>(h);
}

__device__ __forceinline__ float4 unpack4_bf16(uint2 w) {
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ void store4_ws(void* base, int esize, int64_t i, float4 v, int64_t ps = 0) {
  if (esize == 2) {
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(base) + i) = pack4_bf16(v.x, v.y, v.z, v.w);
  } else if (esize == 6) {
    __nv_bfloat16 h[4][3];
    const float f[4] = {v.x, v.y, v.z, v.w};
    #pragma unroll
    for (int k = 0; k < 4; ++k) tc::split3(f[k], h[k][0], h[k][1], h[k][2]);
    __nv_bfloat16* b = reinterpret_cast<__nv_bfloat16*>(base) + i;
    #pragma unroll
    for (int pl = 0; pl < 3; ++pl) {
      __nv_bfloat16 q[4] = {h[0][pl], h[1][pl], h[2][pl], h[3][pl]};
      *reinterpret_cast<uint2*>(b + pl * ps) = *reinterpret_cast<const uint2*>(q);
    }
  } else {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + i) = v;
  }
}

__device__ __forceinline__ float4 load4_ws(const void* base, int esize, int64_t i, int64_t ps = 0) {
  if (esize == 2)
    return unpack4_bf16(*reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(base) + i));
  if (esize == 6) {
    const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(base) + i;
    const float4 h = unpack4_bf16(*reinterpret_cast<const uint2*>(b));
    const float4 m = unpack4_bf16(*reinterpret_cast<const uint2*>(b + ps));
    const float4 l = unpack4_bf16(*reinterpret_cast<const uint2*>(b + 2 * ps));
    return make_float4(__fadd_rn(__fadd_rn(h.x, m.x), l.x), __fadd_rn(__fadd_rn(h.y, m.y), l.y),
                       __fadd_rn(__fadd_rn(h.z, m.z), l.z), __fadd_rn(__fadd_rn(h.w, m.w), l.w));
  }
  return *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + i);
}

// rows of a non-transposed block: owner elements [e0, e1), X0 index = rel
template <class F>
__device__ __forceinline__ void gather_fast_rows(const StreamLaunchArgs& a, const ETile& t,
                                                 const Owner& o, float d, float cpre, char* x0) {
  constexpr int U = 4;
  const int64_t e0 = int64_t(t.r0) * o.cols, e1 = int64_t(t.r0 + t.nr) * o.cols;
  float* __restrict__ M = a.momentum + t.sdelta;
  const int64_t stride = int64_t(4) * kStreamThreads;
  for (int64_t i0 = e0 + 4 * threadIdx.x; i0 < e1; i0 += stride * U) {
    float4 g[U], m[U];
    #pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < e1) {
        g[u] = grad_at4<F>(a, t.sdelta + i);
        m[u] = *reinterpret_cast<const float4*>(M + i);
      }
    }
    #pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < e1) {
        float4 mv;
        mv.x = momentum_of(a.beta, m[u].x, grad_m(a, cpre, g[u].x));
        mv.y = momentum_of(a.beta, m[u].y, grad_m(a, cpre, g[u].y));
        mv.z = momentum_of(a.beta, m[u].z, grad_m(a, cpre, g[u].z));
        mv.w = momentum_of(a.beta, m[u].w, grad_m(a, cpre, g[u].w));
        *reinterpret_cast<float4*>(M + i) = mv;
        store4_ws(x0, a.esize, i,
                  make_float4(__fdiv_rn(mv.x, d), __fdiv_rn(mv.y, d), __fdiv_rn(mv.z, d),
                              __fdiv_rn(mv.w, d)),
                  a.x_ps);
      }
    }
  }
}

// gather_fast_rows with eight elements per thread and step: used when the
// gradient is formed from bf16 micro-batches (16-byte loads of each instead
// of 8-byte ones; measured faster), the tile's storage 8-element aligned and
// its length a multiple of 8
__device__ __forceinline__ void gather_math4(const StreamLaunchArgs& a, float d, float cpre, float4 g,
                                             float4 m, float* M, char* x0, int64_t xi) {
  float4 mv;
  mv.x = momentum_of(a.beta, m.x, grad_m(a, cpre, g.x));
  mv.y = momentum_of(a.beta, m.y, grad_m(a, cpre, g.y));
  mv.z = momentum_of(a.beta, m.z, grad_m(a, cpre, g.z));
  mv.w = momentum_of(a.beta, m.w, grad_m(a, cpre, g.w));
  *reinterpret_cast<float4*>(M) = mv;
  store4_ws(x0, a.esize, xi,
            make_float4(__fdiv_rn(mv.x, d), __fdiv_rn(mv.y, d), __fdiv_rn(mv.z, d), __fdiv_rn(mv.w, d)),
            a.x_ps);
}

template <class F>
__device__ __forceinline__ void gather_fast_rows8(const StreamLaunchArgs& a, const ETile& t,
                                                  const Owner& o, float d, float cpre, char* x0) {
  constexpr int U = 2;
  const int64_t e0 = int64_t(t.r0) * o.cols, e1 = int64_t(t.r0 + t.nr) * o.cols;
  float* __restrict__ M = a.momentum + t.sdelta;
  const int64_t stride = int64_t(8) * kStreamThreads;
  for (int64_t i0 = e0 + 8 * threadIdx.x; i0 < e1; i0 += stride * U) {
    float4 g[U][2], m[U][2];
    #pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < e1) {
        grad_at8<F>(a, t.sdelta + i, g[u][0], g[u][1]);
        m[u][0] = *reinterpret_cast<const float4*>(M + i);
        m[u][1] = *reinterpret_cast<const float4*>(M + i + 4);
      }
    }
    #pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < e1) {
        gather_math4(a, d, cpre, g[u][0], m[u][0], M + i, x0, i);
        gather_math4(a, d, cpre, g[u][1], m[u][1], M + i + 4, x0, i + 4);
      }
    }
  }
}

// 64 x 64 tile of a transposed block: read rows, write X0 = tile^T
template <class F>
__device__ __forceinline__ void gather_fast_tr(const StreamLaunchArgs& a, const ETile& t,
                                               const Owner& o, float d, float cpre, char* x0,
                                               float (*tile)[kTT + 1]) {
  const int r_end = min(t.r0 + kTT, o.rows);
  const int rq = threadIdx.x >> 4, cq = (threadIdx.x & 15) * 4;   // 16 rows x 16 float4 per pass
  float4 g[4], m[4];
  #pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = t.r0 + rq + 16 * k;
    if (r < r_end) {
      const int64_t i = t.sdelta + int64_t(r) * o.cols + t.c0 + cq;
      g[k] = grad_at4<F>(a, i);
      m[k] = *reinterpret_cast<const float4*>(a.momentum + i);
    }
  }
  #pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = t.r0 + rq + 16 * k;
    if (r < r_end) {
      const int64_t i = t.sdelta + int64_t(r) * o.cols + t.c0 + cq;
      float4 mv;
      mv.x = momentum_of(a.beta, m[k].x, grad_m(a, cpre, g[k].x));
      mv.y = momentum_of(a.beta, m[k].y, grad_m(a, cpre, g[k].y));
      mv.z = momentum_of(a.beta, m[k].z, grad_m(a, cpre, g[k].z));
      mv.w = momentum_of(a.beta, m[k].w, grad_m(a, cpre, g[k].w));
      *reinterpret_cast<float4*>(a.momentum + i) = mv;
      float* tr = tile[rq + 16 * k];
      tr[cq] = __fdiv_rn(mv.x, d);
      tr[cq + 1] = __fdiv_rn(mv.y, d);
      tr[cq + 2] = __fdiv_rn(mv.z, d);
      tr[cq + 3] = __fdiv_rn(mv.w, d);
    }
  }
  __syncthreads();
  // X0 rows c0..c0+63 (block columns), 8 elements per thread, 32 rows per pass
  const int xr = threadIdx.x >> 3, rs = (threadIdx.x & 7) * 8;
  #pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int cc = xr + 32 * pass;
    const int64_t xi = int64_t(t.c0 + cc) * o.ldx + t.r0 + rs;
    if (t.r0 + rs + 8 <= r_end) {
      float v[8];
      #pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = tile[rs + k][cc];
      store4_ws(x0, a.esize, xi, make_float4(v[0], v[1], v[2], v[3]), a.x_ps);
      store4_ws(x0, a.esize, xi + 4, make_float4(v[4], v[5], v[6], v[7]), a.x_ps);
    } else {
      for (int k = 0; k < 8 && t.r0 + rs + k < r_end; ++k)
        store_ws(x0, a.esize, xi + k, tile[rs + k][cc], a.x_ps);
    }
  }
}

// 64 x 128 tile of a transposed block (kind 3): 128-column row pieces, eight
// rows of 32 float4 per pass in two halves of four passes; X0 = tile^T
template <class F>
__device__ __forceinline__ void gather_fast_tr2(const StreamLaunchArgs& a, const ETile& t,
                                                const Owner& o, float d, float cpre, char* x0,
                                                float (*tile)[2 * kTT + 1]) {
  const int r_end = min(t.r0 + kTT, o.rows);
  const int rq = threadIdx.x >> 5, cq = (threadIdx.x & 31) * 4;
  #pragma unroll
  for (int h = 0; h < 2; ++h) {
    float4 g[4], m[4];
    #pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int r = t.r0 + rq + 8 * (4 * h + k);
      if (r < r_end) {
        const int64_t i = t.sdelta + int64_t(r) * o.cols + t.c0 + cq;
        g[k] = grad_at4<F>(a, i);
        m[k] = *reinterpret_cast<const float4*>(a.momentum + i);
      }
    }
    #pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int rr = rq + 8 * (4 * h + k);
      if (t.r0 + rr < r_end) {
        const int64_t i = t.sdelta + int64_t(t.r0 + rr) * o.cols + t.c0 + cq;
        float4 mv;
        mv.x = momentum_of(a.beta, m[k].x, grad_m(a, cpre, g[k].x));
        mv.y = momentum_of(a.beta, m[k].y, grad_m(a, cpre, g[k].y));
        mv.z = momentum_of(a.beta, m[k].z, grad_m(a, cpre, g[k].z));
        mv.w = momentum_of(a.beta, m[k].w, grad_m(a, cpre, g[k].w));
        *reinterpret_cast<float4*>(a.momentum + i) = mv;
        float* tr = tile[rr];
        tr[cq] = __fdiv_rn(mv.x, d);
        tr[cq + 1] = __fdiv_rn(mv.y, d);
        tr[cq + 2] = __fdiv_rn(mv.z, d);
        tr[cq + 3] = __fdiv_rn(mv.w, d);
      }
    }
  }
  __syncthreads();
  // X0 rows c0..c0+127 (block columns), 8 elements per thread, 32 rows per pass
  const int xr = threadIdx.x >> 3, rs = (threadIdx.x & 7) * 8;
  #pragma unroll
  for (int pass = 0; pass < 4; ++pass) {
    const int cc = xr + 32 * pass;
    const int64_t xi = int64_t(t.c0 + cc) * o.ldx + t.r0 + rs;
    if (t.r0 + rs + 8 <= r_end) {
      float v[8];
      #pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = tile[rs + k][cc];
      store4_ws(x0, a.esize, xi, make_float4(v[0], v[1], v[2], v[3]), a.x_ps);
      store4_ws(x0, a.esize, xi + 4, make_float4(v[4], v[5], v[6], v[7]), a.x_ps);
    } else {
      for (int k = 0; k < 8 && t.r0 + rs + k < r_end; ++k)
        store_ws(x0, a.esize, xi + k, tile[rs + k][cc], a.x_ps);
    }
  }
}

// gather_fast_tr2 with eight columns per thread (16 rows of 16 threads per
// pass, two halves of two passes), for gradients formed from 16-byte aligned
// bf16 micro-batches; the tile's storage rows 8-element aligned
template <class F>
__device__ __forceinline__ void gather_fast_tr2x8(const StreamLaunchArgs& a, const ETile& t,
                                                  const Owner& o, float d, float cpre, char* x0,
                                                  float (*tile)[2 * kTT + 1]) {
  const int r_end = min(t.r0 + kTT, o.rows);
  const int rq = threadIdx.x >> 4, cq = (threadIdx.x & 15) * 8;
  #pragma unroll
  for (int h = 0; h < 2; ++h) {
    float4 g[2][2], m[2][2];
    #pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int r = t.r0 + rq + 16 * (2 * h + k);
      if (r < r_end) {
        const int64_t i = t.sdelta + int64_t(r) * o.cols + t.c0 + cq;
        grad_at8<F>(a, i, g[k][0], g[k][1]);
        m[k][0] = *reinterpret_cast<const float4*>(a.momentum + i);
        m[k][1] = *reinterpret_cast<const float4*>(a.momentum + i + 4);
      }
    }
    #pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int rr = rq + 16 * (2 * h + k);
      if (t.r0 + rr < r_end) {
        const int64_t i = t.sdelta + int64_t(t.r0 + rr) * o.cols + t.c0 + cq;
        float* tr = tile[rr];
        #pragma unroll
        for (int q = 0; q < 2; ++q) {
          float4 mv;
          mv.x = momentum_of(a.beta, m[k][q].x, grad_m(a, cpre, g[k][q].x));
          mv.y = momentum_of(a.beta, m[k][q].y, grad_m(a, cpre, g[k][q].y));
          mv.z = momentum_of(a.beta, m[k][q].z, grad_m(a, cpre, g[k][q].z));
          mv.w = momentum_of(a.beta, m[k][q].w, grad_m(a, cpre, g[k][q].w));
          *reinterpret_cast<float4*>(a.momentum + i + 4 * q) = mv;
          tr[cq + 4 * q] = __fdiv_rn(mv.x, d);
          tr[cq + 4 * q + 1] = __fdiv_rn(mv.y, d);
          tr[cq + 4 * q + 2] = __fdiv_rn(mv.z, d);
          tr[cq + 4 * q + 3] = __fdiv_rn(mv.w, d);
        }
      }
    }
  }
  __syncthreads();
  const int xr = threadIdx.x >> 3, rs = (threadIdx.x & 7) * 8;
  #pragma unroll
  for (int pass = 0; pass < 4; ++pass) {
    const int cc = xr + 32 * pass;
    const int64_t xi = int64_t(t.c0 + cc) * o.ldx + t.r0 + rs;
    if (t.r0 + rs + 8 <= r_end) {
      float v[8];
      #pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = tile[rs + k][cc];
      store4_ws(x0, a.esize, xi, make_float4(v[0], v[1], v[2], v[3]), a.x_ps);
      store4_ws(x0, a.esize, xi + 4, make_float4(v[4], v[5], v[6], v[7]), a.x_ps);
    } else {
      for (int k = 0; k < 8 && t.r0 + rs + k < r_end; ++k)
        store_ws(x0, a.esize, xi + k, tile[rs + k][cc], a.x_ps);
    }
  }
}

__device__ __forceinline__ void scatter_fast_rows(const StreamLaunchArgs& a, const ETile& t,
                                                  const Owner& o, float coef, bool wm, const char* y) {
  constexpr int U = 4;
  const int64_t e0 = int64_t(t.r0) * o.cols, e1 = int64_t(t.r0 + t.nr) * o.cols;
  float* __restrict__ A = a.accum + t.sdelta;
  float* __restrict__ W = a.master + t.sdelta;
  const int64_t stride = int64_t(4) * kStreamThreads;
  for (int64_t i0 = e0 + 4 * threadIdx.x; i0 < e1; i0 += stride * U) {
    float4 u4[U], w[U];
    #pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < e1) {
        u4[u] = load4_ws(y, a.esize, i, a.x_ps);
        if (wm) w[u] = *reinterpret_cast<const float4*>(W + i);
      }
    }
    #pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < e1) {
        const float4 v = make_float4(__fmul_rn(coef, u4[u].x), __fmul_rn(coef, u4[u].y),
                                     __fmul_rn(coef, u4[u].z), __fmul_rn(coef, u4[u].w));
        *reinterpret_cast<float4*>(A + i) = v;
        if (wm)
          *reinterpret_cast<float4*>(W + i) =
              make_float4(__fsub_rn(w[u].x, __fmul_rn(a.lr, v.x)), __fsub_rn(w[u].y, __fmul_rn(a.lr, v.y)),
                          __fsub_rn(w[u].z, __fmul_rn(a.lr, v.z)), __fsub_rn(w[u].w, __fmul_rn(a.lr, v.w)));
      }
    }
  }
}

__device__ __forceinline__ void scatter_fast_tr(const StreamLaunchArgs& a, const ETile& t,
                                                const Owner& o, float coef, bool wm, const char* y,
                                                float (*tile)[kTT + 1]) {
  const int r_end = min(t.r0 + kTT, o.rows);
  // Y rows c0..c0+63 hold block columns; 8 elements per thread, 32 rows per pass
  const int yr = threadIdx.x >> 3, rs = (threadIdx.x & 7) * 8;
  float4 lo[2], hi[2];
  #pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int64_t yi = int64_t(t.c0 + yr + 32 * pass) * o.ldx + t.r0 + rs;
    if (t.r0 + rs + 8 <= r_end) {
      lo[pass] = load4_ws(y, a.esize, yi, a.x_ps);
      hi[pass] = load4_ws(y, a.esize, yi + 4, a.x_ps);
    } else {
      float v[8];
      for (int k = 0; k < 8; ++k)
        v[k] = (t.r0 + rs + k < r_end) ? load_ws(y, a.esize, yi + k, a.x_ps) : 0.f;
      lo[pass] = make_float4(v[0], v[1], v[2], v[3]);
      hi[pass] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
  #pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int cc = yr + 32 * pass;
    tile[rs + 0][cc] = lo[pass].x; tile[rs + 1][cc] = lo[pass].y;
    tile[rs + 2][cc] = lo[pass].z; tile[rs + 3][cc] = lo[pass].w;
    tile[rs + 4][cc] = hi[pass].x; tile[rs + 5][cc] = hi[pass].y;
    tile[rs + 6][cc] = hi[pass].z; tile[rs + 7][cc] = hi[pass].w;
  }
  __syncthreads();
  const int rq = threadIdx.x >> 4, cq = (threadIdx.x & 15) * 4;
  float4 w[4];
  #pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = t.r0 + rq + 16 * k;
    if (wm && r < r_end)
      w[k] = *reinterpret_cast<const float4*>(a.master + t.sdelta + int64_t(r) * o.cols + t.c0 + cq);
  }
  #pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = t.r0 + rq + 16 * k;
    if (r < r_end) {
      const int64_t i = t.sdelta + int64_t(r) * o.cols + t.c0 + cq;
      const float* tr = tile[rq + 16 * k];
      const float4 v = make_float4(__fmul_rn(coef, tr[cq]), __fmul_rn(coef, tr[cq + 1]),
                                   __fmul_rn(coef, tr[cq + 2]), __fmul_rn(coef, tr[cq + 3]));
      *reinterpret_cast<float4*>(a.accum + i) = v;
      if (wm)
        *reinterpret_cast<float4*>(a.master + i) =
            make_float4(__fsub_rn(w[k].x, __fmul_rn(a.lr, v.x)), __fsub_rn(w[k].y, __fmul_rn(a.lr, v.y)),
                        __fsub_rn(w[k].z, __fmul_rn(a.lr, v.z)), __fsub_rn(w[k].w, __fmul_rn(a.lr, v.w)));
    }
  }
}

// auxiliary elements [rel_begin, rel_begin + len): accum = coef * g, plus
// Adam on the master when enabled
template <class F>
__device__ __forceinline__ void scatter_fast_aux(const StreamLaunchArgs& a, const ETile& t, float coef) {
  constexpr int U = 4;
  float* __restrict__ A = a.accum + t.sdelta;
  const int64_t e0 = t.rel_begin, e1 = t.rel_begin + t.len;
  const int64_t stride = int64_t(4) * kStreamThreads;
  for (int64_t i0 = e0 + 4 * threadIdx.x; i0 < e1; i0 += stride * U) {
    float4 g[U];
    #pragma unroll
    for (int u = 0; u < U; ++u)
      if (i0 + u * stride < e1) g[u] = grad_at4<F>(a, t.sdelta + i0 + u * stride);
    #pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < e1) {
        const float4 v = make_float4(__fmul_rn(coef, grad_in(a, g[u].x)), __fmul_rn(coef, grad_in(a, g[u].y)),
                                     __fmul_rn(coef, grad_in(a, g[u].z)), __fmul_rn(coef, grad_in(a, g[u].w)));
        *reinterpret_cast<float4*>(A + i) = v;
        if (a.adam) adam_four(a, t.sdelta + i, v);
      }
    }
  }
}

// Bounded workspace, final pass over a Muon tile whose unclipped update u
// is parked in accum: accum = coef * u, master -= lr * coef * u.
__device__ __forceinline__ float4 apply4(const StreamLaunchArgs& a, float coef, float* A, float* W) {
  const float4 u = *reinterpret_cast<const float4*>(A);
  const float4 w = *reinterpret_cast<const float4*>(W);
  const float4 v = make_float4(__fmul_rn(coef, u.x), __fmul_rn(coef, u.y), __fmul_rn(coef, u.z),
                               __fmul_rn(coef, u.w));
  *reinterpret_cast<float4*>(W) =
      make_float4(__fsub_rn(w.x, __fmul_rn(a.lr, v.x)), __fsub_rn(w.y, __fmul_rn(a.lr, v.y)),
                  __fsub_rn(w.z, __fmul_rn(a.lr, v.z)), __fsub_rn(w.w, __fmul_rn(a.lr, v.w)));
  return v;
}

__device__ __forceinline__ void apply_parked(const StreamLaunchArgs& a, const ETile& t, const Owner& o,
                                             float coef) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  if (t.fast && t.kind == 0) {
    const int64_t e0 = int64_t(t.r0) * o.cols, e1 = int64_t(t.r0 + t.nr) * o.cols;
    for (int64_t i = e0 + 4 * threadIdx.x; i < e1; i += int64_t(4) * kStreamThreads) {
      float* A = a.accum + t.sdelta + i;
      *reinterpret_cast<float4*>(A) = apply4(a, coef, A, a.master + t.sdelta + i);
    }
    return;
  }
  if (t.fast) {   // 64 x 64 tile of a transposed block, 16 float4 per row
    const int r_end = min(t.r0 + kTT, o.rows);
    const int rq = threadIdx.x >> 4, cq = (threadIdx.x & 15) * 4;
    for (int r = t.r0 + rq; r < r_end; r += kStreamThreads / 16) {
      const int64_t i = t.sdelta + int64_t(r) * o.cols + t.c0 + cq;
      *reinterpret_cast<float4*>(a.accum + i) = apply4(a, coef, a.accum + i, a.master + i);
    }
    return;
  }
  const Segment* segs = a.segs + o.seg_begin;
  const int r_end = t.kind == 0 ? t.r0 + t.nr : min(t.r0 + kTT, o.rows);
  const int c0 = t.kind == 0 ? 0 : t.c0, c_end = t.kind == 0 ? o.cols : min(t.c0 + kTT, o.cols);
  for (int r = t.r0 + warp; r < r_end; r += nw) {
    const int64_t rb = int64_t(r) * o.cols;
    for_row(segs, o.seg_count, rb + c0, rb + c_end, lane, [&](int64_t, int64_t st) {
      const float v = __fmul_rn(coef, a.accum[st]);
      a.accum[st] = v;
      a.master[st] = __fsub_rn(a.master[st], __fmul_rn(a.lr, v));
    });
  }
}

template <class F>
__global__ void __launch_bounds__(kStreamThreads)
k_gather(StreamLaunchArgs a) {
  if (a.state->overflow) return;
  __shared__ float tile2[kTT][2 * kTT + 1];   // kind 3; kind 1 uses it as kTT x (kTT + 1)
  float (*tile)[kTT + 1] = reinterpret_cast<float (*)[kTT + 1]>(&tile2[0][0]);
  const ETile t = a.etiles[blockIdx.x];
  const Owner o = a.owners[t.owner];
#ifdef MUON_DEBUG
  {
    int64_t lo, hi;
    dbg_etile_range(t, o, lo, hi);
    MUON_DBG_CHECK(dbg_tile_ok(a, o, t.fast, t.sdelta, lo, hi, true), a.dbg_flag);
  }
#endif
  const Segment* segs = a.segs + o.seg_begin;
  const float d = a.owner_div[t.owner];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  char* x0 = static_cast<char*>(a.x0) + o.x_off * ebytes(a.esize);
  const float cpre = a.clip_mode == 1 ? a.state->coef : 1.f;
  if (t.fast) {
    // gradients formed from bf16 micro-batches: 16-byte loads where aligned
    const bool v8 = F::kind > 0 && !F::old && a.fold_vec16;
    if (t.kind == 0) {
      const int64_t e0 = int64_t(t.r0) * o.cols, n = int64_t(t.nr) * o.cols;
      if (v8 && ((t.sdelta + e0) & 7) == 0 && (n & 7) == 0) gather_fast_rows8<F>(a, t, o, d, cpre, x0);
      else gather_fast_rows<F>(a, t, o, d, cpre, x0);
    } else if (t.kind == 1) {
      gather_fast_tr<F>(a, t, o, d, cpre, x0, tile);
    } else if (v8 && ((t.sdelta + int64_t(t.r0) * o.cols + t.c0) & 7) == 0 && (o.cols & 7) == 0) {
      gather_fast_tr2x8<F>(a, t, o, d, cpre, x0, tile2);
    } else {
      gather_fast_tr2<F>(a, t, o, d, cpre, x0, tile2);
    }
    return;
  }
  if (t.kind == 0) {
    for (int r = t.r0 + warp; r < t.r0 + t.nr; r += nw) {
      const int64_t rb = int64_t(r) * o.cols;
      for_row(segs, o.seg_count, rb, rb + o.cols, lane, [&](int64_t rel, int64_t st) {
        const float mv = momentum_of(a.beta, a.momentum[st], grad_m(a, cpre, grad_at<F>(a, st)));
        a.momentum[st] = mv;
        store_ws(x0, a.esize, int64_t(r) * o.ldx + (rel - rb), __fdiv_rn(mv, d), a.x_ps);
      });
    }
  } else {
    // transposed block: rows x cols with rows > cols; X0 = block^T (cols x rows)
    const int r_end = min(t.r0 + kTT, o.rows), c_end = min(t.c0 + kTT, o.cols);
    for (int rr = warp; rr < kTT; rr += nw) {
      const int r = t.r0 + rr;
      if (r >= r_end) break;
      const int64_t rb = int64_t(r) * o.cols;
      for_row(segs, o.seg_count, rb + t.c0, rb + c_end, lane, [&](int64_t rel, int64_t st) {
        const float mv = momentum_of(a.beta, a.momentum[st], grad_m(a, cpre, grad_at<F>(a, st)));
        a.momentum[st] = mv;
        tile[rr][rel - rb - t.c0] = __fdiv_rn(mv, d);
      });
    }
    __syncthreads();
    for (int cc = warp; cc < kTT; cc += nw) {
      const int c = t.c0 + cc;
      if (c >= c_end) break;
      for (int rr = lane; rr < kTT && t.r0 + rr < r_end; rr += 32)
        store_ws(x0, a.esize, int64_t(c) * o.ldx + t.r0 + rr, tile[rr][cc], a.x_ps);
    }
  }
}

// ------------------------------------------------------------------ S4a

__global__ void __launch_bounds__(kStreamThreads)
k_update_sumsq(StreamLaunchArgs a) {
  if (a.state->overflow) return;
  const YTile t = a.ytiles[blockIdx.x];
  const Owner o = a.owners[t.owner];
  MUON_DBG_CHECK(dbg_in(o.x_off, o.x_off + int64_t(o.m) * o.ldx, a.dbg_x_extent), a.dbg_flag);
  const char* y = static_cast<const char*>(a.y) + o.x_off * ebytes(a.esize);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per = a.esize == 4 ? 4 : 8;             // elements per 16-byte load (per plane)
  const int nv = (o.n / per) * per;                 // vectorised part of each row
  float acc = 0.f;
  for (int r = t.r0 + warp; r < t.r0 + t.nr; r += kStreamThreads / 32) {
    const int64_t rb = int64_t(r) * o.ldx;
    for (int c = lane * per; c < nv; c += 32 * per) {
      if (a.esize == 4) {
        const uint4 w = *reinterpret_cast<const uint4*>(y + (rb + c) * 4);
        const float* f = reinterpret_cast<const float*>(&w);
        #pragma unroll
        for (int k = 0; k < 4; ++k) acc = __fmaf_rn(f[k], f[k], acc);
      } else {
        float f[8];
        const uint4 w = *reinterpret_cast<const uint4*>(y + (rb + c) * 2);
        const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&w);
        #pragma unroll
        for (int k = 0; k < 8; ++k) f[k] = __bfloat162float(h[k]);
        if (a.esize == 6) {
          const uint4 wm = *reinterpret_cast<const uint4*>(y + (rb + c + a.x_ps) * 2);
          const uint4 wl = *reinterpret_cast<const uint4*>(y + (rb + c + 2 * a.x_ps) * 2);
          const __nv_bfloat16* hm = reinterpret_cast<const __nv_bfloat16*>(&wm);
          const __nv_bfloat16* hl = reinterpret_cast<const __nv_bfloat16*>(&wl);
          #pragma unroll
          for (int k = 0; k < 8; ++k)
            f[k] = __fadd_rn(__fadd_rn(f[k], __bfloat162float(hm[k])), __bfloat162float(hl[k]));
        }
        #pragma unroll
        for (int k = 0; k < 8; ++k) acc = __fmaf_rn(f[k], f[k], acc);
      }
    }
    for (int c = nv + lane; c < o.n; c += 32) {
      const float v = load_ws(y, a.esize, rb + c, a.x_ps);
      acc = __fmaf_rn(v, v, acc);
    }
  }
  const double s = block_sum<kStreamThreads>(static_cast<double>(acc));
  if (threadIdx.x == 0) a.ytile_sum[blockIdx.x] = s;
}

constexpr int kFinThreads = 1024;

// norm = sqrt(tot), coef = min(1, clip / (norm + 1e-6)) (1 when clip <= 0),
// both kept in the step state.
__device__ __forceinline__ void set_clip(const StreamLaunchArgs& a, double tot) {
  const double norm = sqrt(tot);
  double coef = 1.0;
  if (a.clip > 0.f) {
    coef = static_cast<double>(a.clip) / (norm + kClipEps);
    if (coef > 1.0) coef = 1.0;
  }
  a.state->coef = static_cast<float>(coef);
  a.state->norm = static_cast<float>(norm);
  a.state->sumsq = tot;
}

// First level of the global sum of squares: block b of kFinParts adds a
// fixed contiguous range of the tile sums, each thread a fixed strided part
// of it, so the order depends on the tile counts alone.  all_rtiles = 0: the
// update tile sums, then the auxiliary owners' first-pass tile sums (the
// norm over the updates and the auxiliary gradients); 1: every first-pass
// tile sum (clip before Muon: the gradient norm).
__global__ void __launch_bounds__(kStreamThreads)
k_finalize_parts(StreamLaunchArgs a, int all_rtiles) {
  if (a.state->overflow) return;
  const int64_t ny = all_rtiles ? 0 : a.n_ytiles;
  const int64_t total = ny + a.n_rtiles;
  const int64_t per = (total + kFinParts - 1) / kFinParts;
  const int64_t b0 = int64_t(blockIdx.x) * per, b1 = min(total, b0 + per);
  double s = 0.0;
  for (int64_t i = b0 + threadIdx.x; i < b1; i += kStreamThreads) {
    if (i < ny) {
      s += a.ytile_sum[i];
    } else {
      const int64_t j = i - ny;
      if (all_rtiles || !a.owners[a.rtiles[j].owner].is_muon) s += a.rtile_sum[j];
    }
  }
  const double tot = block_sum<kStreamThreads>(s);
  if (threadIdx.x == 0) a.fin_part[blockIdx.x] = tot;
}

__device__ __forceinline__ double fin_total(const StreamLaunchArgs& a) {
  double s = 0.0;
  for (int i = threadIdx.x; i < kFinParts; i += kFinThreads) s += a.fin_part[i];
  return block_sum<kFinThreads>(s);
}

// Clip before Muon: the global norm over every parameter's gradient, from
// the tile sums of reduce mode 1, in a fixed order.
__global__ void __launch_bounds__(kFinThreads)
k_finalize_pre(StreamLaunchArgs a) {
  if (a.state->overflow) return;
  const double tot = fin_total(a);
  if (threadIdx.x == 0) set_clip(a, tot);
}

__global__ void __launch_bounds__(kFinThreads)
k_finalize(StreamLaunchArgs a) {
  if (a.state->overflow) {
    if (threadIdx.x == 0) {
      a.state->applied = 0;
      a.state->coef = 0.f;
      muon_result_t r{0, 0, 0.f, 0.f};
      *a.result = r;
      if (a.stats_out) {
        a.stats_out[0] = 0.0;
        a.stats_out[1] = 1.0;
        a.stats_out[2] = 0.0;
        a.stats_out[3] = 0.0;
      }
    }
    return;
  }
  const int applied = (a.err_flag != nullptr && *a.err_flag != 0) ? -1 : 1;
  if (a.clip_mode == 0) {
    const double tot = fin_total(a);
    if (threadIdx.x == 0) set_clip(a, tot);
  }
  if (threadIdx.x == 0) {
    a.state->applied = applied;
    muon_result_t r{applied, a.ns_calls, a.state->norm, a.state->coef};
    *a.result = r;
    if (a.stats_out) {
      a.stats_out[0] = a.state->sumsq;
      a.stats_out[1] = applied == 1 ? 0.0 : 1.0;
      a.stats_out[2] = static_cast<double>(a.ns_calls);
      a.stats_out[3] = 0.0;
    }
  }
}

// ------------------------------------------------------------------ S4b

// Five blocks per SM (48 registers, a few spilled to L1): the write-heavy
// pass gains from more requests in flight (Llama-3-8B 16.5 -> 15.8 ms); the
// gather at the same bound measured slower, so it keeps four.
template <class F>
__global__ void __launch_bounds__(kStreamThreads, 5)
k_scatter(StreamLaunchArgs a) {
  if (a.state->overflow) return;
  __shared__ float tile[kTT][kTT + 1];
  // clip before Muon: the update is written unscaled (the gradient already
  // carried the coefficient); auxiliary gradients take coef either way
  // Bounded workspace: park 1 (per wave) writes Muon updates only, unscaled
  // and without the master when the coefficient is not known yet; park 2
  // (final pass) applies it to the parked updates and writes the
  // auxiliary parameters.
  const float coef = a.state->coef, lr = a.lr;
  const ETile t = a.etiles[blockIdx.x];
  const Owner o = a.owners[t.owner];
#ifdef MUON_DEBUG
  {
    int64_t lo, hi;
    dbg_etile_range(t, o, lo, hi);
    MUON_DBG_CHECK(dbg_tile_ok(a, o, t.fast, t.sdelta, lo, hi, t.kind != 2), a.dbg_flag);
  }
#endif
  if (a.park == 2 && t.kind != 2) {
    if (a.clip_mode == 0) apply_parked(a, t, o, coef);
    return;
  }
  if (a.park == 1 && t.kind == 2) return;
  const float post = (a.clip_mode == 1 || a.park == 1) ? 1.f : coef;
  const bool wm = !(a.park == 1 && a.clip_mode == 0);
  const Segment* segs = a.segs + o.seg_begin;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  if (t.fast) {
    const char* yb = static_cast<const char*>(a.y) + o.x_off * ebytes(a.esize);
    if (t.kind == 0) scatter_fast_rows(a, t, o, post, wm, yb);
    else if (t.kind == 1) scatter_fast_tr(a, t, o, post, wm, yb, tile);
    else scatter_fast_aux<F>(a, t, coef);
    return;
  }
  if (t.kind == 2) {
    // auxiliary parameter: accum = coef * g; master untouched unless Adam
    const int64_t te = t.rel_begin + t.len;
    int si = find_seg(segs, o.seg_count, t.rel_begin);
    for (; si < o.seg_count && segs[si].rel_begin < te; ++si) {
      const Segment sg = segs[si];
      const int64_t lo = sg.rel_begin > t.rel_begin ? sg.rel_begin : t.rel_begin;
      const int64_t hi = (sg.rel_begin + sg.len) < te ? (sg.rel_begin + sg.len) : te;
      const int64_t base = sg.storage_begin - sg.rel_begin;
      for (int64_t rel = lo + threadIdx.x; rel < hi; rel += blockDim.x) {
        const float v = __fmul_rn(coef, grad_in(a, grad_at<F>(a, base + rel)));
        a.accum[base + rel] = v;
        if (a.adam) adam_one(a, base + rel, v);
      }
    }
    return;
  }
  const char* y = static_cast<const char*>(a.y) + o.x_off * ebytes(a.esize);
  if (t.kind == 0) {
    for (int r = t.r0 + warp; r < t.r0 + t.nr; r += nw) {
      const int64_t rb = int64_t(r) * o.cols;
      for_row(segs, o.seg_count, rb, rb + o.cols, lane, [&](int64_t rel, int64_t st) {
        const float v = __fmul_rn(post, load_ws(y, a.esize, int64_t(r) * o.ldx + (rel - rb), a.x_ps));
        a.accum[st] = v;
        if (wm) a.master[st] = __fsub_rn(a.master[st], __fmul_rn(lr, v));
      });
    }
  } else {
    const int r_end = min(t.r0 + kTT, o.rows), c_end = min(t.c0 + kTT, o.cols);
    // Y is cols x rows here: Y row c holds block column c
    for (int cc = warp; cc < kTT; cc += nw) {
      const int c = t.c0 + cc;
      if (c >= c_end) break;
      for (int rr = lane; rr < kTT && t.r0 + rr < r_end; rr += 32)
        tile[rr][cc] = load_ws(y, a.esize, int64_t(c) * o.ldx + t.r0 + rr, a.x_ps);
    }
    __syncthreads();
    for (int rr = warp; rr < kTT; rr += nw) {
      const int r = t.r0 + rr;
      if (r >= r_end) break;
      const int64_t rb = int64_t(r) * o.cols;
      for_row(segs, o.seg_count, rb + t.c0, rb + c_end, lane, [&](int64_t rel, int64_t st) {
        const float v = __fmul_rn(post, tile[rr][rel - rb - t.c0]);
        a.accum[st] = v;
        if (wm) a.master[st] = __fsub_rn(a.master[st], __fmul_rn(lr, v));
      });
    }
  }
}

// ------------------------------------------------------------------ NS-only entry

__global__ void __launch_bounds__(kStreamThreads)
k_ns_sumsq(const void* X, int io_esize, int64_t numel, double* tile_sum) {
  const int64_t tb = int64_t(blockIdx.x) * kReduceTile;
  const int64_t te = min(tb + kReduceTile, numel);
  float acc = 0.f;
  #pragma unroll 4
  for (int64_t i = tb + threadIdx.x; i < te; i += kStreamThreads) {
    const float v = load_ws(X, io_esize, i);
    acc = __fmaf_rn(v, v, acc);
  }
  const double s = block_sum<kStreamThreads>(static_cast<double>(acc));
  if (threadIdx.x == 0) tile_sum[blockIdx.x] = s;
}

__global__ void __launch_bounds__(kFinThreads)
k_ns_norm(double* tile_sum, int ntiles) {
  double s = 0.0;
  for (int i = threadIdx.x; i < ntiles; i += kFinThreads) s += tile_sum[i];
  const double tot = block_sum<kFinThreads>(s);
  // the divisor is stored as a float in slot ntiles
  if (threadIdx.x == 0)
    reinterpret_cast<float*>(tile_sum + ntiles)[0] = static_cast<float>(sqrt(tot) + kNormEps);
}

// X (rows x cols, io dtype) -> X0 (m x n canonical, workspace dtype) = X / d
__global__ void __launch_bounds__(kStreamThreads)
k_ns_load(const void* X, int io_esize, int rows, int cols, const double* tile_sum, int ntiles,
          void* X0, int esize, int ldx, int64_t ps) {
  __shared__ float tile[kTT][kTT + 1];
  const float d = reinterpret_cast<const float*>(tile_sum + ntiles)[0];
  const int r0 = blockIdx.y * kTT, c0 = blockIdx.x * kTT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool tr = rows > cols;
  for (int rr = warp; rr < kTT; rr += 8) {
    const int r = r0 + rr;
    if (r >= rows) break;
    for (int cc = lane; cc < kTT && c0 + cc < cols; cc += 32) {
      const float v = __fdiv_rn(load_ws(X, io_esize, int64_t(r) * cols + c0 + cc), d);
      if (tr) tile[rr][cc] = v;
      else store_ws(X0, esize, int64_t(r) * ldx + c0 + cc, v, ps);
    }
  }
  if (!tr) return;
  __syncthreads();
  for (int cc = warp; cc < kTT; cc += 8) {
    const int c = c0 + cc;
    if (c >= cols) break;
    for (int rr = lane; rr < kTT && r0 + rr < rows; rr += 32)
      store_ws(X0, esize, int64_t(c) * ldx + r0 + rr, tile[rr][cc], ps);
  }
}

// Y workspace (m x n canonical) -> Y (rows x cols, io dtype)
__global__ void __launch_bounds__(kStreamThreads)
k_ns_store(const void* Yws, int esize, int ldx, int64_t ps, void* Y, int io_esize, int rows,
           int cols) {
  __shared__ float tile[kTT][kTT + 1];
  const int r0 = blockIdx.y * kTT, c0 = blockIdx.x * kTT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool tr = rows > cols;
  if (!tr) {
    for (int rr = warp; rr < kTT; rr += 8) {
      const int r = r0 + rr;
      if (r >= rows) break;
      for (int cc = lane; cc < kTT && c0 + cc < cols; cc += 32)
        store_ws(Y, io_esize, int64_t(r) * cols + c0 + cc,
                 load_ws(Yws, esize, int64_t(r) * ldx + c0 + cc, ps));
    }
    return;
  }
  for (int cc = warp; cc < kTT; cc += 8) {
    const int c = c0 + cc;
    if (c >= cols) break;
    for (int rr = lane; rr < kTT && r0 + rr < rows; rr += 32)
      tile[rr][cc] = load_ws(Yws, esize, int64_t(c) * ldx + r0 + rr, ps);
  }
  __syncthreads();
  for (int rr = warp; rr < kTT; rr += 8) {
    const int r = r0 + rr;
    if (r >= rows) break;
    for (int cc = lane; cc < kTT && c0 + cc < cols; cc += 32)
      store_ws(Y, io_esize, int64_t(r) * cols + c0 + cc, tile[rr][cc]);
  }
}

}  // namespace

// ------------------------------------------------------------------ launchers

void launch_accumulate(float* accum, const uint16_t* grad, const Run* runs, int nruns,
                       float scale, int overwrite, int64_t dbg_extent, int* dbg_flag,
                       cudaStream_t s) {
  if (nruns > 0)
    k_accumulate<<<nruns, kStreamThreads, 0, s>>>(accum, grad, runs, scale, overwrite, dbg_extent,
                                                  dbg_flag);
}
// The instantiation for the launch's gradient source (Fold above).
#define MUON_FOLD_LAUNCH(kernel, grid, a, s)                                                  \
  do {                                                                                       \
    const bool lg = (a).last_grad != nullptr;                                                \
    const bool two = lg && (a).prev_grad != nullptr && !(a).last_overwrite;                  \
    const bool old = !lg || !((a).last_overwrite || (two && (a).prev_overwrite));            \
    if (!lg) kernel<Fold<0, true>><<<(grid), kStreamThreads, 0, (s)>>>(a);                   \
    else if (!two && old) kernel<Fold<1, true>><<<(grid), kStreamThreads, 0, (s)>>>(a);      \
    else if (!two) kernel<Fold<1, false>><<<(grid), kStreamThreads, 0, (s)>>>(a);            \
    else if (old) kernel<Fold<2, true>><<<(grid), kStreamThreads, 0, (s)>>>(a);              \
    else kernel<Fold<2, false>><<<(grid), kStreamThreads, 0, (s)>>>(a);                      \
  } while (0)

void launch_accumulate_n(float* accum, const GradSet& gs, const Run* runs, int nruns, int overwrite,
                         int64_t dbg_extent, int* dbg_flag, cudaStream_t s) {
  if (nruns <= 0) return;
  switch (gs.count) {
#define MUON_ACC_CASE(C)                                                                         \
  case C:                                                                                        \
    k_accumulate_n<C><<<nruns, kStreamThreads, 0, s>>>(accum, gs, runs, overwrite, dbg_extent,  \
                                                       dbg_flag);                                \
    break;
    MUON_ACC_CASE(1) MUON_ACC_CASE(2) MUON_ACC_CASE(3) MUON_ACC_CASE(4)
    MUON_ACC_CASE(5) MUON_ACC_CASE(6) MUON_ACC_CASE(7) MUON_ACC_CASE(8)
#undef MUON_ACC_CASE
    default:
      break;
  }
}
void launch_reduce(const StreamLaunchArgs& a, cudaStream_t s) {
  if (a.n_rtiles > 0) MUON_FOLD_LAUNCH(k_reduce, a.n_rtiles, a, s);
}
void launch_fold_commit(const StreamLaunchArgs& a, cudaStream_t s) {
  if (a.n_rtiles > 0 && a.last_grad)
    MUON_FOLD_LAUNCH(k_fold_commit, std::min(a.n_rtiles, kFoldCommitCtas), a, s);
}
bool fold_reads_accum(const StreamLaunchArgs& a) {
  return a.last_grad && !(a.last_overwrite || (a.prev_grad && a.prev_overwrite));
}
void launch_owner_norm(const StreamLaunchArgs& a, cudaStream_t s) {
  if (a.n_owners > 0) k_owner_norm<<<(a.n_owners + 127) / 128, 128, 0, s>>>(a);
}
void launch_gather(const StreamLaunchArgs& a, cudaStream_t s) {
  if (a.n_etiles > 0) MUON_FOLD_LAUNCH(k_gather, a.n_etiles, a, s);
}
void launch_update_sumsq(const StreamLaunchArgs& a, cudaStream_t s) {
  if (a.n_ytiles > 0) k_update_sumsq<<<a.n_ytiles, kStreamThreads, 0, s>>>(a);
}
void launch_finalize(const StreamLaunchArgs& a, cudaStream_t s) {
  if (a.clip_mode == 0) k_finalize_parts<<<kFinParts, kStreamThreads, 0, s>>>(a, 0);
  k_finalize<<<1, kFinThreads, 0, s>>>(a);
}
void launch_finalize_pre(const StreamLaunchArgs& a, cudaStream_t s) {
  k_finalize_parts<<<kFinParts, kStreamThreads, 0, s>>>(a, 1);
  k_finalize_pre<<<1, kFinThreads, 0, s>>>(a);
}
void launch_scatter(const StreamLaunchArgs& a, cudaStream_t s) {
  if (a.n_etiles > 0) MUON_FOLD_LAUNCH(k_scatter, a.n_etiles, a, s);
}

void launch_ns_sumsq(const void* X, int io_esize, int64_t numel, double* tile_sum, int ntiles,
                     cudaStream_t s) {
  k_ns_sumsq<<<ntiles, kStreamThreads, 0, s>>>(X, io_esize, numel, tile_sum);
  k_ns_norm<<<1, kFinThreads, 0, s>>>(tile_sum, ntiles);
}
void launch_ns_load(const void* X, int io_esize, int rows, int cols, const double* tile_sum,
                    int ntiles, void* X0, int esize, int ldx, int64_t ps, cudaStream_t s) {
  dim3 g((cols + kTT - 1) / kTT, (rows + kTT - 1) / kTT);
  k_ns_load<<<g, kStreamThreads, 0, s>>>(X, io_esize, rows, cols, tile_sum, ntiles, X0, esize, ldx,
                                         ps);
}
void launch_ns_store(const void* Yws, int esize, int ldx, int64_t ps, void* Y, int io_esize,
                     int rows, int cols, cudaStream_t s) {
  dim3 g((cols + kTT - 1) / kTT, (rows + kTT - 1) / kTT);
  k_ns_store<<<g, kStreamThreads, 0, s>>>(Yws, esize, ldx, ps, Y, io_esize, rows, cols);
}

}  // namespace muon
