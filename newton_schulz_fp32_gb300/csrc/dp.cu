// Data parallelism across ranks: the plan (every parameter assigned to one
// owner rank, the exchange tables of the slices each rank holds) and the
// pack / unpack / write-back kernels around the two all-to-all exchanges.
//
// The pages split the step over ranks that each hold their partitions of the
// flat buffers: the slices of a matrix that crosses partitions are exchanged
// with static send/recv split tables computed once ("Support Muon in
// BF16_Optimizer with FP32 gradient accumulation", review thread on
// all_to_all_single), Muon runs on whole matrices spread over the ranks
// ("Run Muon once per optimizer step under ZeRO-3, not once per
// micro-batch", "The change"), and each rank writes back only its owned
// intersection (the BF16 PR's description).  The collectives themselves are
// the caller's (one all-to-all each way and one all-reduce of four doubles);
// this file computes the tables and moves the bytes on this GPU.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <memory>
#include <mutex>
#include <numeric>
#include <string>
#include <vector>

#include "muon_internal.h"

namespace muon {
namespace {

constexpr int kDpChunk = 16384;      // elements per block of the copy kernels
constexpr int kDpThreads = 256;
constexpr double kStreamCost = 12500.0;   // flop-equivalents per element streamed

int dpfail(int code, const std::string& msg) {
  set_last_error(msg.c_str());
  return code;
}

int64_t up4(int64_t x) { return (x + 3) & ~int64_t(3); }

// One block's share of a segment.  buf_m < 0: no momentum slice.
struct DpChunk {
  int64_t local;
  int64_t buf_g;
  int64_t buf_m;
  int32_t len;
  int32_t fast;   // local, buf_g, buf_m and len all multiples of 4: 16-byte accesses
};

double ns_cost(const muon_param_t& p, int method) {
  if (!p.use_muon) return kStreamCost * double(p.rows) * p.cols;
  const int h = p.num_heads > 1 ? p.num_heads : 1;
  const double r = double(p.rows / h), c = double(p.cols);
  const double m = std::min(r, c), n = std::max(r, c);
  const double f = method == MUON_NS_STANDARD ? 5.0 * (4.0 * m * m * n + 2.0 * m * m * m)
                                              : 4.0 * m * m * n + 34.0 * m * m * m;
  return h * f + kStreamCost * double(p.rows) * p.cols;
}

}  // namespace
}  // namespace muon

using namespace muon;

struct muon_dp_plan {
  int world = 1, rank = 0, nparams = 0;
  std::vector<int32_t> owner;
  std::vector<int64_t> send_counts, recv_counts;
  std::vector<muon_param_t> owned;
  int64_t owned_elems = 0;
  std::vector<muon_dp_segment_t> send, recv;
  int64_t send_elems = 0, recv_elems = 0;
  double owned_cost = 0.0, max_cost = 0.0;
  std::vector<DpChunk> send_chunks, recv_chunks;
  int device = -1;
  DpChunk* d_send = nullptr;
  DpChunk* d_recv = nullptr;
};

namespace muon {
namespace {

// Splits segments into blocks of at most kDpChunk elements.
std::vector<DpChunk> chunks_of(const std::vector<muon_dp_segment_t>& segs) {
  std::vector<DpChunk> out;
  for (const muon_dp_segment_t& s : segs)
    for (int64_t o = 0; o < s.len; o += kDpChunk) {
      DpChunk c{};
      c.len = static_cast<int32_t>(std::min<int64_t>(kDpChunk, s.len - o));
      c.local = s.local + o;
      c.buf_g = s.buf + o;
      c.buf_m = s.is_muon ? s.buf + up4(s.len) + o : -1;
      c.fast = (c.local % 4 == 0 && c.buf_g % 4 == 0 && (c.buf_m < 0 || c.buf_m % 4 == 0) &&
                c.len % 4 == 0) ? 1 : 0;
      out.push_back(c);
    }
  return out;
}

int upload_chunks(muon_dp_plan* P) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return dpfail(MUON_ERR_CUDA, "cudaGetDevice failed");
  if (P->device == dev) return MUON_OK;
  if (P->device >= 0) return dpfail(MUON_ERR_INVALID, "a data-parallel plan serves one device");
  auto up = [](const std::vector<DpChunk>& v, DpChunk** d) {
    const size_t bytes = std::max<size_t>(1, v.size()) * sizeof(DpChunk);
    if (cudaMalloc(reinterpret_cast<void**>(d), bytes) != cudaSuccess) return false;
    return v.empty() ||
           cudaMemcpy(*d, v.data(), v.size() * sizeof(DpChunk), cudaMemcpyHostToDevice) == cudaSuccess;
  };
  if (!up(P->send_chunks, &P->d_send) || !up(P->recv_chunks, &P->d_recv))
    return dpfail(MUON_ERR_OOM, "uploading the exchange tables failed");
  P->device = dev;
  return MUON_OK;
}

__global__ void __launch_bounds__(kDpThreads)
k_dp_gather(const DpChunk* __restrict__ ch, float* __restrict__ buf, const float* __restrict__ a,
            const float* __restrict__ b) {
  const DpChunk c = ch[blockIdx.x];
  if (c.fast) {
    for (int i = 4 * threadIdx.x; i < c.len; i += 4 * kDpThreads) {
      *reinterpret_cast<float4*>(buf + c.buf_g + i) = *reinterpret_cast<const float4*>(a + c.local + i);
      if (c.buf_m >= 0)
        *reinterpret_cast<float4*>(buf + c.buf_m + i) = *reinterpret_cast<const float4*>(b + c.local + i);
    }
    return;
  }
  for (int i = threadIdx.x; i < c.len; i += kDpThreads) {
    buf[c.buf_g + i] = a[c.local + i];
    if (c.buf_m >= 0) buf[c.buf_m + i] = b[c.local + i];
  }
}

__global__ void __launch_bounds__(kDpThreads)
k_dp_scatter(const DpChunk* __restrict__ ch, const float* __restrict__ buf, float* __restrict__ a,
             float* __restrict__ b) {
  const DpChunk c = ch[blockIdx.x];
  if (c.fast) {
    for (int i = 4 * threadIdx.x; i < c.len; i += 4 * kDpThreads) {
      *reinterpret_cast<float4*>(a + c.local + i) = *reinterpret_cast<const float4*>(buf + c.buf_g + i);
      if (c.buf_m >= 0)
        *reinterpret_cast<float4*>(b + c.local + i) = *reinterpret_cast<const float4*>(buf + c.buf_m + i);
    }
    return;
  }
  for (int i = threadIdx.x; i < c.len; i += kDpThreads) {
    a[c.local + i] = buf[c.buf_g + i];
    if (c.buf_m >= 0) b[c.local + i] = buf[c.buf_m + i];
  }
}

// The clip coefficient from the all-reduced sum of squares, as the
// single-GPU step forms it: norm = sqrt(sum) in double, coef = min(1,
// clip / (norm + 1e-6)) in double, both rounded to FP32.
__device__ __forceinline__ void dp_coef(const double* stats, float clip, float* coef, float* norm) {
  const double n = sqrt(stats[0]);
  double c = 1.0;
  if (clip > 0.f) {
    c = static_cast<double>(clip) / (n + kClipEps);
    if (c > 1.0) c = 1.0;
  }
  *coef = static_cast<float>(c);
  *norm = static_cast<float>(n);
}

// Write-back of the held slices: Muon v = coef u, accum = v, master -= lr v,
// momentum = m'; auxiliary accum = coef g (the same FP32 operations as the
// single-GPU write-back).  Nothing is written when any rank skipped.
__global__ void __launch_bounds__(kDpThreads)
k_dp_finish(const DpChunk* __restrict__ ch, const float* __restrict__ buf, float* __restrict__ accum,
            float* __restrict__ momentum, float* __restrict__ master, const double* __restrict__ stats,
            float lr, float clip) {
  if (stats[1] > 0.0) return;
  float coef, norm;
  dp_coef(stats, clip, &coef, &norm);
  const DpChunk c = ch[blockIdx.x];
  if (c.fast) {
    for (int i = 4 * threadIdx.x; i < c.len; i += 4 * kDpThreads) {
      const float4 u = *reinterpret_cast<const float4*>(buf + c.buf_g + i);
      const float4 v = make_float4(__fmul_rn(coef, u.x), __fmul_rn(coef, u.y), __fmul_rn(coef, u.z),
                                   __fmul_rn(coef, u.w));
      *reinterpret_cast<float4*>(accum + c.local + i) = v;
      if (c.buf_m >= 0) {
        const float4 w = *reinterpret_cast<const float4*>(master + c.local + i);
        *reinterpret_cast<float4*>(master + c.local + i) =
            make_float4(__fsub_rn(w.x, __fmul_rn(lr, v.x)), __fsub_rn(w.y, __fmul_rn(lr, v.y)),
                        __fsub_rn(w.z, __fmul_rn(lr, v.z)), __fsub_rn(w.w, __fmul_rn(lr, v.w)));
        *reinterpret_cast<float4*>(momentum + c.local + i) =
            *reinterpret_cast<const float4*>(buf + c.buf_m + i);
      }
    }
    return;
  }
  for (int i = threadIdx.x; i < c.len; i += kDpThreads) {
    const float v = __fmul_rn(coef, buf[c.buf_g + i]);
    accum[c.local + i] = v;
    if (c.buf_m >= 0) {
      master[c.local + i] = __fsub_rn(master[c.local + i], __fmul_rn(lr, v));
      momentum[c.local + i] = buf[c.buf_m + i];
    }
  }
}

__global__ void k_dp_result(const double* __restrict__ stats, float clip, muon_result_t* r) {
  if (stats[1] > 0.0) {
    muon_result_t z{0, 0, 0.f, 0.f};
    *r = z;
    return;
  }
  float coef, norm;
  dp_coef(stats, clip, &coef, &norm);
  muon_result_t o{1, static_cast<int32_t>(stats[2]), norm, coef};
  *r = o;
}

bool misaligned(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 != 0; }

}  // namespace
}  // namespace muon

extern "C" int muon_dp_plan_create(const muon_param_t* params, int nparams,
                                   const muon_partition_t* parts, const int32_t* part_rank,
                                   int nparts, int world, int rank, int ns_method, int assign,
                                   muon_dp_plan_t** out) {
  std::lock_guard<std::mutex> lk(library_mutex());
  set_last_error(nullptr);
  if (!out) return dpfail(MUON_ERR_INVALID, "out is NULL");
  *out = nullptr;
  if (world < 1 || rank < 0 || rank >= world)
    return dpfail(MUON_ERR_INVALID, "world must be >= 1 and rank in [0, world)");
  if (ns_method != MUON_NS_STANDARD && ns_method != MUON_NS_GRAM)
    return dpfail(MUON_ERR_UNSUPPORTED, "unknown ns_method");
  if (assign != MUON_DP_BALANCED && assign != MUON_DP_ROUND_ROBIN)
    return dpfail(MUON_ERR_INVALID, "unknown assignment");
  if (nparts > 0 && !part_rank) return dpfail(MUON_ERR_INVALID, "part_rank is NULL");
  if (nparts < 0 || (nparts > 0 && !parts)) return dpfail(MUON_ERR_INVALID, "bad partition table");
  for (int p = 0; p < nparts; ++p)
    if (part_rank[p] < 0 || part_rank[p] >= world)
      return dpfail(MUON_ERR_INVALID, "part_rank[" + std::to_string(p) + "] outside [0, world)");
  // The tables as one flat space (storage offsets made distinct: each rank's
  // storage is its own) go through the single-GPU step's validation; then
  // storage overlaps are checked rank by rank.
  std::vector<muon_partition_t> flat(parts, parts + nparts);
  for (muon_partition_t& q : flat) {
    if (q.storage_offset < 0) return dpfail(MUON_ERR_INVALID, "negative storage offset");
    q.storage_offset = q.flat_begin;
  }
  int rc = validate_tables(params, nparams, flat.data(), nparts);
  if (rc != MUON_OK) return rc;
  for (int r = 0; r < world; ++r) {
    std::vector<std::pair<int64_t, int64_t>> st;
    for (int p = 0; p < nparts; ++p)
      if (part_rank[p] == r && parts[p].flat_end > parts[p].flat_begin)
        st.push_back({parts[p].storage_offset,
                      parts[p].storage_offset + parts[p].flat_end - parts[p].flat_begin});
    std::sort(st.begin(), st.end());
    for (size_t i = 1; i < st.size(); ++i)
      if (st[i - 1].second > st[i].first)
        return dpfail(MUON_ERR_INVALID, "partitions of rank " + std::to_string(r) + " overlap in storage");
  }

  std::unique_ptr<muon_dp_plan> P(new muon_dp_plan());
  P->world = world;
  P->rank = rank;
  P->nparams = nparams;
  P->owner.assign(nparams, 0);
  // assignment
  std::vector<double> cost(nparams), load(world, 0.0);
  for (int k = 0; k < nparams; ++k) cost[k] = ns_cost(params[k], ns_method);
  if (assign == MUON_DP_ROUND_ROBIN) {
    for (int k = 0; k < nparams; ++k) P->owner[k] = k % world;
  } else {
    std::vector<int> order(nparams);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return cost[x] > cost[y]; });
    for (int k : order) {
      int best = 0;
      for (int r = 1; r < world; ++r)
        if (load[r] < load[best]) best = r;
      P->owner[k] = best;
      load[best] += cost[k];
    }
  }
  std::fill(load.begin(), load.end(), 0.0);
  for (int k = 0; k < nparams; ++k) load[P->owner[k]] += cost[k];
  P->owned_cost = load[rank];
  P->max_cost = *std::max_element(load.begin(), load.end());

  // packed owned layout: owned parameters in table order, 32-element aligned
  std::vector<int64_t> owned_off(nparams, -1);
  for (int k = 0; k < nparams; ++k)
    if (P->owner[k] == rank) {
      owned_off[k] = P->owned_elems;
      muon_param_t q = params[k];
      q.offset = P->owned_elems;
      P->owned.push_back(q);
      P->owned_elems += (int64_t(params[k].rows) * params[k].cols + 31) / 32 * 32;
    }

  // every (parameter, partition) intersection that this rank sends or receives
  struct Raw { int32_t param, src, dst, muon; int64_t rel, len, src_storage; };
  std::vector<Raw> raws;
  for (int k = 0; k < nparams; ++k) {
    const muon_param_t& p = params[k];
    const int64_t b = p.offset, e = p.offset + int64_t(p.rows) * p.cols;
    for (int q = 0; q < nparts; ++q) {
      const int64_t lo = std::max(b, parts[q].flat_begin), hi = std::min(e, parts[q].flat_end);
      if (lo >= hi) continue;
      const int src = part_rank[q], dst = P->owner[k];
      if (src != rank && dst != rank) continue;
      raws.push_back({k, src, dst, p.use_muon ? 1 : 0, lo - b, hi - lo,
                      parts[q].storage_offset + (lo - parts[q].flat_begin)});
    }
  }
  P->send_counts.assign(world, 0);
  P->recv_counts.assign(world, 0);
  auto build = [&](bool sending) {
    std::vector<Raw> v;
    for (const Raw& r : raws)
      if ((sending ? r.src : r.dst) == rank) v.push_back(r);
    std::stable_sort(v.begin(), v.end(), [&](const Raw& x, const Raw& y) {
      const int px = sending ? x.dst : x.src, py = sending ? y.dst : y.src;
      if (px != py) return px < py;
      if (x.param != y.param) return x.param < y.param;
      return x.rel < y.rel;
    });
    std::vector<muon_dp_segment_t> segs;
    int64_t off = 0;
    for (const Raw& r : v) {
      muon_dp_segment_t s{};
      s.param = r.param;
      s.peer = sending ? r.dst : r.src;
      s.is_muon = r.muon;
      s.len = r.len;
      s.local = sending ? r.src_storage : owned_off[r.param] + r.rel;
      s.buf = off;
      const int64_t payload = up4(r.len) * (r.muon ? 2 : 1);
      off += payload;
      (sending ? P->send_counts : P->recv_counts)[s.peer] += payload;
      segs.push_back(s);
    }
    (sending ? P->send_elems : P->recv_elems) = off;
    return segs;
  };
  P->send = build(true);
  P->recv = build(false);
  P->send_chunks = chunks_of(P->send);
  P->recv_chunks = chunks_of(P->recv);
  *out = P.release();
  return MUON_OK;
}

extern "C" void muon_dp_plan_destroy(muon_dp_plan_t* plan) {
  if (!plan) return;
  std::lock_guard<std::mutex> lk(library_mutex());
  if (plan->d_send) cudaFree(plan->d_send);
  if (plan->d_recv) cudaFree(plan->d_recv);
  delete plan;
}

extern "C" int muon_dp_plan_sizes(const muon_dp_plan_t* plan, muon_dp_sizes_t* out) {
  std::lock_guard<std::mutex> lk(library_mutex());
  set_last_error(nullptr);
  if (!plan || !out) return dpfail(MUON_ERR_INVALID, "plan or out is NULL");
  std::memset(out, 0, sizeof(*out));
  out->world = plan->world;
  out->rank = plan->rank;
  out->owned_params = static_cast<int32_t>(plan->owned.size());
  out->nparams = plan->nparams;
  out->owned_elems = plan->owned_elems;
  out->send_segments = static_cast<int64_t>(plan->send.size());
  out->recv_segments = static_cast<int64_t>(plan->recv.size());
  out->send_elems = plan->send_elems;
  out->recv_elems = plan->recv_elems;
  out->owned_cost = plan->owned_cost;
  out->max_cost = plan->max_cost;
  return MUON_OK;
}

extern "C" int muon_dp_plan_tables(const muon_dp_plan_t* plan, int32_t* owner,
                                   int64_t* send_counts, int64_t* recv_counts,
                                   muon_param_t* owned_params, muon_dp_segment_t* send_segs,
                                   muon_dp_segment_t* recv_segs) {
  std::lock_guard<std::mutex> lk(library_mutex());
  set_last_error(nullptr);
  if (!plan) return dpfail(MUON_ERR_INVALID, "plan is NULL");
  auto put = [](auto* dst, const auto& v) {
    if (dst && !v.empty()) std::memcpy(dst, v.data(), v.size() * sizeof(v[0]));
  };
  put(owner, plan->owner);
  put(send_counts, plan->send_counts);
  put(recv_counts, plan->recv_counts);
  put(owned_params, plan->owned);
  put(send_segs, plan->send);
  put(recv_segs, plan->recv);
  return MUON_OK;
}

extern "C" int muon_dp_pack(muon_dp_plan_t* plan, int direction, float* buf, const float* a,
                            const float* b, void* stream) {
  std::lock_guard<std::mutex> lk(library_mutex());
  NvtxRange nvtx_("muon_dp_pack");
  set_last_error(nullptr);
  if (!plan) return dpfail(MUON_ERR_INVALID, "plan is NULL");
  if (direction != MUON_DP_SEND && direction != MUON_DP_RECV)
    return dpfail(MUON_ERR_INVALID, "unknown direction");
  const auto& chunks = direction == MUON_DP_SEND ? plan->send_chunks : plan->recv_chunks;
  if (chunks.empty()) return MUON_OK;
  if (!buf || !a || !b) return dpfail(MUON_ERR_INVALID, "NULL buffer");
  if (misaligned(buf) || misaligned(a) || misaligned(b))
    return dpfail(MUON_ERR_INVALID, "exchange and state buffers must be 16-byte aligned");
  int rc = upload_chunks(plan);
  if (rc != MUON_OK) return rc;
  const DpChunk* d = direction == MUON_DP_SEND ? plan->d_send : plan->d_recv;
  k_dp_gather<<<static_cast<unsigned>(chunks.size()), kDpThreads, 0,
                static_cast<cudaStream_t>(stream)>>>(d, buf, a, b);
  if (cudaGetLastError() != cudaSuccess) return dpfail(MUON_ERR_CUDA, "kernel launch failed");
  count_launches(1);
  return MUON_OK;
}

extern "C" int muon_dp_unpack(muon_dp_plan_t* plan, int direction, const float* buf, float* a,
                              float* b, void* stream) {
  std::lock_guard<std::mutex> lk(library_mutex());
  NvtxRange nvtx_("muon_dp_unpack");
  set_last_error(nullptr);
  if (!plan) return dpfail(MUON_ERR_INVALID, "plan is NULL");
  if (direction != MUON_DP_SEND && direction != MUON_DP_RECV)
    return dpfail(MUON_ERR_INVALID, "unknown direction");
  const auto& chunks = direction == MUON_DP_SEND ? plan->send_chunks : plan->recv_chunks;
  if (chunks.empty()) return MUON_OK;
  if (!buf || !a || !b) return dpfail(MUON_ERR_INVALID, "NULL buffer");
  if (misaligned(buf) || misaligned(a) || misaligned(b))
    return dpfail(MUON_ERR_INVALID, "exchange and state buffers must be 16-byte aligned");
  int rc = upload_chunks(plan);
  if (rc != MUON_OK) return rc;
  const DpChunk* d = direction == MUON_DP_SEND ? plan->d_send : plan->d_recv;
  k_dp_scatter<<<static_cast<unsigned>(chunks.size()), kDpThreads, 0,
                 static_cast<cudaStream_t>(stream)>>>(d, buf, a, b);
  if (cudaGetLastError() != cudaSuccess) return dpfail(MUON_ERR_CUDA, "kernel launch failed");
  count_launches(1);
  return MUON_OK;
}

extern "C" int muon_dp_finish(muon_dp_plan_t* plan, const float* buf, float* accum,
                              float* momentum, float* master, const double* stats, float lr,
                              float clip, muon_result_t* d_result, void* stream) {
  std::lock_guard<std::mutex> lk(library_mutex());
  NvtxRange nvtx_("muon_dp_finish");
  set_last_error(nullptr);
  if (!plan) return dpfail(MUON_ERR_INVALID, "plan is NULL");
  if (!stats || !d_result) return dpfail(MUON_ERR_INVALID, "stats or d_result is NULL");
  if (reinterpret_cast<uintptr_t>(stats) % 8) return dpfail(MUON_ERR_INVALID, "stats must be 8-byte aligned");
  if (!std::isfinite(lr) || !std::isfinite(clip)) return dpfail(MUON_ERR_INVALID, "lr and clip must be finite");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!plan->send_chunks.empty()) {
    if (!buf || !accum || !momentum || !master) return dpfail(MUON_ERR_INVALID, "NULL buffer");
    if (misaligned(buf) || misaligned(accum) || misaligned(momentum) || misaligned(master))
      return dpfail(MUON_ERR_INVALID, "exchange and state buffers must be 16-byte aligned");
    int rc = upload_chunks(plan);
    if (rc != MUON_OK) return rc;
    k_dp_finish<<<static_cast<unsigned>(plan->send_chunks.size()), kDpThreads, 0, s>>>(
        plan->d_send, buf, accum, momentum, master, stats, lr, clip);
  }
  k_dp_result<<<1, 1, 0, s>>>(stats, clip, d_result);
  if (cudaGetLastError() != cudaSuccess) return dpfail(MUON_ERR_CUDA, "kernel launch failed");
  count_launches(plan->send_chunks.empty() ? 1 : 2);
  return MUON_OK;
}
