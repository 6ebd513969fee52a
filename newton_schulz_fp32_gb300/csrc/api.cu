// C ABI of libmuon: argument and table validation, the planner (tables ->
// owners, segments, tiles, grouped GEMM work lists, workspace), the plan
// cache, and the launch sequence of one Muon step.
//
// The tables are static for a training run, so everything derived from them
// is computed once, copied to the device and reused ("layout is static,
// computed once in init": "Support Muon in BF16_Optimizer with FP32 gradient
// accumulation", review thread on the all_to_all_single split tables).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "muon_internal.h"

namespace muon {
namespace {

thread_local std::string g_err;

int fail(int code, const std::string& msg) {
  g_err = msg;
  return code;
}

#define MUON_CUDA_TRY(expr)                                                        \
  do {                                                                             \
    cudaError_t e_ = (expr);                                                       \
    if (e_ != cudaSuccess)                                                         \
      return fail(e_ == cudaErrorMemoryAllocation ? MUON_ERR_OOM : MUON_ERR_CUDA,  \
                  std::string(#expr) + ": " + cudaGetErrorString(e_));             \
  } while (0)

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// ------------------------------------------------------------------ device memory

struct DevBuf {
  void* p = nullptr;
  size_t bytes = 0;
  DevBuf() = default;
  DevBuf(const DevBuf&) = delete;
  DevBuf& operator=(const DevBuf&) = delete;
  ~DevBuf() { reset(); }
  void reset() {
    if (p) cudaFree(p);
    p = nullptr;
    bytes = 0;
  }
  cudaError_t alloc(size_t n) {
    reset();
    if (n == 0) n = 16;
    cudaError_t e = cudaMalloc(&p, n);
    if (e == cudaSuccess) bytes = n;
    else p = nullptr;
    return e;
  }
  template <class T>
  T* as() const { return static_cast<T*>(p); }
};

template <class T>
cudaError_t upload(DevBuf& b, const std::vector<T>& v) {
  cudaError_t e = b.alloc(v.size() * sizeof(T));
  if (e != cudaSuccess || v.empty()) return e;
  return cudaMemcpy(b.p, v.data(), v.size() * sizeof(T), cudaMemcpyHostToDevice);
}

// ------------------------------------------------------------------ counters, profiling

struct Counters {
  int64_t steps = 0, ns_calls_last = 0, muon_mats_last = 0, launches_last = 0, launches_total = 0;
};
Counters g_cnt;
std::mutex g_mu;

// Cross-check settings (muon_testing_set): plans built while they differ
// from the defaults run other kernels or schedules.
struct TestKnobs {
  int gemm = 0;         // 0 product path, 1 CUDA-core GEMM everywhere, 2 no SM pairs
  int stack = 1;        // 0: one NS problem per block
  int flow = 1;         // 0: one pair launch per product
  int flow_lag = 0;     // pair task wavefront lag (0: half the problems)
  int flow_waves = 1;   // pair task order by groups of problems
  int raster = 0;       // 0: default column groups; 1: row-major; k >= 2: groups of k column tiles
  int extent_shrink = 0; // debug builds: the storage extent the checks use, made this much smaller
};
TestKnobs g_knobs;

struct PendingEvent {
  int phase;
  cudaEvent_t start, stop;
  double bytes, flops;
};
uint32_t g_profile = 0;   // phases (bit 1 << muon_phase_t) whose launches are timed
std::vector<PendingEvent> g_pending;
std::vector<cudaEvent_t> g_event_pool;
muon_phase_time_t g_phase[MUON_PHASE_COUNT];

cudaEvent_t get_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Records a profiling event on s.  While s is being captured into a CUDA
// graph the record becomes an event node of the graph (external record),
// so every replay of the graph times the phase again.
void record_event(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) == cudaSuccess && st == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    cudaEventRecord(e, s);
}

const char* const kPhaseNames[MUON_PHASE_COUNT] = {
    "muon:accumulate", "muon:reduce", "muon:gather", "muon:ns_gemm", "muon:norm", "muon:scatter"};

// Brackets one launch group with events (when profiling), an NVTX range
// and counts kernels.
struct PhaseScope {
  int phase, kernels;
  double bytes, flops;
  cudaStream_t s;
  NvtxRange range_;
  cudaEvent_t a = nullptr, b = nullptr;
  PhaseScope(int ph, cudaStream_t st, int nkern, double by, double fl)
      : phase(ph), kernels(nkern), bytes(by), flops(fl), s(st), range_(kPhaseNames[ph]) {
    if ((g_profile >> ph & 1u) && nkern > 0) {
      a = get_event();
      b = get_event();
      record_event(a, s);
    }
  }
  ~PhaseScope() {
    g_cnt.launches_last += kernels;
    g_cnt.launches_total += kernels;
    if (a) {
      record_event(b, s);
      g_pending.push_back({phase, a, b, bytes, flops});
      g_phase[phase].launches += kernels;
    }
  }
};

// ------------------------------------------------------------------ layout (table plan)

struct Layout {
  std::vector<Owner> owners;
  std::vector<Segment> segs;
  std::vector<RTile> rtiles;
  std::vector<ETile> gtiles;   // gather: Muon owners
  std::vector<ETile> stiles;   // scatter: all owners
  std::vector<YTile> ytiles;
  std::vector<Run> runs;       // accumulate: every parameter element
  int n_muon_params = 0;
  int n_muon_owners = 0;
  int64_t muon_elems = 0, aux_elems = 0;
  int64_t x_elems = 0, sq_elems = 0;   // per workspace region
  int64_t storage_extent = 0;          // storage elements the partitions describe
};

int validate_and_build(const muon_param_t* params, int nparams, const muon_partition_t* parts,
                       int nparts, Layout& L) {
  if (nparams < 0 || nparts < 0) return fail(MUON_ERR_INVALID, "negative table size");
  if (nparams > 0 && !params) return fail(MUON_ERR_INVALID, "params is NULL");
  if (nparts > 0 && !parts) return fail(MUON_ERR_INVALID, "parts is NULL");
  if (nparams > 0 && nparts == 0) return fail(MUON_ERR_INVALID, "parameters but no partitions");
  for (int i = 0; i < nparts; ++i) {
    const muon_partition_t& q = parts[i];
    if (q.flat_begin < 0 || q.flat_end < q.flat_begin || q.storage_offset < 0)
      return fail(MUON_ERR_INVALID, "partition " + std::to_string(i) + " has a bad range");
    if (i > 0 && parts[i - 1].flat_end > q.flat_begin)
      return fail(MUON_ERR_INVALID,
                  "partitions must be sorted by flat_begin and must not overlap (at " +
                      std::to_string(i) + ")");
  }
  {  // storage ranges must not overlap
    std::vector<std::pair<int64_t, int64_t>> st;
    for (int i = 0; i < nparts; ++i)
      if (parts[i].flat_end > parts[i].flat_begin)
        st.push_back({parts[i].storage_offset,
                      parts[i].storage_offset + parts[i].flat_end - parts[i].flat_begin});
    std::sort(st.begin(), st.end());
    for (size_t i = 1; i < st.size(); ++i)
      if (st[i - 1].second > st[i].first)
        return fail(MUON_ERR_INVALID, "partitions overlap in storage");
  }
  for (int i = 0; i < nparts; ++i)
    L.storage_extent = std::max(L.storage_extent,
                                parts[i].storage_offset + parts[i].flat_end - parts[i].flat_begin);
  std::vector<std::pair<int64_t, int64_t>> pr;
  for (int i = 0; i < nparams; ++i) {
    const muon_param_t& p = params[i];
    if (p.rows < 1 || p.cols < 1)
      return fail(MUON_ERR_INVALID, "parameter " + std::to_string(i) + " has rows or cols < 1");
    if (p.offset < 0) return fail(MUON_ERR_INVALID, "parameter " + std::to_string(i) + " offset < 0");
    if (p.num_heads < 0)
      return fail(MUON_ERR_INVALID, "parameter " + std::to_string(i) + " num_heads < 0");
    if (p.use_muon && p.num_heads > 1 && p.rows % p.num_heads != 0)
      return fail(MUON_ERR_INVALID,
                  "parameter " + std::to_string(i) + ": rows not a multiple of num_heads");
    pr.push_back({p.offset, p.offset + int64_t(p.rows) * p.cols});
  }
  std::sort(pr.begin(), pr.end());
  for (size_t i = 1; i < pr.size(); ++i)
    if (pr[i - 1].second > pr[i].first) return fail(MUON_ERR_INVALID, "parameters overlap");

  auto first_part = [&](int64_t flat) {   // first partition with flat_end > flat
    int lo = 0, hi = nparts;
    while (lo < hi) {
      int mid = (lo + hi) / 2;
      if (parts[mid].flat_end > flat) hi = mid; else lo = mid + 1;
    }
    return lo;
  };
  // segments of [fb, fb + n) -> appended to L.segs; returns false if not covered
  auto add_segments = [&](int64_t fb, int64_t n, Owner& o) {
    o.seg_begin = static_cast<int32_t>(L.segs.size());
    int64_t covered = 0, cursor = fb;
    for (int j = first_part(fb); j < nparts && parts[j].flat_begin < fb + n; ++j) {
      const int64_t lo = std::max(fb, parts[j].flat_begin);
      const int64_t hi = std::min(fb + n, parts[j].flat_end);
      if (lo >= hi) continue;
      if (lo != cursor) return false;   // a hole between partitions
      L.segs.push_back({lo - fb, parts[j].storage_offset + (lo - parts[j].flat_begin), hi - lo});
      covered += hi - lo;
      cursor = hi;
    }
    o.seg_count = static_cast<int32_t>(L.segs.size()) - o.seg_begin;
    return covered == n;
  };

  for (int i = 0; i < nparams; ++i) {
    const muon_param_t& p = params[i];
    const int h = (p.use_muon && p.num_heads > 1) ? p.num_heads : 1;
    const int br = p.rows / h;
    if (p.use_muon) ++L.n_muon_params;
    for (int b = 0; b < h; ++b) {
      Owner o{};
      o.flat_begin = p.offset + int64_t(b) * br * p.cols;
      o.is_muon = p.use_muon ? 1 : 0;
      o.rows = p.use_muon ? br : p.rows;
      o.cols = p.cols;
      o.numel = int64_t(o.rows) * o.cols;
      o.transposed = (o.is_muon && o.rows > o.cols) ? 1 : 0;
      o.m = std::min(o.rows, o.cols);
      o.n = std::max(o.rows, o.cols);
      if (!add_segments(o.flat_begin, o.numel, o))
        return fail(MUON_ERR_INVALID,
                    "parameter " + std::to_string(i) + " is not covered by the partitions");
      if (o.is_muon) {
        o.ldx = static_cast<int32_t>(round_up(o.n, 8));
        o.ldm = static_cast<int32_t>(round_up(o.m, 8));
        L.muon_elems += o.numel;
        ++L.n_muon_owners;
      } else {
        L.aux_elems += o.numel;
      }
      L.owners.push_back(o);
    }
  }

  // Newton-Schulz problems stack runs of consecutive Muon blocks of one
  // shape (ns_blocks).  A table that interleaves shapes (many small matrices
  // of mixed sizes) stacks far better with its Muon blocks ordered by shape,
  // so that order is taken when it gives fewer problems at the single-SM
  // stack cap; otherwise (GPT-2's head blocks already run together) the
  // table order stays.  The order depends on the parameters alone, so it is
  // the same for every partitioning.
  {
    auto problems_at_128 = [](const std::vector<Owner>& v) {
      int64_t n = 0;
      int run_m = 0, run_n = 0, run_rows = 0;
      bool prev_muon = false;
      for (const Owner& o : v) {
        if (!o.is_muon) { prev_muon = false; continue; }
        const bool join = prev_muon && o.m % 32 == 0 && 2 * o.m <= 128 && o.m == run_m &&
                          o.n == run_n && run_rows + o.m <= 128;
        if (join) {
          run_rows += o.m;
        } else {
          ++n;
          run_m = o.m;
          run_n = o.n;
          run_rows = o.m;
        }
        prev_muon = true;
      }
      return n;
    };
    std::vector<Owner> by_shape = L.owners;
    std::stable_sort(by_shape.begin(), by_shape.end(), [](const Owner& x, const Owner& y) {
      if (x.is_muon != y.is_muon) return x.is_muon > y.is_muon;
      if (!x.is_muon) return false;
      if (x.m != y.m) return x.m < y.m;
      return x.n < y.n;
    });
    if (problems_at_128(by_shape) < problems_at_128(L.owners)) L.owners.swap(by_shape);
  }
  for (Owner& o : L.owners)
    if (o.is_muon) {
      o.x_off = L.x_elems;
      o.sq_off = L.sq_elems;
      L.x_elems += round_up(int64_t(o.m) * o.ldx, 64);
      L.sq_elems += round_up(int64_t(o.m) * o.ldm, 64);
    }

  // A tile qualifies for the kernels' 16-byte path when it lies in one
  // segment with 16-byte aligned storage (see ETile).
  auto mark_fast = [&](ETile& t, const Owner& o) {
    int64_t a, b;
    bool shape_ok;
    if (t.kind == 0) {
      a = int64_t(t.r0) * o.cols;
      b = int64_t(t.r0 + t.nr) * o.cols;
      shape_ok = o.cols % 4 == 0 && o.ldx == o.cols;
    } else if (t.kind == 1 || t.kind == 3) {
      const int re = std::min(t.r0 + kTT, o.rows), w = t.kind == 3 ? 2 * kTT : kTT;
      a = int64_t(t.r0) * o.cols + t.c0;
      b = int64_t(re - 1) * o.cols + t.c0 + w;
      shape_ok = o.cols % 4 == 0 && t.c0 + w <= o.cols;
    } else {
      a = t.rel_begin;
      b = t.rel_begin + t.len;
      shape_ok = t.rel_begin % 4 == 0 && t.len % 4 == 0;
    }
    if (!shape_ok) return;
    for (int k = o.seg_begin; k < o.seg_begin + o.seg_count; ++k) {
      const Segment& sg = L.segs[k];
      if (a < sg.rel_begin || a >= sg.rel_begin + sg.len) continue;
      const int64_t delta = sg.storage_begin - sg.rel_begin;
      if (b <= sg.rel_begin + sg.len && ((delta + a) & 3) == 0) {
        t.fast = 1;
        t.sdelta = delta;
      }
      return;
    }
  };

  // tiles
  for (int oi = 0; oi < static_cast<int>(L.owners.size()); ++oi) {
    Owner& o = L.owners[oi];
    o.rtile_begin = static_cast<int32_t>(L.rtiles.size());
    for (int64_t r = 0; r < o.numel; r += kReduceTile)
    {
      RTile rt{};
      rt.owner = oi;
      rt.len = static_cast<int32_t>(std::min<int64_t>(kReduceTile, o.numel - r));
      rt.rel_begin = r;
      for (int k = o.seg_begin; k < o.seg_begin + o.seg_count; ++k) {
        const Segment& sg = L.segs[k];
        if (r < sg.rel_begin || r >= sg.rel_begin + sg.len) continue;
        const int64_t delta = sg.storage_begin - sg.rel_begin;
        if (r + rt.len <= sg.rel_begin + sg.len && rt.len % 4 == 0 && ((delta + r) & 3) == 0) {
          rt.fast = 1;
          rt.sdelta = delta;
        }
        break;
      }
      L.rtiles.push_back(rt);
    }
    o.rtile_count = static_cast<int32_t>(L.rtiles.size()) - o.rtile_begin;
    if (o.is_muon) {
      if (!o.transposed) {
        const int rows_per = std::max<int>(1, kRowTile / o.cols);
        for (int r = 0; r < o.rows; r += rows_per) {
          ETile t{};
          t.owner = oi; t.kind = 0; t.r0 = r; t.nr = std::min(rows_per, o.rows - r);
          mark_fast(t, o);
          L.gtiles.push_back(t);
          L.stiles.push_back(t);
        }
      } else {
        for (int r = 0; r < o.rows; r += kTT)
          for (int c = 0; c < o.cols; c += kTT) {
            ETile t{};
            t.owner = oi; t.kind = 1; t.r0 = r; t.c0 = c;
            mark_fast(t, o);
            L.stiles.push_back(t);
          }
        // the gather reads 128-column row pieces where it can (each folded
        // bf16 micro-batch then arrives in 256-byte runs)
        for (int r = 0; r < o.rows; r += kTT)
          for (int c = 0; c < o.cols;) {
            ETile t{};
            t.owner = oi; t.kind = 3; t.r0 = r; t.c0 = c;
            mark_fast(t, o);
            if (t.fast) {
              L.gtiles.push_back(t);
              c += 2 * kTT;
              continue;
            }
            t = ETile{};
            t.owner = oi; t.kind = 1; t.r0 = r; t.c0 = c;
            mark_fast(t, o);
            L.gtiles.push_back(t);
            c += kTT;
          }
      }
      o.ytile_begin = static_cast<int32_t>(L.ytiles.size());
      const int yrows = std::max<int>(1, kRowTile / o.n);
      for (int r = 0; r < o.m; r += yrows)
        L.ytiles.push_back({oi, r, std::min(yrows, o.m - r), 0});
      o.ytile_count = static_cast<int32_t>(L.ytiles.size()) - o.ytile_begin;
    } else {
      for (int64_t r = 0; r < o.numel; r += kRowTile) {
        ETile t{};
        t.owner = oi; t.kind = 2; t.rel_begin = r;
        t.len = std::min<int64_t>(kRowTile, o.numel - r);
        mark_fast(t, o);
        L.stiles.push_back(t);
      }
    }
    for (int s = 0; s < o.seg_count; ++s) {
      const Segment& sg = L.segs[o.seg_begin + s];
      for (int64_t r = 0; r < sg.len; r += 32768)
        L.runs.push_back({sg.storage_begin + r, std::min<int64_t>(32768, sg.len - r)});
    }
  }
  return MUON_OK;
}

// ------------------------------------------------------------------ NS plan

enum Engine { ENGINE_TC = 0, ENGINE_SIMT = 1, ENGINE_CONVERT = 2, ENGINE_X3 = 3, ENGINE_TC2 = 4 };

// One launch of the NS iteration: a grouped GEMM over every block, or (for
// ENGINE_CONVERT) the fp32 -> bf16 rounding of a whole workspace region.
struct GemmPhase {
  int engine = ENGINE_SIMT;
  int ab_es = 4;   // A/B operand bytes for the CUDA-core engine
  std::vector<GemmProblem> probs;
  std::vector<GemmTile> tiles;
  int program = -1;            // pair engine: the task program this phase belongs to
  bool program_head = false;   // its first phase: the one launch of the program
  DevBuf d_probs, d_maps, d_tiles;
  double flops = 0.0;   // algorithmic (full products)
  const float* conv_src = nullptr;
  void* conv_dst = nullptr;
  int64_t conv_n = 0;
};

struct PairProgram {
  int first_phase = 0, nphases = 0;
  std::vector<GemmProblem> probs;
  std::vector<PairTask> tasks;
  int ncounters = 1;
  double flops = 0.0;
  DevBuf d_probs, d_maps, d_tasks, d_counters;
};

// Tile ranges of one wave of a bounded-workspace plan (owner order).
struct WaveRange {
  int g0, g1;   // gather tiles
  int s0, s1;   // scatter tiles
  int y0, y1;   // update tiles
  double elems; // Muon elements of the wave
};

struct NsPlan {
  int esize = 2;       // X0 / Y element format: 2 bf16, 4 fp32, 6 split-3
  int64_t x_ps = 0;    // split-3: elements between the planes of an X region
  int64_t x_elems = 0; // elements of one X region
  bool use_tc = false;
  int method = 0, steps = 5;
  DevBuf ws;
  void* x0 = nullptr;
  void* y = nullptr;
  std::vector<std::unique_ptr<GemmPhase>> phases;
  double flops = 0.0;
  // Bounded workspace: the Muon owners run in waves that share `ws`; each
  // wave is a plan of its own over owners whose x_off / sq_off are relative
  // to the wave (the owner table with those offsets is d_owners).
  std::vector<std::unique_ptr<NsPlan>> waves;
  std::vector<WaveRange> ranges;
  DevBuf d_owners;
  // Sums of squares of the update, written by the last product's epilogue
  // (per tile and epilogue warp, problems in owner order; null when the
  // last product runs on the CUDA cores)
  DevBuf ssq;
  double* ssq_ptr = nullptr;
  int64_t n_ssq = 0;
  std::vector<std::unique_ptr<PairProgram>> programs;
};

void engine_tile(int engine, int& bm, int& bn) {
  bm = bn = kSimtTile;
  if (engine == ENGINE_TC) { bm = kTcBM; bn = kTcBN; }
  if (engine == ENGINE_TC2) { bm = kTcPairBM; bn = kTcPairBN; }
  if (engine == ENGINE_X3) { bm = kX3BM; bn = kX3BN; }
}

// Slots of the fused sums of squares for problems of m x n outputs.
int64_t ssq_slots(int engine, int m, int n) {
  int bm, bn;
  engine_tile(engine, bm, bn);
  return int64_t((m + bm - 1) / bm) * ((n + bn - 1) / bn) * kSsqSlots;
}

// Adds one GEMM D = alpha A op(B) + beta E + gamma I (per block) to a phase.
struct PhaseBuilder {
  GemmPhase* ph;
  // useful: the fraction of the product's 2 M N K flops that is algorithmic
  // work (stacked blocks: rows per block / stacked rows)
  void add(const GemmProblem& p, double useful = 1.0) {
    int bm, bn;
    engine_tile(ph->engine, bm, bn);
    const int idx = static_cast<int>(ph->probs.size());
    ph->probs.push_back(p);
    const int tm_n = (p.M + bm - 1) / bm, tn_n = (p.N + bn - 1) / bn;
    for (int tm = 0; tm < tm_n; ++tm)
      for (int tn = 0; tn < tn_n; ++tn) {
        if (p.symmetric && tn * bn + bn - 1 < tm * bm) continue;   // strictly lower tile
        ph->tiles.push_back({idx, tm, tn});
      }
    ph->flops += 2.0 * p.M * double(p.N) * p.K * useful;
  }
};

int finish_phase(GemmPhase& ph) {
  if (ph.engine == ENGINE_CONVERT || ph.engine == ENGINE_TC2) return MUON_OK;   // see PairProgram
  // heavy tiles first (K descending) for the static round-robin schedule
  std::stable_sort(ph.tiles.begin(), ph.tiles.end(), [&](const GemmTile& a, const GemmTile& b) {
    return ph.probs[a.problem].K > ph.probs[b.problem].K;
  });
  MUON_CUDA_TRY(upload(ph.d_probs, ph.probs));
  MUON_CUDA_TRY(upload(ph.d_tiles, ph.tiles));
  if (ph.engine == ENGINE_TC || ph.engine == ENGINE_X3) {
    std::vector<TcMaps> maps(ph.probs.size());
    for (size_t i = 0; i < ph.probs.size(); ++i) {
      const bool ok = ph.engine == ENGINE_TC ? tc_encode_maps(ph.probs[i], &maps[i])
                                             : x3_encode_maps(ph.probs[i], &maps[i]);
      if (!ok) return fail(MUON_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    }
    MUON_CUDA_TRY(upload(ph.d_maps, maps));
  }
  return MUON_OK;
}

// Consecutive pair-engine phases of a plan run as one task program: the
// problems of all its phases in one array, one task per output tile, and
// for every phase after the first, each tile of NS problem j waits for the
// tiles of problem j's previous product (every epilogue warp of both CTAs
// of each adds one to its counter).  Tasks are ordered wave by wave (groups of consecutive
// problems), phase by phase inside a wave, heavy tiles first inside a
// (wave, phase), so a wave's operands tend to stay in L2 from one product
// to the next while the other waves fill the gaps.

constexpr int kRasterCols = 4;        // column tiles per raster group (1024 columns)
constexpr int kRasterMinTiles = 128;  // products with fewer tiles keep row-major order

int build_pair_program(std::vector<std::unique_ptr<GemmPhase>>& phases, int a, int b,
                       int waves, PairProgram& G) {
  G.first_phase = a;
  G.nphases = b - a;
  const int np = static_cast<int>(phases[a]->probs.size());
  for (int k = a; k < b; ++k)
    if (static_cast<int>(phases[k]->probs.size()) != np)
      return fail(MUON_ERR_INVALID, "internal: pair phases of unequal problem counts");
  // tiles of (phase, problem)
  std::vector<std::vector<std::vector<GemmTile>>> tl(b - a, std::vector<std::vector<GemmTile>>(np));
  for (int k = a; k < b; ++k) {
    for (const GemmTile& t : phases[k]->tiles) tl[k - a][t.problem].push_back(t);
    for (const GemmProblem& q : phases[k]->probs) G.probs.push_back(q);
    G.flops += phases[k]->flops;
  }
  // Products with an MN-major B (X' = B X + a X, Y = Q X0) and many tiles
  // run their tiles in groups of kRasterCols column tiles, every row of a
  // group before the next group: the concurrent tiles then share the m x m
  // operand (small enough to stay in L2) and one column panel of X, so X is
  // read from DRAM about once.  In row-major order every row of tiles
  // streams the whole of X again (for a 4096 x 14336 X, 117 MB, next to a
  // 129 MB L2).
  const int group = g_knobs.raster == 0 ? kRasterCols : g_knobs.raster;   // 1: row-major
  if (group > 1)
    for (int k = 0; k < b - a; ++k)
      for (int j = 0; j < np; ++j) {
        std::vector<GemmTile>& v = tl[k][j];
        if (phases[a + k]->probs[j].b_kmajor != 0 || static_cast<int>(v.size()) < kRasterMinTiles)
          continue;
        std::stable_sort(v.begin(), v.end(), [group](const GemmTile& x, const GemmTile& y) {
          if (x.tn / group != y.tn / group) return x.tn / group < y.tn / group;
          if (x.tm != y.tm) return x.tm < y.tm;
          return x.tn < y.tn;
        });
      }
  auto counter = [&](int k, int j) { return 1 + k * np + j; };
  G.ncounters = 1 + (b - a) * np;
  waves = std::max(1, std::min(waves, np));
  // Units (product k, problem j) in wavefront order: unit (k, j) has key
  // j + k * lag, ties by k; lag >= np is product-major.  A unit always
  // follows the previous product of its problem, so dependencies point
  // backwards; a small lag keeps a problem's products close together (its
  // operands stay in L2) but leaves less slack before each dependency.
  // (GPT-2-small, 120 problems: lag 4 / 8 / 16 / 32 / 64 / product-major
  // gave 1.274 / 1.194 / 1.145 / 1.135 / 1.134 / 1.158 ms per iteration)
  const int lag = g_knobs.flow_lag > 0 ? g_knobs.flow_lag : std::max(1, np / 2);
  auto make_tasks = [&](int k, int j, std::vector<PairTask>& out) {
    const GemmProblem& q = phases[a + k]->probs[j];
    for (const GemmTile& t : tl[k][j]) {
      PairTask pt{};
      pt.problem = k * np + j;
      pt.tm = t.tm;
      pt.tn = t.tn;
      pt.dep = k > 0 ? counter(k - 1, j) : -1;
      pt.dep_target = k > 0 ? kPairArrivals * static_cast<int>(tl[k - 1][j].size()) : 0;
      pt.done = k + 1 < b - a ? counter(k, j) : -1;
      pt.nk = (q.K + kTcBK - 1) / kTcBK;
      pt.b_kmajor = q.b_kmajor;
      out.push_back(pt);
    }
  };
  auto heavy_first = [&](std::vector<PairTask>& group) {
    std::stable_sort(group.begin(), group.end(), [&](const PairTask& x, const PairTask& y) {
      return G.probs[x.problem].K > G.probs[y.problem].K;
    });
  };
  if (lag >= np) {
    for (int w = 0; w < waves; ++w) {
      const int j0 = int(int64_t(np) * w / waves), j1 = int(int64_t(np) * (w + 1) / waves);
      for (int k = 0; k < b - a; ++k) {
        std::vector<PairTask> group;
        for (int j = j0; j < j1; ++j) make_tasks(k, j, group);
        heavy_first(group);
        G.tasks.insert(G.tasks.end(), group.begin(), group.end());
      }
    }
  } else {
    // group the units of one key together, heavy tiles first within it
    const int nk_prod = b - a;
    const int64_t max_key = int64_t(np - 1) + int64_t(nk_prod - 1) * lag;
    for (int64_t key = 0; key <= max_key; ++key) {
      std::vector<PairTask> group;
      for (int k = 0; k < nk_prod; ++k) {
        const int64_t j = key - int64_t(k) * lag;
        if (j >= 0 && j < np) make_tasks(k, static_cast<int>(j), group);
      }
      heavy_first(group);
      G.tasks.insert(G.tasks.end(), group.begin(), group.end());
    }
  }
  std::vector<TcMaps> maps(G.probs.size());
  for (size_t i = 0; i < G.probs.size(); ++i)
    if (!tc2_encode_maps(G.probs[i], &maps[i])) return fail(MUON_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  MUON_CUDA_TRY(upload(G.d_probs, G.probs));
  MUON_CUDA_TRY(upload(G.d_maps, maps));
  MUON_CUDA_TRY(upload(G.d_tasks, G.tasks));
  MUON_CUDA_TRY(G.d_counters.alloc(sizeof(int) * G.ncounters));
  return MUON_OK;
}

// A matrix in a workspace region: element format (2 bf16, 4 fp32, 6
// split-3), plane stride, leading dimension.
struct WsMat {
  char* p;
  int es;
  int64_t ps;
  int64_t ld;
};

// Work lists of the NS iteration over every Muon block (owner), laid out in
// per-owner slices of the workspace regions (x_off for m x n, sq_off for
// m x m).
//
// standard: per step A = X X^T (symmetric: upper tiles, mirrored),
//   B = c A A + b A (symmetric), X' = B X + a X, ping-ponging X.  The
//   oracle's A and B are exactly symmetric too (bf16 products summed in
//   float64 are exact), so mirroring changes no value.
// gram: R0 = X0 X0^T (symmetric), then the m x m recurrence
//   P = c R R + b R + a I, Q <- P Q, T = P R, R = T P in FP32 with B read
//   MN-major, upper tiles mirrored (each product is symmetric in exact
//   arithmetic); then Y = bf16(Q) X0 (BF16 mode) or Q X0 (FP32 mode).
// Engines: BF16 operands on the tensor cores, on SM pairs with 256 x 256
// tiles (ENGINE_TC2) when every block has at least 192 rows, else on single
// SMs with 128 x 256 tiles (ENGINE_TC; the MUON_TEST_GEMM cross-check can
// force it); FP32 operands on the tensor cores through split-3 planes
// (ENGINE_X3); the CUDA-core cross-check runs everything on the CUDA-core
// kernel with plain bf16 / fp32 storage.
// Element formats and region counts of a plan: X regions (m x n) in xe,
// the m x m regions in se, nsq of them, and a bf16 copy of Q for the
// CUDA-core gram path.
struct NsFormats {
  bool tc = false;
  int xe = 2, fe = 4, se = 2, nsq = 2;
  bool need_qbf = false;
  static size_t bytes_of(int es) { return size_t(es == 6 ? 6 : es); }
  size_t ws_bytes(int64_t x_elems, int64_t sq_elems) const {
    size_t b = 2 * bytes_of(xe) * size_t(x_elems) + nsq * bytes_of(se) * size_t(sq_elems);
    if (need_qbf) b += 2 * size_t(sq_elems);
    return b;
  }
};

// Element formats of a plan given whether the tensor-core kernels run.
void ns_formats_for(bool tc, int method, int mode, NsFormats& f) {
  const bool bf16 = mode == MUON_OPERANDS_BF16;
  f.tc = tc;
  f.xe = bf16 ? 2 : (f.tc ? 6 : 4);
  f.fe = f.tc ? 6 : 4;
  f.se = method == MUON_NS_STANDARD ? f.xe : f.fe;
  f.nsq = method == MUON_NS_STANDARD ? 2 : 5;
  f.need_qbf = method == MUON_NS_GRAM && bf16 && !f.tc;
}

int ns_formats(int method, int mode, NsFormats& f) {
  const bool bf16 = mode == MUON_OPERANDS_BF16;
  const bool force_simt = g_knobs.gemm == 1;
  const bool tc = !force_simt && tc_available();
  if (bf16 && !tc && !force_simt)
    return fail(MUON_ERR_UNSUPPORTED, "BF16 operand mode needs an sm_103 (GB300) GPU");
  ns_formats_for(tc, method, mode, f);
  return MUON_OK;
}

// Newton-Schulz problems of a plan.  A run of consecutive Muon blocks of
// one shape whose X0 regions are adjacent is stacked into one problem of up
// to `cap` rows (the engine's row tile) when the blocks have a multiple of
// 32 rows: the Gram product of the stack (X X^T, or R = X0 X0^T) is masked
// to its block diagonal, every later product of the iteration keeps the
// zeros exactly, and each block's rows of the result are those of its own
// iteration.  Each problem gets m x m regions of its own (sq_off, ldm).
struct NsBlocks {
  std::vector<Owner> probs;                 // m = stacked rows; ns_blk = rows per block
  std::vector<std::pair<int, int>> members; // first owner index and block count
  int64_t sq_elems = 0;
  int cap = 0;
  bool pairs = false;                       // BF16 products on SM pairs
};

// The gram form stacks no further than the single-SM tile (128 rows), and
// takes SM pairs only for blocks of 192+ rows unstacked: its m x m
// recurrence runs on the split-3 kernel over each problem's whole stacked
// square, so a 256-row stack of four 64-row heads costs 16 times the
// recurrence flops and 4 times its bytes of the heads alone (GPT-2-small,
// gram, BF16: NS 3.11 ms with 256-row stacks on pairs, 2.91 ms unstacked),
// while the ragged set's stacks of 32- and 64-row blocks into 128 gain 3%.
// force_cap >= 0 (the waves of a bounded plan) repeats the unbounded plan's
// choice, force_pairs included.
NsBlocks ns_blocks(const std::vector<Owner>& owners, bool tc, bool bf16, bool gram, int force_cap,
                   bool force_pairs) {
  const bool allow_pairs = tc && bf16 && g_knobs.gemm != 2;
  const bool stack = g_knobs.stack != 0;
  auto group = [&](int cap) {
    NsBlocks B;
    if (!stack) cap = 0;
    B.cap = cap;
    int last = -2;
    for (int i = 0; i < static_cast<int>(owners.size()); ++i) {
      const Owner& o = owners[i];
      if (!o.is_muon) continue;
      bool extend = false;
      if (cap > 0 && last == i - 1 && o.m % 32 == 0 && 2 * o.m <= cap) {
        const Owner& prev = owners[i - 1];
        extend = prev.m == o.m && prev.n == o.n && prev.ldx == o.ldx &&
                 o.x_off == prev.x_off + int64_t(prev.m) * prev.ldx &&
                 B.probs.back().m + o.m <= cap && B.probs.back().ns_blk == o.m;
      }
      if (extend) {
        B.probs.back().m += o.m;
        B.members.back().second += 1;
      } else {
        Owner q = o;
        q.ns_blk = o.m;
        B.probs.push_back(q);
        B.members.push_back({i, 1});
      }
      last = i;
    }
    for (size_t k = 0; k < B.probs.size(); ++k) {
      Owner& q = B.probs[k];
      if (B.members[k].second == 1) q.ns_blk = 0;
      q.ldm = static_cast<int32_t>(round_up(q.m, 8));
      q.sq_off = B.sq_elems;
      B.sq_elems += round_up(int64_t(q.m) * q.ldm, 64);
    }
    return B;
  };
  if (!tc) return group(0);
  if (force_cap >= 0) {
    NsBlocks B = group(force_cap);
    B.pairs = allow_pairs && force_pairs;
    return B;
  }
  if (allow_pairs) {
    NsBlocks B = group(gram ? 0 : kTcPairBM);
    bool ok = true;
    for (const Owner& q : B.probs) ok = ok && q.m >= 192;   // a 256-row tile at least 3/4 used
    if (ok) {
      B.pairs = true;
      return B;
    }
  }
  return group(128);
}

// Builds the GEMM phases of `owners` (their x_off index an X region of
// x_elems elements; the m x m regions are laid out per NS problem).  The
// workspace is allocated unless `ext` is given, in which case the m x m
// regions hold ext_sq elements (at least the problems' need) and the
// problems are stacked with rows cap `force_cap` on the engine `force_pairs`
// names.
int build_ns_plan(const std::vector<Owner>& owners, int64_t x_elems, int method, int mode,
                  int steps, NsPlan& P, char* ext = nullptr, int64_t ext_sq = 0,
                  int force_cap = -1, double* ext_ssq = nullptr, bool force_pairs = false) {
  const bool bf16 = mode == MUON_OPERANDS_BF16;
  NsFormats F;
  int rc0 = ns_formats(method, mode, F);
  if (rc0 != MUON_OK) return rc0;
  P.use_tc = F.tc;
  const bool tc = F.tc;
  const int xe = F.xe, fe = F.fe, se = F.se, nsq = F.nsq;
  const bool need_qbf = F.need_qbf;
  auto bytes_of = NsFormats::bytes_of;
  auto eb = [](int es) { return int64_t(es == 6 ? 2 : es); };
  const NsBlocks NB = ns_blocks(owners, tc, bf16, method == MUON_NS_GRAM, force_cap, force_pairs);
  const std::vector<Owner>& probs = NB.probs;
  int64_t sq_elems = NB.sq_elems;
  if (ext) {
    if (ext_sq < sq_elems) return fail(MUON_ERR_INVALID, "internal: wave workspace too small");
    sq_elems = ext_sq;
  }
  P.esize = xe;
  P.x_ps = xe == 6 ? x_elems : 0;
  P.method = method;
  P.steps = steps;
  char* base = ext;
  if (!base) {
    MUON_CUDA_TRY(P.ws.alloc(F.ws_bytes(x_elems, sq_elems) + 256));
    base = P.ws.as<char>();
  }
  char* X[2] = {base, base + bytes_of(xe) * x_elems};
  char* sq_base = base + 2 * bytes_of(xe) * x_elems;
  char* S[5];
  for (int i = 0; i < nsq; ++i) S[i] = sq_base + i * bytes_of(se) * size_t(sq_elems);
  char* Qbf = sq_base + nsq * bytes_of(se) * size_t(sq_elems);
  P.x0 = X[0];
  P.x_elems = x_elems;
  const float a = kNsA, b = kNsB, c = kNsC;

  auto xm = [&](char* r, const Owner& o) {
    return WsMat{r + eb(xe) * o.x_off, xe, xe == 6 ? x_elems : 0, o.ldx};
  };
  auto sm = [&](char* r, const Owner& o, int es) {
    return WsMat{r + eb(es) * o.sq_off, es, es == 6 ? sq_elems : 0, o.ldm};
  };
  const WsMat none{nullptr, 2, 0, 0};
  auto mk = [&](WsMat A, WsMat B, int bk, WsMat D, WsMat E, int M, int N, int K, int sym, float al,
                float be, float ga) {
    GemmProblem p{};
    p.A = A.p; p.B = B.p; p.D = D.p; p.E = E.p;
    p.lda = A.ld; p.ldb = B.ld; p.ldd = D.ld; p.lde = E.ld;
    p.a_ps = A.ps; p.b_ps = B.ps; p.d_ps = D.ps; p.e_ps = E.ps;
    p.M = M; p.N = N; p.K = K;
    p.b_kmajor = bk; p.symmetric = sym;
    p.alpha = al; p.beta = be; p.gamma = ga;
    p.d_es = D.es; p.e_es = E.p ? E.es : D.es;
    return p;
  };
  auto new_phase = [&](int engine, int ab_es) {
    P.phases.emplace_back(new GemmPhase());
    P.phases.back()->engine = engine;
    P.phases.back()->ab_es = ab_es;
    return PhaseBuilder{P.phases.back().get()};
  };
  // engine for products whose operands have format es
  const int bf16_engine = NB.pairs ? ENGINE_TC2 : ENGINE_TC;
  auto fs = [](const Owner& o) { return o.ns_blk ? double(o.ns_blk) / o.m : 1.0; };
  // Gram products of stacked blocks are masked to the block diagonal
  auto gram = [](GemmProblem p, const Owner& o) {
    p.blk = o.ns_blk;
    return p;
  };
  auto engine_for = [&](int es) { return !tc ? ENGINE_SIMT : (es == 2 ? bf16_engine : ENGINE_X3); };

  if (method == MUON_NS_STANDARD) {
    const int eng = engine_for(xe);
    for (int st = 0; st < steps; ++st) {
      char* src = X[st & 1];
      char* dst = X[(st + 1) & 1];
      PhaseBuilder g = new_phase(eng, xe);   // A = X X^T
      for (const Owner& o : probs)
        if (o.is_muon)
          g.add(gram(mk(xm(src, o), xm(src, o), 1, sm(S[0], o, se), none, o.m, o.m, o.n, 1, 1.f, 0.f,
                        0.f), o), fs(o));
      // B = c A A + b A.  On single SMs every tile is computed: with the
      // addend in flight that epilogue has no buffer to stage a mirror, and
      // scattered mirror stores cost more than the lower tiles.  The pair
      // engine mirrors through a buffer of its own.
      const int q_sym = eng == ENGINE_TC ? 0 : 1;
      PhaseBuilder q = new_phase(eng, xe);
      for (const Owner& o : probs)
        if (o.is_muon)
          q.add(mk(sm(S[0], o, se), sm(S[0], o, se), 1, sm(S[1], o, se), sm(S[0], o, se), o.m, o.m,
                   o.m, q_sym, c, b, 0.f), fs(o));
      PhaseBuilder u = new_phase(eng, xe);   // X' = B X + a X
      for (const Owner& o : probs)
        if (o.is_muon)
          u.add(mk(sm(S[1], o, se), xm(src, o), 0, xm(dst, o), xm(src, o), o.m, o.n, o.m, 0, 1.f, a,
                   0.f), fs(o));
    }
    P.y = X[steps & 1];
  } else {
    char *R = S[0], *Pm = S[1], *Qa = S[2], *Qb = S[3], *T = S[4];
    const int rec = tc ? ENGINE_X3 : ENGINE_SIMT;
    // R = X0 X0^T.  On single SMs (blocks below 192 rows) every tile is
    // computed: a 128-row block is one tile either way, and that kernel
    // mirrors split-3 outputs element by element, which cost more than the
    // lower tiles (ragged 8192-block step: 1.26 -> 0.41 ms for this product)
    const int r0_eng = engine_for(xe);
    const int r0_sym = r0_eng == ENGINE_TC ? 0 : 1;
    PhaseBuilder g0 = new_phase(r0_eng, xe);
    for (const Owner& o : probs)
      if (o.is_muon)
        g0.add(gram(mk(xm(X[0], o), xm(X[0], o), 1, sm(R, o, fe), none, o.m, o.m, o.n, r0_sym, 1.f,
                       0.f, 0.f), o), fs(o));
    char* Qcur = Qa;
    // Every matrix of the recurrence is a polynomial in R0 in exact
    // arithmetic, so every product (R R, P Q, P R, T P) is symmetric: only
    // tiles touching the upper triangle are computed and mirrored, which
    // halves the work on large blocks and keeps each iterate exactly
    // symmetric.
    const int rs = 1;
    for (int k = 0; k < steps; ++k) {
      char* Pk = (k == 0) ? Qa : Pm;   // Q1 = P0 (Q0 = I)
      PhaseBuilder pp = new_phase(rec, fe);   // P = c R R + b R + a I
      for (const Owner& o : probs)
        if (o.is_muon)
          pp.add(mk(sm(R, o, fe), sm(R, o, fe), 0, sm(Pk, o, fe), sm(R, o, fe), o.m, o.m, o.m, rs, c,
                    b, a), fs(o));
      // Q <- P Q and T = P R need only P: one phase, each block's two
      // products side by side so they share P's panels in L2
      const bool q_upd = k > 0, t_upd = k < steps - 1;
      char* Qn = (Qcur == Qa) ? Qb : Qa;
      {
        PhaseBuilder qt = new_phase(rec, fe);
        for (const Owner& o : probs)
          if (o.is_muon) {
            if (q_upd)
              qt.add(mk(sm(Pk, o, fe), sm(Qcur, o, fe), 0, sm(Qn, o, fe), none, o.m, o.m, o.m, rs, 1.f,
                        0.f, 0.f), fs(o));
            if (t_upd)
              qt.add(mk(sm(Pk, o, fe), sm(R, o, fe), 0, sm(T, o, fe), none, o.m, o.m, o.m, rs, 1.f,
                        0.f, 0.f), fs(o));
          }
      }
      if (q_upd) Qcur = Qn;
      if (t_upd) {
        PhaseBuilder rr = new_phase(rec, fe);   // R = T P
        for (const Owner& o : probs)
          if (o.is_muon)
            rr.add(mk(sm(T, o, fe), sm(Pk, o, fe), 0, sm(R, o, fe), none, o.m, o.m, o.m, rs, 1.f,
                      0.f, 0.f), fs(o));
      }
    }
    PhaseBuilder* yy = nullptr;
    if (bf16 && tc) {
      // bf16(Q) is exactly the hi plane of the split-3 Q
      PhaseBuilder ph = new_phase(bf16_engine, 2);
      for (const Owner& o : probs)
        if (o.is_muon) {
          WsMat q = sm(Qcur, o, fe);
          q.es = 2;
          q.ps = 0;
          ph.add(mk(q, xm(X[0], o), 0, xm(X[1], o), none, o.m, o.n, o.m, 0, 1.f, 0.f, 0.f), fs(o));
        }
      yy = nullptr;
    } else if (need_qbf) {   // CUDA-core path: round Q to bf16, then Y = Q X0
      P.phases.emplace_back(new GemmPhase());
      GemmPhase& cv = *P.phases.back();
      cv.engine = ENGINE_CONVERT;
      cv.conv_src = reinterpret_cast<const float*>(Qcur);
      cv.conv_dst = Qbf;
      cv.conv_n = sq_elems;
      PhaseBuilder ph = new_phase(ENGINE_SIMT, 2);
      for (const Owner& o : probs)
        if (o.is_muon)
          ph.add(mk(WsMat{Qbf + 2 * o.sq_off, 2, 0, o.ldm}, xm(X[0], o), 0, xm(X[1], o), none, o.m,
                    o.n, o.m, 0, 1.f, 0.f, 0.f), fs(o));
    } else {   // FP32 mode: Y = Q X0 in FP32 (split-3 or fp32)
      PhaseBuilder ph = new_phase(engine_for(xe), xe);
      for (const Owner& o : probs)
        if (o.is_muon)
          ph.add(mk(sm(Qcur, o, fe), xm(X[0], o), 0, xm(X[1], o), none, o.m, o.n, o.m, 0, 1.f, 0.f,
                    0.f), fs(o));
    }
    (void)yy;
    P.y = X[1];
  }
  // The last product's epilogue writes the sums of squares of the update,
  // problems in owner order (into ext_ssq for a wave of a bounded plan).
  if (!P.phases.empty()) {
    GemmPhase& last = *P.phases.back();
    if (last.engine == ENGINE_TC || last.engine == ENGINE_TC2 || last.engine == ENGINE_X3) {
      int64_t n = 0;
      for (const GemmProblem& q : last.probs) n += ssq_slots(last.engine, q.M, q.N);
      double* buf = ext_ssq;
      if (buf == nullptr) {
        MUON_CUDA_TRY(P.ssq.alloc(sizeof(double) * std::max<int64_t>(n, 1)));
        MUON_CUDA_TRY(cudaMemset(P.ssq.p, 0, sizeof(double) * std::max<int64_t>(n, 1)));
        buf = P.ssq.as<double>();
      }
      int64_t off = 0;
      for (GemmProblem& q : last.probs) {
        q.ssq = buf + off;
        off += ssq_slots(last.engine, q.M, q.N);
      }
      P.ssq_ptr = buf;
      P.n_ssq = n;
    }
  }
  for (auto& ph : P.phases) {
    int rc = finish_phase(*ph);
    if (rc != MUON_OK) return rc;
    P.flops += ph->flops;
  }
  // runs of consecutive pair-engine phases become task programs
  const int flow_waves = std::max(1, g_knobs.flow_waves);
  const bool flow = g_knobs.flow != 0;   // 0: a program per phase
  for (int k = 0; k < static_cast<int>(P.phases.size());) {
    if (P.phases[k]->engine != ENGINE_TC2) { ++k; continue; }
    int e = k + 1;
    while (flow && e < static_cast<int>(P.phases.size()) && P.phases[e]->engine == ENGINE_TC2) ++e;
    std::unique_ptr<PairProgram> G(new PairProgram());
    int rc = build_pair_program(P.phases, k, e, flow_waves, *G);
    if (rc != MUON_OK) return rc;
    for (int i = k; i < e; ++i) P.phases[i]->program = static_cast<int>(P.programs.size());
    P.phases[k]->program_head = true;
    P.programs.push_back(std::move(G));
    k = e;
  }
  return MUON_OK;
}

// ------------------------------------------------------------------ table plans

struct TablePlan {
  int device = -1;
  uint64_t hash = 0;
  std::vector<uint8_t> key;
  Layout L;
  DevBuf d_owners, d_segs, d_rtiles, d_gtiles, d_stiles, d_ytiles, d_runs;
  DevBuf d_rsum, d_ysum, d_fin, d_div, d_state, d_err;
  std::map<std::tuple<int, int, int, uint64_t>, std::unique_ptr<NsPlan>> ns;
};

std::vector<std::unique_ptr<TablePlan>> g_plans;

uint64_t fnv1a(const void* data, size_t n, uint64_t h = 1469598103934665603ull) {
  const uint8_t* p = static_cast<const uint8_t*>(data);
  for (size_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= 1099511628211ull;
  }
  return h;
}

int get_table_plan(const muon_param_t* params, int nparams, const muon_partition_t* parts,
                   int nparts, TablePlan** out) {
  if (nparams < 0 || nparts < 0) return fail(MUON_ERR_INVALID, "negative table size");
  if ((nparams > 0 && !params) || (nparts > 0 && !parts))
    return fail(MUON_ERR_INVALID, "table pointer is NULL");
  std::vector<uint8_t> key(sizeof(int) * 2 + sizeof(muon_param_t) * nparams +
                           sizeof(muon_partition_t) * nparts);
  std::memcpy(key.data(), &nparams, sizeof(int));
  std::memcpy(key.data() + sizeof(int), &nparts, sizeof(int));
  if (nparams) std::memcpy(key.data() + 2 * sizeof(int), params, sizeof(muon_param_t) * nparams);
  if (nparts)
    std::memcpy(key.data() + 2 * sizeof(int) + sizeof(muon_param_t) * nparams, parts,
                sizeof(muon_partition_t) * nparts);
  const uint64_t h = fnv1a(key.data(), key.size());
  bool known = false;   // validated before (on some device)
  for (auto& tp : g_plans) known = known || (tp->hash == h && tp->key == key);
  std::unique_ptr<TablePlan> tp(new TablePlan());
  if (!known) {
    // validation needs no GPU: a bad table is reported before any CUDA call
    int rc = validate_and_build(params, nparams, parts, nparts, tp->L);
    if (rc != MUON_OK) return rc;
  }
  int dev = 0;
  MUON_CUDA_TRY(cudaGetDevice(&dev));
  for (auto& p : g_plans)
    if (p->device == dev && p->hash == h && p->key == key) {
      *out = p.get();
      return MUON_OK;
    }
  if (known) {
    int rc = validate_and_build(params, nparams, parts, nparts, tp->L);
    if (rc != MUON_OK) return rc;
  }
  tp->device = dev;
  tp->hash = h;
  tp->key = std::move(key);
  const Layout& L = tp->L;
  MUON_CUDA_TRY(upload(tp->d_owners, L.owners));
  MUON_CUDA_TRY(upload(tp->d_segs, L.segs));
  MUON_CUDA_TRY(upload(tp->d_rtiles, L.rtiles));
  MUON_CUDA_TRY(upload(tp->d_gtiles, L.gtiles));
  MUON_CUDA_TRY(upload(tp->d_stiles, L.stiles));
  MUON_CUDA_TRY(upload(tp->d_ytiles, L.ytiles));
  MUON_CUDA_TRY(upload(tp->d_runs, L.runs));
  MUON_CUDA_TRY(tp->d_rsum.alloc(sizeof(double) * (L.rtiles.size() + 1)));
  MUON_CUDA_TRY(tp->d_ysum.alloc(sizeof(double) * (L.ytiles.size() + 1)));
  MUON_CUDA_TRY(tp->d_fin.alloc(sizeof(double) * kFinParts));
  MUON_CUDA_TRY(tp->d_div.alloc(sizeof(float) * (L.owners.size() + 1)));
  MUON_CUDA_TRY(tp->d_state.alloc(sizeof(StepState)));
  MUON_CUDA_TRY(tp->d_err.alloc(sizeof(int)));
  MUON_CUDA_TRY(cudaMemset(tp->d_err.p, 0, sizeof(int)));
  *out = tp.get();
  g_plans.push_back(std::move(tp));
  return MUON_OK;
}

// Splits the NS problems (stacks of Muon blocks, in owner order) into waves
// whose workspace fits `budget` bytes (a problem larger than the budget is
// a wave of its own) and builds one plan per wave over a shared workspace.
int build_wave_plan(const Layout& L, int method, int mode, int steps, uint64_t budget, NsPlan& P) {
  NsFormats F;
  int rc = ns_formats(method, mode, F);
  if (rc != MUON_OK) return rc;
  const NsBlocks NB = ns_blocks(L.owners, F.tc, mode == MUON_OPERANDS_BF16, method == MUON_NS_GRAM,
                                -1, false);
  // The shared workspace holds the largest wave's m x n regions and the
  // largest wave's m x m regions, which may come from different waves, so
  // a problem joins the current wave only while those running maxima still
  // fit the budget.
  std::vector<Owner> owners = L.owners;
  std::vector<std::vector<int>> waves;   // owner indices per wave
  std::vector<size_t> wave_prob0;        // first problem of each wave
  int64_t cx = 0, csq = 0, mx = 0, msq = 0;
  for (size_t k = 0; k < NB.probs.size(); ++k) {
    const Owner& q = NB.probs[k];
    const int first = NB.members[k].first, count = NB.members[k].second;
    int64_t ox = 0;
    for (int i = first; i < first + count; ++i)
      ox += round_up(int64_t(owners[i].m) * owners[i].ldx, 64);
    const int64_t osq = round_up(int64_t(q.m) * q.ldm, 64);
    if (waves.empty() ||
        F.ws_bytes(std::max(mx, cx + ox), std::max(msq, csq + osq)) > budget) {
      waves.emplace_back();
      wave_prob0.push_back(k);
      cx = csq = 0;
    }
    for (int i = first; i < first + count; ++i) {   // members stay adjacent
      owners[i].x_off = cx;
      cx += round_up(int64_t(owners[i].m) * owners[i].ldx, 64);
      waves.back().push_back(i);
    }
    csq += osq;
    mx = std::max(mx, cx);
    msq = std::max(msq, csq);
  }
  MUON_CUDA_TRY(P.ws.alloc(F.ws_bytes(mx, msq) + 256));
  MUON_CUDA_TRY(upload(P.d_owners, owners));
  // fused sums of squares of all waves in one buffer, problems in owner order
  const int last_engine = !F.tc ? ENGINE_SIMT
                          : (mode == MUON_OPERANDS_BF16 ? (NB.pairs ? ENGINE_TC2 : ENGINE_TC)
                                                        : ENGINE_X3);
  std::vector<int64_t> ssq_off(NB.probs.size() + 1, 0);
  for (size_t k = 0; k < NB.probs.size(); ++k)
    ssq_off[k + 1] = ssq_off[k] + (last_engine == ENGINE_SIMT ? 0
                                   : ssq_slots(last_engine, NB.probs[k].m, NB.probs[k].n));
  if (last_engine != ENGINE_SIMT) {
    const int64_t n = std::max<int64_t>(ssq_off.back(), 1);
    MUON_CUDA_TRY(P.ssq.alloc(sizeof(double) * n));
    MUON_CUDA_TRY(cudaMemset(P.ssq.p, 0, sizeof(double) * n));
    P.ssq_ptr = P.ssq.as<double>();
    P.n_ssq = ssq_off.back();
  }
  P.esize = F.xe;
  P.x_ps = F.xe == 6 ? mx : 0;
  P.x_elems = mx;
  P.use_tc = F.tc;
  P.method = method;
  P.steps = steps;
  // first tile of each owner in the gather / scatter / update tile lists
  auto first_of = [&](auto const& tiles, int owner) {
    int lo = 0, hi = static_cast<int>(tiles.size());
    while (lo < hi) {
      const int mid = (lo + hi) / 2;
      if (tiles[mid].owner < owner) lo = mid + 1; else hi = mid;
    }
    return lo;
  };
  for (size_t w = 0; w < waves.size(); ++w) {
    std::vector<Owner> wo;
    for (int i : waves[w]) wo.push_back(owners[i]);
    std::unique_ptr<NsPlan> sub(new NsPlan());
    rc = build_ns_plan(wo, mx, method, mode, steps, *sub, P.ws.as<char>(), msq, NB.cap,
                       P.ssq_ptr ? P.ssq_ptr + ssq_off[wave_prob0[w]] : nullptr, NB.pairs);
    if (rc != MUON_OK) return rc;
    P.flops += sub->flops;
    P.x0 = sub->x0;
    P.y = sub->y;
    const int ob = waves[w].front(), oe = waves[w].back() + 1;
    double el = 0.0;
    for (int i : waves[w]) el += double(owners[i].numel);
    P.ranges.push_back({first_of(L.gtiles, ob), first_of(L.gtiles, oe), first_of(L.stiles, ob),
                        first_of(L.stiles, oe), first_of(L.ytiles, ob), first_of(L.ytiles, oe), el});
    P.waves.push_back(std::move(sub));
  }
  return MUON_OK;
}

int get_ns_plan(TablePlan& tp, int method, int mode, int steps, uint64_t budget, NsPlan** out) {
  auto k = std::make_tuple(method, mode, steps, budget);
  auto it = tp.ns.find(k);
  if (it != tp.ns.end()) {
    *out = it->second.get();
    return MUON_OK;
  }
  std::unique_ptr<NsPlan> P(new NsPlan());
  int rc = budget ? build_wave_plan(tp.L, method, mode, steps, budget, *P)
                  : build_ns_plan(tp.L.owners, tp.L.x_elems, method, mode, steps, *P);
  if (rc != MUON_OK) return rc;
  *out = P.get();
  tp.ns[k] = std::move(P);
  return MUON_OK;
}

int check_method(int ns_method, int ns_steps, int mode) {
  if (ns_method != MUON_NS_STANDARD && ns_method != MUON_NS_GRAM)
    return fail(MUON_ERR_UNSUPPORTED, "unknown ns_method");
  if (ns_steps < 1 || ns_steps > 64) return fail(MUON_ERR_UNSUPPORTED, "ns_steps must be in [1, 64]");
  if (mode != MUON_OPERANDS_BF16 && mode != MUON_OPERANDS_FP32)
    return fail(MUON_ERR_UNSUPPORTED, "unknown operand mode");
  return MUON_OK;
}

int enqueue_gemms(NsPlan& P, const StepState* state, int* err, cudaStream_t s) {
  for (auto& ph : P.phases) {
    if (ph->engine == ENGINE_CONVERT) {
      PhaseScope sc(MUON_PHASE_NS_GEMM, s, ph->conv_n > 0 ? 1 : 0, 6.0 * ph->conv_n, 0.0);
      launch_convert_bf16(ph->conv_src, ph->conv_dst, ph->conv_n, state, s);
      continue;
    }
    if (ph->engine == ENGINE_TC2) {
      if (!ph->program_head) continue;   // launched with its program's first phase
      PairProgram& G = *P.programs[ph->program];
      PhaseScope sc(MUON_PHASE_NS_GEMM, s, G.tasks.empty() ? 0 : 1, 0.0, G.flops);
      if (launch_gemm_tc2(G.d_probs.as<GemmProblem>(), G.d_maps.as<TcMaps>(),
                          G.d_tasks.as<PairTask>(), static_cast<int>(G.tasks.size()),
                          G.d_counters.as<int>(), G.ncounters, state, err, s) != 0)
        return fail(MUON_ERR_CUDA, "tensor-core pair GEMM launch setup failed");
      continue;
    }
    PhaseScope sc(MUON_PHASE_NS_GEMM, s, ph->tiles.empty() ? 0 : 1, 0.0, ph->flops);
    if (ph->tiles.empty()) continue;
    if (ph->engine == ENGINE_TC) {
      if (launch_gemm_tc(ph->d_probs.as<GemmProblem>(), ph->d_maps.as<TcMaps>(),
                         ph->d_tiles.as<GemmTile>(), static_cast<int>(ph->tiles.size()), state, err,
                         s) != 0)
        return fail(MUON_ERR_CUDA, "tensor-core GEMM launch setup failed");
    } else if (ph->engine == ENGINE_X3) {
      if (launch_gemm_x3(ph->d_probs.as<GemmProblem>(), ph->d_maps.as<TcMaps>(),
                         ph->d_tiles.as<GemmTile>(), static_cast<int>(ph->tiles.size()), state, err,
                         s) != 0)
        return fail(MUON_ERR_CUDA, "split-3 tensor-core GEMM launch setup failed");
    } else {
      launch_gemm_simt(ph->d_probs.as<GemmProblem>(), ph->d_tiles.as<GemmTile>(),
                       static_cast<int>(ph->tiles.size()), ph->ab_es, state, s);
    }
  }
  return MUON_OK;
}

// ------------------------------------------------------------------ NS-only plans

struct SinglePlan {
  int device, rows, cols, method, mode, steps;
  std::vector<Owner> owners;
  int64_t x_elems, sq_elems;
  int ntiles;
  DevBuf tile_sum;
  DevBuf err;
  NsPlan ns;
};
std::vector<std::unique_ptr<SinglePlan>> g_single;

}  // namespace

void set_last_error(const char* msg) {
  if (msg) g_err = msg;
  else g_err.clear();
}

std::mutex& library_mutex() { return g_mu; }

void count_launches(int n) {
  g_cnt.launches_last = n;
  g_cnt.launches_total += n;
}

int validate_tables(const muon_param_t* params, int nparams, const muon_partition_t* parts,
                    int nparts) {
  Layout L;
  return validate_and_build(params, nparams, parts, nparts, L);
}

}  // namespace muon

// ==================================================================== C ABI

using namespace muon;

namespace {

// The runs an accumulation covers: every element (params == NULL, a cached
// list of 32768-element runs over n) or the elements some parameter covers.
struct AccRuns {
  const Run* runs = nullptr;
  int nruns = 0;
  double elems = 0.0;
  int64_t extent = 0;
  int* dbg_flag = nullptr;
};

int accumulate_runs(int64_t n, const muon_param_t* params, int nparams,
                    const muon_partition_t* parts, int nparts, AccRuns* out) {
  if (params == nullptr) {
    if (n < 0) return fail(MUON_ERR_INVALID, "n < 0");
    if (n == 0) return MUON_OK;
    static std::map<std::pair<int, int64_t>, std::unique_ptr<DevBuf>> dense;
    int dev = 0;
    MUON_CUDA_TRY(cudaGetDevice(&dev));
    auto key = std::make_pair(dev, n);
    auto it = dense.find(key);
    if (it == dense.end()) {
      std::vector<Run> runs;
      for (int64_t r = 0; r < n; r += 32768) runs.push_back({r, std::min<int64_t>(32768, n - r)});
      std::unique_ptr<DevBuf> b(new DevBuf());
      MUON_CUDA_TRY(upload(*b, runs));
      it = dense.emplace(key, std::move(b)).first;
    }
    out->runs = it->second->as<Run>();
    out->nruns = static_cast<int>((n + 32767) / 32768);
    out->elems = double(n);
    out->extent = n - g_knobs.extent_shrink;
    return MUON_OK;
  }
  TablePlan* tp = nullptr;
  int rc = get_table_plan(params, nparams, parts, nparts, &tp);
  if (rc != MUON_OK) return rc;
  out->runs = tp->d_runs.as<Run>();
  out->nruns = static_cast<int>(tp->L.runs.size());
  out->elems = double(tp->L.muon_elems + tp->L.aux_elems);
  out->extent = tp->L.storage_extent - g_knobs.extent_shrink;
  out->dbg_flag = tp->d_err.as<int>();
  return MUON_OK;
}

}  // namespace

extern "C" int muon_accumulate(float* accum, const uint16_t* grad, int64_t n, float scale,
                               int overwrite, const muon_param_t* params, int nparams,
                               const muon_partition_t* parts, int nparts, void* stream) {
  NvtxRange nvtx_("muon_accumulate");
  std::lock_guard<std::mutex> lk(g_mu);
  g_err.clear();
  g_cnt.launches_last = 0;
  if (!accum || !grad) return fail(MUON_ERR_INVALID, "accum or grad is NULL");
  if (reinterpret_cast<uintptr_t>(accum) % 16 || reinterpret_cast<uintptr_t>(grad) % 8)
    return fail(MUON_ERR_INVALID, "accum must be 16-byte and grad 8-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  AccRuns r;
  int rc = accumulate_runs(n, params, nparams, parts, nparts, &r);
  if (rc != MUON_OK || r.nruns == 0) return rc;
  PhaseScope sc(MUON_PHASE_ACCUMULATE, s, 1, r.elems * (overwrite ? 6 : 10), 0.0);
  launch_accumulate(accum, grad, r.runs, r.nruns, scale, overwrite, r.extent, r.dbg_flag, s);
  MUON_CUDA_TRY(cudaGetLastError());
  return MUON_OK;
}

extern "C" int muon_accumulate_n(float* accum, const uint16_t* const* grads, const float* scales,
                                 int count, int64_t n, int overwrite, const muon_param_t* params,
                                 int nparams, const muon_partition_t* parts, int nparts,
                                 void* stream) {
  NvtxRange nvtx_("muon_accumulate_n");
  std::lock_guard<std::mutex> lk(g_mu);
  g_err.clear();
  g_cnt.launches_last = 0;
  if (!accum || !grads || !scales) return fail(MUON_ERR_INVALID, "accum, grads or scales is NULL");
  if (count < 1 || count > MUON_ACCUMULATE_MAX)
    return fail(MUON_ERR_INVALID, "count must be 1 .. MUON_ACCUMULATE_MAX");
  if (reinterpret_cast<uintptr_t>(accum) % 16)
    return fail(MUON_ERR_INVALID, "accum must be 16-byte aligned");
  GradSet gs{};
  gs.count = count;
  for (int j = 0; j < count; ++j) {
    if (!grads[j] || reinterpret_cast<uintptr_t>(grads[j]) % 8)
      return fail(MUON_ERR_INVALID, "every grads[j] must be non-NULL and 8-byte aligned");
    gs.grad[j] = grads[j];
    gs.scale[j] = scales[j];
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  AccRuns r;
  int rc = accumulate_runs(n, params, nparams, parts, nparts, &r);
  if (rc != MUON_OK || r.nruns == 0) return rc;
  PhaseScope sc(MUON_PHASE_ACCUMULATE, s, 1, r.elems * ((overwrite ? 4 : 8) + 2.0 * count), 0.0);
  launch_accumulate_n(accum, gs, r.runs, r.nruns, overwrite, r.extent, r.dbg_flag, s);
  MUON_CUDA_TRY(cudaGetLastError());
  return MUON_OK;
}

namespace {

bool misaligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 != 0; }

// Validates the options and fills the option fields of the launch
// arguments; NULL options give muon_step's behaviour.
int apply_options(const muon_step_options_t* opts, StreamLaunchArgs& a) {
  a.grad_scale = 1.f;
  a.clip_mode = MUON_CLIP_UPDATE;
  a.reduce_mode = 0;
  a.adam = 0;
  a.park = 0;
  a.last_grad = nullptr;
  a.last_scale = 1.f;
  a.last_overwrite = 0;
  a.stats_out = nullptr;
  a.prev_grad = nullptr;
  a.prev_scale = 1.f;
  a.prev_overwrite = 0;
  a.fold_vec16 = 0;
  if (!opts) return MUON_OK;
  const bool v3 = opts->struct_size == static_cast<int32_t>(sizeof(muon_step_options_t));
  const bool v2 = v3 || opts->struct_size == MUON_STEP_OPTIONS_V2_SIZE;
  if (!v2 && opts->struct_size != MUON_STEP_OPTIONS_V1_SIZE)
    return fail(MUON_ERR_INVALID,
                "opts->struct_size must be sizeof(muon_step_options_t), MUON_STEP_OPTIONS_V2_SIZE "
                "or MUON_STEP_OPTIONS_V1_SIZE");
  if (v3 && opts->stats_out) {
    if (reinterpret_cast<uintptr_t>(opts->stats_out) % 8)
      return fail(MUON_ERR_INVALID, "stats_out must be 8-byte aligned");
    a.stats_out = opts->stats_out;
  }
  if (v2 && opts->last_grad) {
    if (reinterpret_cast<uintptr_t>(opts->last_grad) % 8)
      return fail(MUON_ERR_INVALID, "last_grad must be 8-byte aligned");
    if (!std::isfinite(opts->last_grad_scale))
      return fail(MUON_ERR_INVALID, "last_grad_scale must be finite");
    if (opts->last_grad_overwrite != 0 && opts->last_grad_overwrite != 1)
      return fail(MUON_ERR_INVALID, "last_grad_overwrite must be 0 or 1");
    a.last_grad = opts->last_grad;
    a.last_scale = opts->last_grad_scale;
    a.last_overwrite = opts->last_grad_overwrite;
  }
  if (v3 && opts->prev_grad) {
    if (!a.last_grad) return fail(MUON_ERR_INVALID, "prev_grad needs last_grad");
    if (reinterpret_cast<uintptr_t>(opts->prev_grad) % 8)
      return fail(MUON_ERR_INVALID, "prev_grad must be 8-byte aligned");
    if (!std::isfinite(opts->prev_grad_scale))
      return fail(MUON_ERR_INVALID, "prev_grad_scale must be finite");
    if (opts->prev_grad_overwrite != 0 && opts->prev_grad_overwrite != 1)
      return fail(MUON_ERR_INVALID, "prev_grad_overwrite must be 0 or 1");
    a.prev_grad = opts->prev_grad;
    a.prev_scale = opts->prev_grad_scale;
    a.prev_overwrite = opts->prev_grad_overwrite;
  }
  a.fold_vec16 = a.last_grad && reinterpret_cast<uintptr_t>(a.last_grad) % 16 == 0 &&
                 reinterpret_cast<uintptr_t>(a.prev_grad) % 16 == 0;
  if (opts->clip_mode != MUON_CLIP_UPDATE && opts->clip_mode != MUON_CLIP_GRAD)
    return fail(MUON_ERR_INVALID, "unknown clip_mode");
  if (!std::isfinite(opts->grad_scale) || opts->grad_scale < 0.f)
    return fail(MUON_ERR_INVALID, "grad_scale must be finite and >= 0");
  a.clip_mode = opts->clip_mode;
  a.grad_scale = opts->grad_scale == 0.f ? 1.f : opts->grad_scale;
  if (opts->aux_adam != 0 && opts->aux_adam != 1) return fail(MUON_ERR_INVALID, "aux_adam must be 0 or 1");
  if (opts->aux_adam) {
    if (!opts->exp_avg || !opts->exp_avg_sq)
      return fail(MUON_ERR_INVALID, "aux_adam needs exp_avg and exp_avg_sq");
    if (misaligned16(opts->exp_avg) || misaligned16(opts->exp_avg_sq))
      return fail(MUON_ERR_INVALID, "exp_avg and exp_avg_sq must be 16-byte aligned");
    if (opts->adam_step < 1) return fail(MUON_ERR_INVALID, "adam_step must be >= 1");
    const float b1 = opts->adam_beta1, b2 = opts->adam_beta2;
    if (!std::isfinite(opts->adam_lr) || !std::isfinite(opts->adam_eps) || opts->adam_eps < 0.f ||
        !(b1 >= 0.f && b1 < 1.f) || !(b2 >= 0.f && b2 < 1.f))
      return fail(MUON_ERR_INVALID, "adam_lr, adam_eps >= 0 finite and betas in [0, 1) required");
    // Kingma & Ba: bias corrections 1 - beta^t, formed in double and rounded
    // once to the FP32 constants the kernel multiplies by
    const double t = static_cast<double>(opts->adam_step);
    const double bc1 = 1.0 - std::pow(static_cast<double>(b1), t);
    const double bc2 = 1.0 - std::pow(static_cast<double>(b2), t);
    a.adam = 1;
    a.adam_b1 = b1;
    a.adam_b2 = b2;
    a.adam_omb1 = static_cast<float>(1.0 - static_cast<double>(b1));
    a.adam_omb2 = static_cast<float>(1.0 - static_cast<double>(b2));
    a.adam_eps = opts->adam_eps;
    a.adam_sqrt_bc2 = static_cast<float>(std::sqrt(bc2));
    a.adam_neg_step = static_cast<float>(-(static_cast<double>(opts->adam_lr) / bc1));
    a.exp_avg = opts->exp_avg;
    a.exp_avg_sq = opts->exp_avg_sq;
  }
  return MUON_OK;
}

int step_impl(float* accum, float* momentum, float* master, const muon_param_t* params,
              int nparams, const muon_partition_t* parts, int nparts, float beta, float lr,
              int ns_method, int ns_steps, float clip, int operand_mode,
              const muon_step_options_t* opts, muon_result_t* d_result, void* stream) {
  g_err.clear();
  g_cnt.launches_last = 0;
  int rc = check_method(ns_method, ns_steps, operand_mode);
  if (rc != MUON_OK) return rc;
  if (!d_result) return fail(MUON_ERR_INVALID, "d_result is NULL");
  if (nparams > 0 && (!accum || !momentum || !master))
    return fail(MUON_ERR_INVALID, "accum, momentum or master is NULL");
  if (misaligned16(accum) || misaligned16(momentum) || misaligned16(master))
    return fail(MUON_ERR_INVALID, "accum, momentum and master must be 16-byte aligned");
  if (!std::isfinite(beta) || !std::isfinite(lr) || !std::isfinite(clip))
    return fail(MUON_ERR_INVALID, "beta, lr and clip must be finite");
  StreamLaunchArgs a{};
  rc = apply_options(opts, a);
  if (rc != MUON_OK) return rc;
  TablePlan* tp = nullptr;
  rc = get_table_plan(params, nparams, parts, nparts, &tp);
  if (rc != MUON_OK) return rc;
  NsPlan* P = nullptr;
  const uint64_t budget = opts ? opts->workspace_budget : 0;
  rc = get_ns_plan(*tp, ns_method, operand_mode, ns_steps, budget, &P);
  if (rc != MUON_OK) return rc;
  const Layout& L = tp->L;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool waves = budget != 0;

  a.owners = waves ? P->d_owners.as<Owner>() : tp->d_owners.as<Owner>();
  a.segs = tp->d_segs.as<Segment>();
  a.rtiles = tp->d_rtiles.as<RTile>();
  a.ytiles = tp->d_ytiles.as<YTile>();
  a.n_rtiles = static_cast<int>(L.rtiles.size());
  a.n_ytiles = static_cast<int>(L.ytiles.size());
  a.n_owners = static_cast<int>(L.owners.size());
  a.accum = accum;
  a.momentum = momentum;
  a.master = master;
  a.rtile_sum = tp->d_rsum.as<double>();
  a.ytile_sum = tp->d_ysum.as<double>();
  a.fin_part = tp->d_fin.as<double>();
  a.owner_div = tp->d_div.as<float>();
  a.x0 = P->x0;
  a.y = P->y;
  a.esize = P->esize;
  a.x_ps = P->x_ps;
  a.beta = beta;
  a.lr = lr;
  a.clip = clip;
  a.state = tp->d_state.as<StepState>();
  a.err_flag = tp->d_err.as<int>();
  a.dbg_flag = tp->d_err.as<int>();
  a.dbg_storage_extent = L.storage_extent - g_knobs.extent_shrink;
  a.dbg_x_extent = P->x_elems;
  a.result = d_result;
  a.ns_calls = L.n_muon_owners;
  const bool pre = a.clip_mode == MUON_CLIP_GRAD;

  const double me = double(L.muon_elems), ae = double(L.aux_elems);
  MUON_CUDA_TRY(cudaMemsetAsync(a.state, 0, sizeof(StepState), s));
  // Folded micro-batches: the first pass reads 2 bytes per folded
  // micro-batch per element, and accum's 4 when they add to its old value;
  // it then writes the gradient into accum (4 bytes), and the later passes
  // read accum.  When a folded micro-batch overwrites accum, every pass forms
  // the gradient from the bf16 micro-batches instead, and a skipped step
  // writes it into accum at the end.
  const bool fold_old = fold_reads_accum(a);
  const double g_first = (a.last_grad && !fold_old ? 0.0 : 4.0) + (a.last_grad ? 2.0 : 0.0) +
                         (a.prev_grad && !a.last_overwrite ? 2.0 : 0.0);
  const double g_write = fold_old ? 4.0 : 0.0;
  const double g_bytes = fold_old ? 4.0 : g_first;   // per element, each later pass
  const bool fold_commit = a.last_grad != nullptr && !fold_old && a.n_rtiles > 0;
  auto first_pass = [&]() {
    launch_reduce(a, s);
    if (fold_old) {
      a.last_grad = nullptr;   // accum now holds the full gradient
      a.prev_grad = nullptr;
    }
  };
  if (!pre) {
    PhaseScope sc(MUON_PHASE_REDUCE, s, (a.n_rtiles ? 1 : 0) + 1,
                  (me + ae) * (g_first + g_write) + me * 4, 0.0);
    a.reduce_mode = 0;
    first_pass();
    launch_owner_norm(a, s);
  } else {
    // gradient norm over every parameter, clip coefficient, then the
    // per-block momentum norms of the clipped gradients
    PhaseScope sc(MUON_PHASE_REDUCE, s, (a.n_rtiles ? 2 : 0) + 3,
                  (me + ae) * (g_first + g_write) + me * (g_bytes + 4), 0.0);
    a.reduce_mode = 1;
    first_pass();
    launch_finalize_pre(a, s);
    a.reduce_mode = 2;
    launch_reduce(a, s);
    launch_owner_norm(a, s);
  }
  if (!waves) {
    {
      a.etiles = tp->d_gtiles.as<ETile>();
      a.n_etiles = static_cast<int>(L.gtiles.size());
      PhaseScope sc(MUON_PHASE_GATHER, s, a.n_etiles ? 1 : 0, me * (g_bytes + 8 + P->esize), 0.0);
      launch_gather(a, s);
    }
    rc = enqueue_gemms(*P, a.state, tp->d_err.as<int>(), s);
    if (rc != MUON_OK) return rc;
    {
      const bool fused = P->ssq_ptr != nullptr;   // the last product summed the squares
      PhaseScope sc(MUON_PHASE_NORM, s, (a.n_ytiles && !pre && !fused ? 1 : 0) + (pre ? 1 : 2),
                    pre || fused ? 0.0 : me * P->esize, 0.0);
      if (fused) {
        a.ytile_sum = P->ssq_ptr;
        a.n_ytiles = static_cast<int>(P->n_ssq);
      } else if (!pre) {
        launch_update_sumsq(a, s);
      }
      launch_finalize(a, s);
    }
    {
      a.etiles = tp->d_stiles.as<ETile>();
      a.n_etiles = static_cast<int>(L.stiles.size());
      PhaseScope sc(MUON_PHASE_SCATTER, s, (a.n_etiles ? 1 : 0) + (fold_commit ? 1 : 0),
                    me * (12 + P->esize) + ae * (g_bytes + (a.adam ? 28 : 4)), 0.0);
      launch_scatter(a, s);
      if (fold_commit) launch_fold_commit(a, s);
    }
  } else {
    // bounded workspace: per wave gather, NS, update sums and the Muon
    // write-back (unscaled and parked in accum when the coefficient comes
    // from the updates); then the coefficient and a final pass
    for (size_t w = 0; w < P->waves.size(); ++w) {
      const WaveRange& R = P->ranges[w];
      StreamLaunchArgs b = a;
      {
        b.etiles = tp->d_gtiles.as<ETile>() + R.g0;
        b.n_etiles = R.g1 - R.g0;
        PhaseScope sc(MUON_PHASE_GATHER, s, b.n_etiles ? 1 : 0, R.elems * (g_bytes + 8 + P->esize),
                      0.0);
        launch_gather(b, s);
      }
      rc = enqueue_gemms(*P->waves[w], a.state, tp->d_err.as<int>(), s);
      if (rc != MUON_OK) return rc;
      if (!pre && P->ssq_ptr == nullptr) {
        b.ytiles = tp->d_ytiles.as<YTile>() + R.y0;
        b.ytile_sum = tp->d_ysum.as<double>() + R.y0;
        b.n_ytiles = R.y1 - R.y0;
        PhaseScope sc(MUON_PHASE_NORM, s, b.n_ytiles ? 1 : 0, R.elems * P->esize, 0.0);
        launch_update_sumsq(b, s);
      }
      {
        b.park = 1;
        b.etiles = tp->d_stiles.as<ETile>() + R.s0;
        b.n_etiles = R.s1 - R.s0;
        PhaseScope sc(MUON_PHASE_SCATTER, s, b.n_etiles ? 1 : 0,
                      R.elems * (pre ? 12 + P->esize : 4 + P->esize), 0.0);
        launch_scatter(b, s);
      }
    }
    {
      if (P->ssq_ptr != nullptr) {
        a.ytile_sum = P->ssq_ptr;
        a.n_ytiles = static_cast<int>(P->n_ssq);
      }
      PhaseScope sc(MUON_PHASE_NORM, s, pre ? 1 : 2, 0.0, 0.0);
      launch_finalize(a, s);
    }
    {
      a.park = 2;
      a.etiles = tp->d_stiles.as<ETile>();
      a.n_etiles = static_cast<int>(L.stiles.size());
      PhaseScope sc(MUON_PHASE_SCATTER, s, (a.n_etiles ? 1 : 0) + (fold_commit ? 1 : 0),
                    (pre ? 0.0 : me * 16) + ae * (g_bytes + (a.adam ? 28 : 4)), 0.0);
      launch_scatter(a, s);
      if (fold_commit) launch_fold_commit(a, s);
    }
  }
  MUON_CUDA_TRY(cudaGetLastError());
  g_cnt.steps += 1;
  g_cnt.ns_calls_last = L.n_muon_owners;
  g_cnt.muon_mats_last = L.n_muon_params;
  return MUON_OK;
}

}  // namespace

extern "C" int muon_step(float* accum, float* momentum, float* master, const muon_param_t* params,
                         int nparams, const muon_partition_t* parts, int nparts, float beta,
                         float lr, int ns_method, int ns_steps, float clip, int operand_mode,
                         muon_result_t* d_result, void* stream) {
  NvtxRange nvtx_("muon_step");
  std::lock_guard<std::mutex> lk(g_mu);
  return step_impl(accum, momentum, master, params, nparams, parts, nparts, beta, lr, ns_method,
                   ns_steps, clip, operand_mode, nullptr, d_result, stream);
}

extern "C" int muon_step_ex(float* accum, float* momentum, float* master,
                            const muon_param_t* params, int nparams,
                            const muon_partition_t* parts, int nparts, float beta, float lr,
                            int ns_method, int ns_steps, float clip, int operand_mode,
                            const muon_step_options_t* opts, muon_result_t* d_result,
                            void* stream) {
  NvtxRange nvtx_("muon_step_ex");
  std::lock_guard<std::mutex> lk(g_mu);
  return step_impl(accum, momentum, master, params, nparams, parts, nparts, beta, lr, ns_method,
                   ns_steps, clip, operand_mode, opts, d_result, stream);
}

extern "C" int muon_newton_schulz(const void* X, void* Y, int rows, int cols, int io_dtype,
                                  int ns_method, int ns_steps, int operand_mode, void* stream) {
  NvtxRange nvtx_("muon_newton_schulz");
  std::lock_guard<std::mutex> lk(g_mu);
  g_err.clear();
  g_cnt.launches_last = 0;
  int rc = check_method(ns_method, ns_steps, operand_mode);
  if (rc != MUON_OK) return rc;
  if (!X || !Y) return fail(MUON_ERR_INVALID, "X or Y is NULL");
  if (X == Y) return fail(MUON_ERR_INVALID, "Y may not alias X");
  if (rows < 1 || cols < 1) return fail(MUON_ERR_INVALID, "rows and cols must be >= 1");
  if (io_dtype != MUON_DTYPE_BF16 && io_dtype != MUON_DTYPE_FP32)
    return fail(MUON_ERR_INVALID, "unknown io_dtype");
  int dev = 0;
  MUON_CUDA_TRY(cudaGetDevice(&dev));
  SinglePlan* sp = nullptr;
  for (auto& p : g_single)
    if (p->device == dev && p->rows == rows && p->cols == cols && p->method == ns_method &&
        p->mode == operand_mode && p->steps == ns_steps)
      sp = p.get();
  if (!sp) {
    std::unique_ptr<SinglePlan> np(new SinglePlan());
    np->device = dev; np->rows = rows; np->cols = cols;
    np->method = ns_method; np->mode = operand_mode; np->steps = ns_steps;
    Owner o{};
    o.rows = rows; o.cols = cols; o.numel = int64_t(rows) * cols; o.is_muon = 1;
    o.transposed = rows > cols; o.m = std::min(rows, cols); o.n = std::max(rows, cols);
    o.ldx = static_cast<int32_t>(round_up(o.n, 8));
    o.ldm = static_cast<int32_t>(round_up(o.m, 8));
    np->owners.push_back(o);
    np->x_elems = round_up(int64_t(o.m) * o.ldx, 64);
    np->sq_elems = round_up(int64_t(o.m) * o.ldm, 64);
    np->ntiles = static_cast<int>((o.numel + kReduceTile - 1) / kReduceTile);
    MUON_CUDA_TRY(np->tile_sum.alloc(sizeof(double) * (np->ntiles + 1)));
    MUON_CUDA_TRY(np->err.alloc(sizeof(int)));
    MUON_CUDA_TRY(cudaMemset(np->err.p, 0, sizeof(int)));
    rc = build_ns_plan(np->owners, np->x_elems, ns_method, operand_mode, ns_steps,
                       np->ns);
    if (rc != MUON_OK) return rc;
    sp = np.get();
    g_single.push_back(std::move(np));
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int io_es = io_dtype == MUON_DTYPE_BF16 ? 2 : 4;
  const double numel = double(rows) * cols;
  {
    PhaseScope sc(MUON_PHASE_REDUCE, s, 2, numel * io_es, 0.0);
    launch_ns_sumsq(X, io_es, int64_t(rows) * cols, sp->tile_sum.as<double>(), sp->ntiles, s);
  }
  {
    PhaseScope sc(MUON_PHASE_GATHER, s, 1, numel * (io_es + sp->ns.esize), 0.0);
    launch_ns_load(X, io_es, rows, cols, sp->tile_sum.as<double>(), sp->ntiles, sp->ns.x0,
                   sp->ns.esize, sp->owners[0].ldx, sp->ns.x_ps, s);
  }
  rc = enqueue_gemms(sp->ns, nullptr, sp->err.as<int>(), s);
  if (rc != MUON_OK) return rc;
  {
    PhaseScope sc(MUON_PHASE_SCATTER, s, 1, numel * (io_es + sp->ns.esize), 0.0);
    launch_ns_store(sp->ns.y, sp->ns.esize, sp->owners[0].ldx, sp->ns.x_ps, Y, io_es, rows, cols, s);
  }
  MUON_CUDA_TRY(cudaGetLastError());
  g_cnt.ns_calls_last = 1;
  return MUON_OK;
}

extern "C" int muon_get_stats(muon_stats_t* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!out) return fail(MUON_ERR_INVALID, "out is NULL");
  out->steps = g_cnt.steps;
  out->ns_calls_last_step = g_cnt.ns_calls_last;
  out->muon_matrices = g_cnt.muon_mats_last;
  out->kernel_launches_last_call = g_cnt.launches_last;
  out->kernel_launches_total = g_cnt.launches_total;
  size_t ws = 0;
  for (auto& tp : g_plans)
    for (auto& kv : tp->ns) ws += kv.second->ws.bytes;
  for (auto& sp : g_single) ws += sp->ns.ws.bytes;
  out->workspace_bytes = ws;
  return MUON_OK;
}

extern "C" const char* muon_last_error(void) { return g_err.c_str(); }

extern "C" void muon_release_workspace(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  cudaDeviceSynchronize();
  g_plans.clear();
  g_single.clear();
}

extern "C" int muon_device_error(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (cudaDeviceSynchronize() != cudaSuccess) return fail(MUON_ERR_CUDA, "device synchronize failed");
  int worst = 0;
  auto check = [&](DevBuf& b) {
    int v = 0;
    if (b.p && cudaMemcpy(&v, b.p, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess && v) {
      worst = v;
      cudaMemset(b.p, 0, sizeof(int));
    }
  };
  for (auto& tp : g_plans) check(tp->d_err);
  for (auto& sp : g_single) check(sp->err);
  const int na = noalloc_take_device_error();
  if (na) worst = na;
  return worst;
}

extern "C" int muon_testing_set(int knob, int value) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_err.clear();
  switch (knob) {
    case MUON_TEST_GEMM:
      if (value < 0 || value > 2) return fail(MUON_ERR_INVALID, "MUON_TEST_GEMM takes 0, 1 or 2");
      g_knobs.gemm = value;
      return MUON_OK;
    case MUON_TEST_STACK:
      if (value != 0 && value != 1) return fail(MUON_ERR_INVALID, "MUON_TEST_STACK takes 0 or 1");
      g_knobs.stack = value;
      return MUON_OK;
    case MUON_TEST_FLOW:
      if (value != 0 && value != 1) return fail(MUON_ERR_INVALID, "MUON_TEST_FLOW takes 0 or 1");
      g_knobs.flow = value;
      return MUON_OK;
    case MUON_TEST_FLOW_LAG:
      if (value < 0) return fail(MUON_ERR_INVALID, "MUON_TEST_FLOW_LAG takes a value >= 0");
      g_knobs.flow_lag = value;
      return MUON_OK;
    case MUON_TEST_FLOW_WAVES:
      if (value < 1) return fail(MUON_ERR_INVALID, "MUON_TEST_FLOW_WAVES takes a value >= 1");
      g_knobs.flow_waves = value;
      return MUON_OK;
    case MUON_TEST_EXTENT_SHRINK:
      if (value < 0) return fail(MUON_ERR_INVALID, "MUON_TEST_EXTENT_SHRINK takes a value >= 0");
      g_knobs.extent_shrink = value;
      return MUON_OK;
    case MUON_TEST_RASTER:
      if (value < 0 || value > 64) return fail(MUON_ERR_INVALID, "MUON_TEST_RASTER takes 0 to 64");
      g_knobs.raster = value;
      return MUON_OK;
    default:
      return fail(MUON_ERR_INVALID, "unknown testing knob");
  }
}

extern "C" int muon_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_profile = on != 0 ? (1u << MUON_PHASE_COUNT) - 1u : 0u;
  return MUON_OK;
}

extern "C" int muon_profile_enable_phases(uint32_t mask) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_profile = mask & ((1u << MUON_PHASE_COUNT) - 1u);
  return MUON_OK;
}

extern "C" int muon_profile_read(muon_phase_time_t* out, int nphases, int reset) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& pe : g_pending) {
    if (cudaEventSynchronize(pe.stop) != cudaSuccess) return fail(MUON_ERR_CUDA, "event sync failed");
    float ms = 0.f;
    cudaEventElapsedTime(&ms, pe.start, pe.stop);
    g_phase[pe.phase].total_ms += ms;
    g_phase[pe.phase].algorithmic_bytes += pe.bytes;
    g_phase[pe.phase].algorithmic_flops += pe.flops;
    g_event_pool.push_back(pe.start);
    g_event_pool.push_back(pe.stop);
  }
  g_pending.clear();
  if (out)
    for (int i = 0; i < nphases && i < MUON_PHASE_COUNT; ++i) out[i] = g_phase[i];
  if (reset) std::memset(g_phase, 0, sizeof(g_phase));
  return MUON_OK;
}

extern "C" int muon_describe_tables(const muon_param_t* params, int nparams,
                                    const muon_partition_t* parts, int nparts, int ns_method,
                                    int operand_mode, muon_table_info_t* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_err.clear();
  if (!out) return fail(MUON_ERR_INVALID, "out is NULL");
  int rc = check_method(ns_method, 5, operand_mode);
  if (rc != MUON_OK) return rc;
  Layout L;
  rc = validate_and_build(params, nparams, parts, nparts, L);
  if (rc != MUON_OK) return rc;
  const bool bf16 = operand_mode == MUON_OPERANDS_BF16;
  const NsBlocks NB = ns_blocks(L.owners, true, bf16, ns_method == MUON_NS_GRAM, -1,
                                false);   // as on a GB300
  NsFormats F;
  ns_formats_for(true, ns_method, operand_mode, F);
  std::memset(out, 0, sizeof(*out));
  out->muon_params = L.n_muon_params;
  out->muon_blocks = L.n_muon_owners;
  out->ns_problems = static_cast<int64_t>(NB.probs.size());
  out->pair_engine = NB.pairs ? 1 : 0;
  out->stack_rows = NB.cap;
  out->muon_elements = L.muon_elems;
  out->aux_elements = L.aux_elems;
  int64_t in_parts = 0;
  for (int i = 0; i < nparts; ++i) in_parts += parts[i].flat_end - parts[i].flat_begin;
  out->padding_elements = in_parts - L.muon_elems - L.aux_elems;
  out->segments = static_cast<int64_t>(L.segs.size());
  out->workspace_bytes = L.n_muon_owners ? F.ws_bytes(L.x_elems, NB.sq_elems) + 256 : 0;
  return MUON_OK;
}
