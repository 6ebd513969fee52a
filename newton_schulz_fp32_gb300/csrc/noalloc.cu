// muon_newton_schulz_noalloc: Newton-Schulz of one matrix without any
// device allocation.
//
// Some callers cannot call cudaMalloc: processes whose device memory is
// handed out by another allocator that reserves it up front (a direct
// cudaMalloc would bypass it or find the memory gone), and runtimes that
// forbid allocation once they serve (cudaMalloc can synchronise the device
// and stall them).  For them this entry point computes what
// muon_newton_schulz computes, but every byte of scratch it needs (norm
// partial sums, the X / X^T products, the m x m matrices, GEMM descriptors
// and TMA tensor maps) lives in one file-scope __device__ array of fixed
// size.  The array exists on every GPU that loads the library, from module
// load until the process exits.  BF16-operand products run on the
// single-SM tensor-core kernel; FP32-operand products and gram's m x m
// recurrence run on the CUDA-core FP32 GEMM (the allocating entry uses SM
// pairs and split-3 tensor-core products there), so results agree with
// muon_newton_schulz within the operand mode's tolerance.
//
// Limits: rows * cols <= 2^20, min(rows, cols) <= 512, max(rows, cols) <=
// 16384; the array is 16 MiB.
//
// Host code cannot use the array's name as a device address (in host code
// it names a host-side stand-in), so the first call on each device asks the
// runtime for the address with cudaGetSymbolAddress, with that device
// current, and keeps it.  Every call shares the array: two calls whose work
// overlaps on the GPU (different streams) race.  The host-side plan tables
// below are shared too, so a call holds the library lock from the address
// lookup until its last copy has been enqueued.
//
// The word at the start of the array is the error flag of the tensor-core
// GEMM's bounded waits.  It is zero when the module loads and is cleared
// only when muon_device_error reads it, so a code is not lost before it is
// queried.
#include <cstring>

#include "muon_internal.h"

namespace muon {
namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int64_t kMaxElems = int64_t(1) << 20;
constexpr int kMaxMinDim = 512;
constexpr int kMaxDim = 16384;
constexpr int kMaxDevices = 64;
constexpr int kMaxPhases = 4 * 64 + 4;
constexpr int kMaxTileLists = 8;
constexpr int kMaxTilesPerList = 512;

unsigned char* g_scratch_addr[kMaxDevices];   // device address of the array, per device

int nofail(int code, const char* msg) {
  set_last_error(msg);
  return code;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
int64_t rup(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

enum { ENG_TC = 0, ENG_SIMT = 1, ENG_CONVERT = 2 };

// One launch of the iteration (one problem: the single matrix).
struct Op {
  int engine;
  int ab_es;
  int tile_list;
  GemmProblem prob;
  const float* conv_src;
  void* conv_dst;
  int64_t conv_n;
};

struct TileList {
  int engine, M, N, sym, count;
  GemmTile tiles[kMaxTilesPerList];
};

// Host-side plan, rebuilt on every call (no heap use).
Op g_ops[kMaxPhases];
TcMaps g_maps[kMaxPhases];
TileList g_lists[kMaxTileLists];

int tile_list_for(int engine, int M, int N, int sym, int* nlists) {
  for (int i = 0; i < *nlists; ++i)
    if (g_lists[i].engine == engine && g_lists[i].M == M && g_lists[i].N == N && g_lists[i].sym == sym)
      return i;
  if (*nlists >= kMaxTileLists) return -1;
  TileList& L = g_lists[*nlists];
  L.engine = engine; L.M = M; L.N = N; L.sym = sym; L.count = 0;
  const int bm = engine == ENG_TC ? kTcBM : kSimtTile, bn = engine == ENG_TC ? kTcBN : kSimtTile;
  for (int tm = 0; tm < (M + bm - 1) / bm; ++tm)
    for (int tn = 0; tn < (N + bn - 1) / bn; ++tn) {
      if (sym && tn * bn + bn - 1 < tm * bm) continue;
      if (L.count >= kMaxTilesPerList) return -1;
      L.tiles[L.count++] = {0, tm, tn};
    }
  return (*nlists)++;
}

}  // namespace
}  // namespace muon

using namespace muon;

int muon::noalloc_take_device_error() {   // the caller holds the library lock
  int worst = 0;
  for (int dev = 0; dev < kMaxDevices; ++dev) {
    if (g_scratch_addr[dev] == nullptr) continue;
    int v = 0;
    if (cudaMemcpy(&v, g_scratch_addr[dev], sizeof(int), cudaMemcpyDefault) == cudaSuccess && v) {
      if (!worst) worst = v;
      cudaMemset(g_scratch_addr[dev], 0, sizeof(int));
    }
  }
  return worst;
}

extern "C" int muon_newton_schulz_noalloc(const void* X, void* Y, int rows, int cols, int io_dtype,
                                          int ns_method, int ns_steps, int operand_mode,
                                          void* stream) {
  std::lock_guard<std::mutex> lk(library_mutex());
  NvtxRange nvtx_("muon_newton_schulz_noalloc");
  set_last_error(nullptr);
  if (!X || !Y || X == Y) return nofail(MUON_ERR_INVALID, "X, Y must be distinct device arrays");
  if (rows < 1 || cols < 1) return nofail(MUON_ERR_INVALID, "rows and cols must be >= 1");
  if (io_dtype != MUON_DTYPE_BF16 && io_dtype != MUON_DTYPE_FP32)
    return nofail(MUON_ERR_INVALID, "unknown io_dtype");
  if (ns_method != MUON_NS_STANDARD && ns_method != MUON_NS_GRAM)
    return nofail(MUON_ERR_UNSUPPORTED, "unknown ns_method");
  if (ns_steps < 1 || ns_steps > 64) return nofail(MUON_ERR_UNSUPPORTED, "ns_steps must be in [1, 64]");
  if (operand_mode != MUON_OPERANDS_BF16 && operand_mode != MUON_OPERANDS_FP32)
    return nofail(MUON_ERR_UNSUPPORTED, "unknown operand mode");
  const int m = rows < cols ? rows : cols, n = rows < cols ? cols : rows;
  if (int64_t(rows) * cols > kMaxElems || m > kMaxMinDim || n > kMaxDim)
    return nofail(MUON_ERR_UNSUPPORTED,
                  "muon_newton_schulz_noalloc: matrix too large for the fixed scratch "
                  "(limits: rows*cols <= 1048576, min(rows,cols) <= 512, max(rows,cols) <= 16384)");
  const bool bf16 = operand_mode == MUON_OPERANDS_BF16;
  if (bf16 && !tc_available())
    return nofail(MUON_ERR_UNSUPPORTED, "BF16 operand mode needs an sm_103 (GB300) GPU");

  // ---- per-device set-up: the array's device address
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return nofail(MUON_ERR_CUDA, "cudaGetDevice failed");
  // The TMA descriptors are encoded by a driver call, which needs the
  // device's context current on this host thread; a thread whose first CUDA
  // call this is has none yet, and cudaSetDevice makes it current.
  if (cudaSetDevice(dev) != cudaSuccess) return nofail(MUON_ERR_CUDA, "cudaSetDevice failed");
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return nofail(MUON_ERR_CUDA, "cudaGetSymbolAddress of the no-alloc scratch failed");
    g_scratch_addr[dev] = static_cast<unsigned char*>(p);
  }
  unsigned char* base = g_scratch_addr[dev];
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // ---- carve the scratch
  const int es = bf16 ? 2 : 4;
  const int io_es = io_dtype == MUON_DTYPE_BF16 ? 2 : 4;
  const int ldx = static_cast<int>(rup(n, 8)), ldm = static_cast<int>(rup(m, 8));
  const int64_t numel = int64_t(rows) * cols;
  const int ntiles = static_cast<int>((numel + kReduceTile - 1) / kReduceTile);
  size_t off = 0;
  int* err_flag = reinterpret_cast<int*>(base + off);
  off = align256(off + sizeof(int));
  double* tile_sum = reinterpret_cast<double*>(base + off);
  off = align256(off + sizeof(double) * (ntiles + 1));
  GemmProblem* d_probs = reinterpret_cast<GemmProblem*>(base + off);
  off = align256(off + sizeof(GemmProblem) * kMaxPhases);
  TcMaps* d_maps = reinterpret_cast<TcMaps*>(base + off);
  off = align256(off + sizeof(TcMaps) * kMaxPhases);
  GemmTile* d_tiles = reinterpret_cast<GemmTile*>(base + off);
  off = align256(off + sizeof(GemmTile) * kMaxTilesPerList * kMaxTileLists);
  unsigned char* X0 = base + off;
  off = align256(off + size_t(es) * m * ldx);
  unsigned char* X1 = base + off;
  off = align256(off + size_t(es) * m * ldx);
  const size_t sq = size_t(m) * ldm;
  unsigned char* S[6];
  const int nsq = ns_method == MUON_NS_STANDARD ? 2 : 5;
  const int sq_es = ns_method == MUON_NS_STANDARD ? es : 4;
  for (int i = 0; i < nsq; ++i) {
    S[i] = base + off;
    off = align256(off + sq_es * sq);
  }
  unsigned char* Qbf = base + off;
  if (ns_method == MUON_NS_GRAM && bf16) off = align256(off + 2 * sq);
  if (off > kScratchBytes) return nofail(MUON_ERR_UNSUPPORTED, "no-alloc scratch layout overflow");

  // ---- the iteration's launches (same products as muon_newton_schulz)
  const int big = bf16 ? ENG_TC : ENG_SIMT;
  int nops = 0, nlists = 0;
  auto add = [&](int engine, int ab_es, const void* A, int lda, const void* B, int ldb, int bk,
                 void* D, int ldd, int d_es, const void* E, int lde, int e_es, int M, int N, int K,
                 int sym, float al, float be, float ga) {
    Op& o = g_ops[nops];
    std::memset(&o, 0, sizeof(Op));
    o.engine = engine;
    o.ab_es = ab_es;
    GemmProblem& p = o.prob;
    p.A = A; p.B = B; p.D = D; p.E = E;
    p.lda = lda; p.ldb = ldb; p.ldd = ldd; p.lde = lde;
    p.M = M; p.N = N; p.K = K;
    p.b_kmajor = bk; p.symmetric = sym;
    p.alpha = al; p.beta = be; p.gamma = ga;
    p.d_es = d_es; p.e_es = e_es;
    o.tile_list = tile_list_for(engine, M, N, sym, &nlists);
    ++nops;
    return o.tile_list >= 0;
  };
  bool ok = true;
  const float a = kNsA, b = kNsB, c = kNsC;
  unsigned char* Yws = X1;
  if (ns_method == MUON_NS_STANDARD) {
    unsigned char* Xs[2] = {X0, X1};
    for (int st = 0; st < ns_steps && ok; ++st) {
      unsigned char* src = Xs[st & 1];
      unsigned char* dst = Xs[(st + 1) & 1];
      ok = ok && add(big, es, src, ldx, src, ldx, 1, S[0], ldm, es, nullptr, 0, es, m, m, n, 1, 1.f, 0.f, 0.f);
      ok = ok && add(big, es, S[0], ldm, S[0], ldm, 1, S[1], ldm, es, S[0], ldm, es, m, m, m, 1, c, b, 0.f);
      ok = ok && add(big, es, S[1], ldm, src, ldx, 0, dst, ldx, es, src, ldx, es, m, n, m, 0, 1.f, a, 0.f);
    }
    Yws = Xs[ns_steps & 1];
  } else {
    unsigned char *R = S[0], *Pm = S[1], *Qa = S[2], *Qb = S[3], *T = S[4];
    ok = ok && add(big, es, X0, ldx, X0, ldx, 1, R, ldm, 4, nullptr, 0, 4, m, m, n, 1, 1.f, 0.f, 0.f);
    unsigned char* Qcur = Qa;
    for (int k = 0; k < ns_steps && ok; ++k) {
      unsigned char* Pk = (k == 0) ? Qa : Pm;
      ok = ok && add(ENG_SIMT, 4, R, ldm, R, ldm, 0, Pk, ldm, 4, R, ldm, 4, m, m, m, 0, c, b, a);
      if (k > 0) {
        unsigned char* Qn = (Qcur == Qa) ? Qb : Qa;
        ok = ok && add(ENG_SIMT, 4, Pk, ldm, Qcur, ldm, 0, Qn, ldm, 4, nullptr, 0, 4, m, m, m, 0, 1.f, 0.f, 0.f);
        Qcur = Qn;
      }
      if (k < ns_steps - 1) {
        ok = ok && add(ENG_SIMT, 4, Pk, ldm, R, ldm, 0, T, ldm, 4, nullptr, 0, 4, m, m, m, 0, 1.f, 0.f, 0.f);
        ok = ok && add(ENG_SIMT, 4, T, ldm, Pk, ldm, 0, R, ldm, 4, nullptr, 0, 4, m, m, m, 0, 1.f, 0.f, 0.f);
      }
    }
    const unsigned char* Qy = Qcur;
    if (bf16) {
      Op& o = g_ops[nops++];
      std::memset(&o, 0, sizeof(Op));
      o.engine = ENG_CONVERT;
      o.conv_src = reinterpret_cast<const float*>(Qcur);
      o.conv_dst = Qbf;
      o.conv_n = static_cast<int64_t>(sq);
      Qy = Qbf;
    }
    ok = ok && add(big, es, Qy, ldm, X0, ldx, 0, X1, ldx, es, nullptr, 0, es, m, n, m, 0, 1.f, 0.f, 0.f);
    Yws = X1;
  }
  if (!ok || nops > kMaxPhases) return nofail(MUON_ERR_UNSUPPORTED, "no-alloc plan exceeds its tables");

  // ---- descriptors into the scratch (host arrays are static: no heap use)
  static GemmProblem h_probs[kMaxPhases];
  static GemmTile h_tiles[kMaxTilesPerList * kMaxTileLists];
  for (int i = 0; i < nops; ++i) {
    h_probs[i] = g_ops[i].prob;
    std::memset(&g_maps[i], 0, sizeof(TcMaps));
    if (g_ops[i].engine == ENG_TC && !tc_encode_maps(g_ops[i].prob, &g_maps[i]))
      return nofail(MUON_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  }
  for (int l = 0; l < nlists; ++l)
    std::memcpy(h_tiles + l * kMaxTilesPerList, g_lists[l].tiles, sizeof(GemmTile) * g_lists[l].count);
  if (cudaMemcpyAsync(d_probs, h_probs, sizeof(GemmProblem) * nops, cudaMemcpyHostToDevice, s) !=
          cudaSuccess ||
      cudaMemcpyAsync(d_maps, g_maps, sizeof(TcMaps) * nops, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(d_tiles, h_tiles, sizeof(GemmTile) * kMaxTilesPerList * nlists,
                      cudaMemcpyHostToDevice, s) != cudaSuccess)
    return nofail(MUON_ERR_CUDA, "copying descriptors into the no-alloc scratch failed");
  // the host arrays are pageable: each copy has staged them when it returns

  // ---- launches
  launch_ns_sumsq(X, io_es, numel, tile_sum, ntiles, s);
  launch_ns_load(X, io_es, rows, cols, tile_sum, ntiles, X0, es, ldx, 0, s);
  for (int i = 0; i < nops; ++i) {
    const Op& o = g_ops[i];
    if (o.engine == ENG_CONVERT) {
      launch_convert_bf16(o.conv_src, o.conv_dst, o.conv_n, nullptr, s);
      continue;
    }
    const GemmTile* tl = d_tiles + o.tile_list * kMaxTilesPerList;
    const int nt = g_lists[o.tile_list].count;
    if (o.engine == ENG_TC) {
      if (launch_gemm_tc(d_probs + i, d_maps + i, tl, nt, nullptr, err_flag, s) != 0)
        return nofail(MUON_ERR_CUDA, "tensor-core GEMM launch setup failed");
    } else {
      launch_gemm_simt(d_probs + i, tl, nt, o.ab_es, nullptr, s);
    }
  }
  launch_ns_store(Yws, es, ldx, 0, Y, io_es, rows, cols, s);
  if (cudaGetLastError() != cudaSuccess) return nofail(MUON_ERR_CUDA, "kernel launch failed");
  return MUON_OK;
}
