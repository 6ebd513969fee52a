// Internal data structures of libmuon, shared by the host planner and the
// CUDA kernels.  Plain structs only; everything here is copied to the device
// once per plan ("static tables computed once": the split tables of
// "Support Muon in BF16_Optimizer with FP32 gradient accumulation", review
// thread on all_to_all_single).
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "../../include/muon.h"

namespace muon {

// Fixed constants of the method (readings documented in the header).
constexpr float kNsA = 3.4445f;
constexpr float kNsB = -4.7750f;
constexpr float kNsC = 2.0315f;
constexpr double kNormEps = 1e-7;   // X0 = m / (||m||_F + kNormEps)
constexpr double kClipEps = 1e-6;   // coef = min(1, clip / (norm + kClipEps))

// Work granularity of the streaming kernels.
// Elements per pass-1 tile (the sum order is fixed by it).  Fewer, longer
// tiles spend less on each block's closing reduction: on Llama-3-8B layers
// the first pass took 4.36 / 4.06 / 3.92 ms with 16384 / 32768 / 65536.
constexpr int kReduceTile = 65536;
constexpr int kRowTile = 16384;     // target elements per row-aligned 1-D tile (32768 and
                                    // 65536 measured the same on Llama-3-8B layers)
constexpr int kTT = 64;             // 2-D transpose tile edge
constexpr int kStreamThreads = 256;
constexpr int kFoldCommitCtas = 152 * 8;   // k_fold_commit: 8 CTAs per SM, tiles strided
constexpr int kFinParts = 256;             // blocks of the global sum's first level

// A contiguous run shared by flat space and storage: the intersection of one
// owner (head block or auxiliary parameter) with one partition.
struct Segment {
  int64_t rel_begin;      // first element, relative to the owner's start
  int64_t storage_begin;  // storage index of that element
  int64_t len;
};

// One unit of the step: a Muon head block (an NS problem) or an auxiliary
// parameter.  Rows/cols are the block's own shape as it lies in the flat
// buffer (row-major); m x n is the canonical NS orientation (m <= n).
struct Owner {
  int64_t flat_begin;
  int64_t numel;
  int32_t rows, cols;
  int32_t m, n;
  int32_t transposed;   // rows > cols: X0 = block^T
  int32_t is_muon;
  int32_t seg_begin, seg_count;
  int32_t rtile_begin, rtile_count;   // pass-1 tiles of this owner
  int32_t ytile_begin, ytile_count;   // update sum-of-squares tiles
  int32_t ldx;          // leading dimension of the m x n workspace matrices
  int32_t ldm;          // leading dimension of the m x m workspace matrices
  int64_t x_off;        // element offset of this owner in each m x n region
  int64_t sq_off;       // element offset of this owner in each m x m region
  int32_t ns_blk;       // NS plans only: rows per stacked block (0: not stacked)
  int32_t ns_pad;
};

// Pass-1 tile: owner elements [rel_begin, rel_begin + len).  Thread t sums
// the elements of 4-element groups t, t + 256, ... in order, so the sum
// order depends only on the owner-relative index.  fast = 1: the tile lies
// in one segment, len % 4 == 0 and storage (sdelta + rel) is 16-byte aligned.
struct RTile {
  int32_t owner;
  int32_t len;
  int64_t rel_begin;
  int32_t fast, pad;
  int64_t sdelta;
};

// Tile of the gather (pass 2) and scatter kernels.
//   kind 0: rows [r0, r0 + nr) of a non-transposed Muon owner
//   kind 1: 64 x 64 tile at (r0, c0) of a transposed Muon owner
//   kind 2: elements [rel_begin, rel_begin + len) of an auxiliary owner
//   kind 3: gather only, 64 x 128 tile at (r0, c0) of a transposed Muon
//           owner, always fast (where it would not be, two kind-1 tiles)
// fast = 1 when the whole tile lies in one segment, its storage is 16-byte
// aligned and its rows are whole multiples of 4 elements: then storage index
// = sdelta + owner-relative index and the kernels use 16-byte accesses.
struct ETile {
  int32_t owner;
  int32_t kind;
  int32_t r0, nr;
  int32_t c0, fast;
  int64_t rel_begin;
  int64_t len;
  int64_t sdelta;
};

// Tile of the update sum of squares: rows [r0, r0 + nr) of an owner's
// canonical m x n result.
struct YTile {
  int32_t owner;
  int32_t r0, nr;
  int32_t pad;
};

// Accumulate work: storage run [begin, begin + len).
struct Run {
  int64_t begin;
  int64_t len;
};

// Device-side state of one step, reset at its start.
struct StepState {
  int32_t overflow;
  int32_t applied;
  float coef;
  float norm;
  double sumsq;
};

// One matrix product of the NS iteration:
//   D = alpha * A op(B) + beta * E + gamma * I
// A is M x K row-major (lda); B is N x K row-major when b_kmajor (ldb),
// else K x N row-major; D and E are M x N row-major.  When symmetric, only
// tiles touching the upper triangle are computed and each upper element is
// mirrored, so D is exactly symmetric.  A and B share one element type per
// launch (bf16 or fp32); D and E carry their own (d_es, e_es: 2 or 4 bytes).
struct GemmProblem {
  const void* A;
  const void* B;
  void* D;
  const void* E;
  int64_t lda, ldb, ldd, lde;
  int32_t M, N, K;
  int32_t b_kmajor;
  int32_t symmetric;
  float alpha, beta, gamma;
  int32_t d_es, e_es;   // 2 bf16, 4 fp32, 6 split-3 (three bf16 planes)
  // > 0: the problem stacks independent blocks of `blk` rows (a multiple of
  // 32); output chunks whose row and column fall in different blocks are
  // written as zeros (Gram products of stacked blocks)
  int32_t blk;
  // split-3 operands: element distance between the hi, mid and lo planes
  int64_t a_ps, b_ps, d_ps, e_ps;
  // non-null on the last product of the iteration: each epilogue warp writes
  // the sum of squares of the values it stored (as stored: bf16-rounded for
  // bf16 outputs) to ssq[(tm * tiles_n + tn) * kSsqSlots + its slot]
  double* ssq;
};
constexpr int kSsqSlots = 16;   // per output tile: 2 CTAs x 8 epilogue warps at most

struct GemmTile {
  int32_t problem;
  int32_t tm, tn;
};

// TMA descriptors of one problem for the tensor-core path.
struct TcMaps {   // CUtensorMap carries its own 64-byte alignment
  CUtensorMap a;   // A tiles: 128 rows x 64 K, 128-byte swizzle
  CUtensorMap b;   // B tiles: 256 x 64 (K-major) or 64 x 64 boxes (MN-major)
  CUtensorMap e;   // addend chunks 32 x 32 bf16, 64-byte swizzle (if E)
  CUtensorMap d;   // output boxes: 32 rows of 64 bytes (32 bf16 or 16 fp32), 64-byte swizzle
};

// ---------------------------------------------------------------- launches
// (defined in the .cu files; all enqueue on `stream`)

struct StreamLaunchArgs {
  const Owner* owners;
  const Segment* segs;
  const RTile* rtiles;
  const ETile* etiles;
  const YTile* ytiles;
  int n_rtiles, n_etiles, n_ytiles, n_owners;
  float* accum;
  float* momentum;
  float* master;
  double* rtile_sum;
  double* ytile_sum;
  double* fin_part;      // kFinParts partial sums of the global sum of squares
  float* owner_div;
  void* x0;          // X0 region (m x n per owner)
  const void* y;     // final NS result region
  int esize;         // workspace element format: 2 bf16, 4 fp32, 6 split-3 planes
  int64_t x_ps;      // split-3: elements between the planes of the X0 / Y regions
  float beta, lr, clip;
  StepState* state;
  const int* err_flag;   // set by a tensor-core kernel whose wait ran out
  muon_result_t* result;
  int ns_calls;
  // step options (muon_step_ex)
  float grad_scale;      // g = accum * grad_scale
  int clip_mode;         // 0: clip the updates; 1: clip the gradients first
  int reduce_mode;       // k_reduce: 0 update-mode sums, 1 gradient norm, 2 momentum after pre-clip
  int adam;              // auxiliary Adam on/off
  float adam_b1, adam_omb1, adam_b2, adam_omb2, adam_eps, adam_sqrt_bc2, adam_neg_step;
  float* exp_avg;
  float* exp_avg_sq;
  int park;              // bounded workspace: scatter writes the unclipped update to accum only
  // non-null: a micro-batch folded into the step's gradient (see Fold in
  // stream_kernels.cu: formed by every pass that reads the gradient, or by
  // the first pass alone, which then writes it into accum)
  const uint16_t* last_grad;
  float last_scale;
  int last_overwrite;
  // non-null (with last_grad): a micro-batch accumulated before last_grad
  const uint16_t* prev_grad;
  float prev_scale;
  int prev_overwrite;
  int fold_vec16;        // the folded micro-batches are 16-byte aligned (16-byte loads)
  // non-null: k_finalize writes {sum of squares, skipped, NS problems, 0}
  double* stats_out;
  // Debug builds (MUON_DEBUG): the extents the tables describe -- storage
  // elements of accum / momentum / master / grads, elements of one X region
  // of the workspace -- and the flag a tile that would leave them records
  // kErrBounds in (the tile is then skipped).  Unused in release builds.
  int64_t dbg_storage_extent;
  int64_t dbg_x_extent;
  int* dbg_flag;
};

// Error code of a debug build's bounds check (muon_device_error).
constexpr int kErrBounds = 16;

void launch_accumulate(float* accum, const uint16_t* grad, const Run* runs, int nruns,
                       float scale, int overwrite, int64_t dbg_extent, int* dbg_flag,
                       cudaStream_t s);
// Several micro-batches in one pass (muon_accumulate_n).
struct GradSet {
  const uint16_t* grad[MUON_ACCUMULATE_MAX];
  float scale[MUON_ACCUMULATE_MAX];
  int count;
};
void launch_accumulate_n(float* accum, const GradSet& gs, const Run* runs, int nruns, int overwrite,
                         int64_t dbg_extent, int* dbg_flag, cudaStream_t s);
void launch_reduce(const StreamLaunchArgs& a, cudaStream_t s);
void launch_fold_commit(const StreamLaunchArgs& a, cudaStream_t s);
// folded micro-batches that add to accum's old value (the first pass then writes the gradient)
bool fold_reads_accum(const StreamLaunchArgs& a);
void launch_owner_norm(const StreamLaunchArgs& a, cudaStream_t s);
void launch_gather(const StreamLaunchArgs& a, cudaStream_t s);
void launch_update_sumsq(const StreamLaunchArgs& a, cudaStream_t s);
void launch_finalize(const StreamLaunchArgs& a, cudaStream_t s);
void launch_finalize_pre(const StreamLaunchArgs& a, cudaStream_t s);
void launch_scatter(const StreamLaunchArgs& a, cudaStream_t s);

// NS-only entry: one matrix, io dtype bf16 or fp32.
void launch_ns_sumsq(const void* X, int io_esize, int64_t numel, double* tile_sum,
                     int ntiles, cudaStream_t s);
void launch_ns_load(const void* X, int io_esize, int rows, int cols, const double* tile_sum,
                    int ntiles, void* X0, int esize, int ldx, int64_t ps, cudaStream_t s);
void launch_ns_store(const void* Yws, int esize, int ldx, int64_t ps, void* Y, int io_esize,
                     int rows, int cols, cudaStream_t s);

// Matrix products.  ab_es selects bf16 (2) or fp32 (4) A/B operands.
void launch_gemm_simt(const GemmProblem* probs, const GemmTile* tiles, int ntiles, int ab_es,
                      const StepState* state, cudaStream_t s);
// dst[i] = bf16(src[i]) for i < n
void launch_convert_bf16(const float* src, void* dst, int64_t n, const StepState* state,
                         cudaStream_t s);
constexpr int kSimtTile = 128;

// FP32-accurate products on the BF16 tensor cores from split-3 operands
// (three exact bf16 planes per FP32 matrix; gemm_tc3.cu).
bool x3_encode_maps(const GemmProblem& p, TcMaps* out);
int launch_gemm_x3(const GemmProblem* probs, const TcMaps* maps, const GemmTile* tiles, int ntiles,
                   const StepState* state, int* err_flag, cudaStream_t s);
constexpr int kX3BM = 128, kX3BN = 128;

// Sets (msg != nullptr) or clears the text muon_last_error() returns.
void set_last_error(const char* msg);
// An NVTX range over a scope (host side): each entry point and each launch
// group of a step is named in timeline tools (Nsight Systems, ncu's NVTX
// filters).  Without a tool attached the calls cost a branch.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// The lock every entry point holds for the whole call.
std::mutex& library_mutex();
// Adds n kernel launches to muon_get_stats' counters (the caller holds the
// library lock).
void count_launches(int n);
// The table checks of muon_step (host only): MUON_OK or the error it would
// report, with muon_last_error() set.
int validate_tables(const muon_param_t* params, int nparams, const muon_partition_t* parts,
                    int nparts);
// The allocation-free entry's device error flag on every device that has
// used it: the first nonzero code, cleared once read (0 = none).
int noalloc_take_device_error();

// Tensor-core (tcgen05) path, BF16 operands.
constexpr int kTcBM = 128;
constexpr int kTcBN = 256;
constexpr int kTcBK = 64;
bool tc_available();
// Encodes the TMA descriptors of one problem; false if the driver refuses.
bool tc_encode_maps(const GemmProblem& p, TcMaps* out);
int launch_gemm_tc(const GemmProblem* probs, const TcMaps* maps, const GemmTile* tiles,
                   int ntiles, const StepState* state, int* err_flag, cudaStream_t s);

// Tensor-core path on SM pairs (tcgen05 cta_group::2, clusters of two
// CTAs), BF16 operands, 256 x 256 tiles, fed from a task list.
constexpr int kTcPairBM = 256;
constexpr int kTcPairBN = 256;
constexpr int kPairArrivals = 2;   // one arrival per CTA of the pair per tile
// One output tile of one product.  dep >= 0: its operands are ready when
// counters[dep] >= dep_target (each tile of an earlier product of the same
// NS problem adds kPairArrivals when its outputs are in memory);
// done >= 0: the counter this tile raises.  counters[0] hands out tasks.
struct PairTask {
  int32_t problem;
  int32_t tm, tn;
  int32_t dep, dep_target;
  int32_t done;
  int32_t nk;        // K blocks of 64
  int32_t b_kmajor;  // the problem's B layout
};
bool tc2_encode_maps(const GemmProblem& p, TcMaps* out);
int tc2_pairs();   // SM pairs of the current device
// Zeroes counters[0, ncounters) on `s`, then runs the tasks.
int launch_gemm_tc2(const GemmProblem* probs, const TcMaps* maps, const PairTask* tasks,
                    int ntasks, int* counters, int ncounters, const StepState* state,
                    int* err_flag, cudaStream_t s);

}  // namespace muon
