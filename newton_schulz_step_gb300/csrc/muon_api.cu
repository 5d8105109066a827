// muon_api.cu -- host side of the C ABI declared in include/muon_gb300.h:
// argument validation, workspace planning, TMA tensor maps, and the launch
// sequence of one Muon step:
//
//   small groups (min(rows,cols) < 64):  one fp32 kernel, whole step
//   tensor-core groups:                  prologue per group, then per NS round
//                                        Gram -> Poly -> Update, each one
//                                        grouped persistent launch over all
//                                        groups (up to kMaxProblems at a time)
//
// Everything is enqueued on the caller's stream; nothing here synchronises
// (except muon_workspace_status and muon_trace_end) or allocates device memory.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include <cudaTypedefs.h>

#include "internal.h"

using namespace muon;

namespace {

// ------------------------------------------------------------ bookkeeping
std::atomic<unsigned long long> g_launch_count{0};
// 1: matrices with 64 <= m <= 256 and n <= 512 take the one-kernel fused path
std::atomic<int> g_fused_enabled{1};
// NS rounds of tensor-core groups: 0 one launch per stage and round, 1 one
// persistent launch per chunk, 2 (default) persistent when a round is short
std::atomic<int> g_rounds_enabled{2};
// 1: the parameter write streams beside the last update (apply_stream_kernel)
// when one staged chunk covers every tensor-core matrix of the call
std::atomic<int> g_stream_apply_enabled{1};
// ... and only while what it waits beside (the whole rounds launch, or one
// round) is estimated under this (the streamed write's waits give up after 2 s)
constexpr double kStreamMaxUs = 1e5;

// The persistent launch pays off while stage boundaries (launch, pipeline fill,
// last-wave tail: a few microseconds each) weigh on a round; on rounds of
// milliseconds it was measured slower (d=2048 model: 37.4 vs 31.3 ms per
// step).  Estimated tensor-core time of one round of a chunk, in microseconds:
// 512 clocks per pair tile and 64-deep k-block, at ~1.9 GHz on sms / 2 pairs
// (round_mma_us below).

struct TraceSlot {
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  int kind = 0, round = -1;
  double flops = 0, bytes = 0;
};

std::mutex g_trace_mu;
bool g_trace_on = false;
int g_trace_cap = 0;
std::vector<TraceSlot> g_trace;

struct LaunchInfo {
  int kind;
  int round;
  double flops;
  double bytes;
};

// Runs `fn` (which launches one kernel), counting it and, when tracing,
// bracketing it with events on `st`.
template <typename F>
cudaError_t tracked_launch(cudaStream_t st, const LaunchInfo& info, F&& fn) {
  TraceSlot* slot = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (g_trace_on && static_cast<int>(g_trace.size()) < g_trace_cap) {
      TraceSlot ts;
      ts.kind = info.kind;
      ts.round = info.round;
      ts.flops = info.flops;
      ts.bytes = info.bytes;
      if (cudaEventCreate(&ts.e0) == cudaSuccess && cudaEventCreate(&ts.e1) == cudaSuccess) {
        g_trace.push_back(ts);
        slot = &g_trace.back();
        cudaEventRecord(slot->e0, st);
      }
    }
  }
  const cudaError_t e = fn();
  g_launch_count.fetch_add(1, std::memory_order_relaxed);
  if (slot) cudaEventRecord(slot->e1, st);
  return e;
}

// ------------------------------------------------------------ device info
struct DevInfo {
  int checked = 0;
  int ok = 0;
  int sms = 0;
};
DevInfo g_dev[64];
std::mutex g_dev_mu;

muon_status current_device(int* sms) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return MUON_ERR_UNSUPPORTED;
  if (dev >= 64) return MUON_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.checked) {
    int maj = 0, min = 0, n = 0;
    if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MUON_ERR_CUDA;
    d.checked = 1;
    d.ok = (maj == 10 && min == 3);  // the cubin is built for sm_103a only
    d.sms = n;
  }
  if (!d.ok) return MUON_ERR_UNSUPPORTED;
  *sms = d.sms;
  return MUON_OK;
}

// ------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// bf16 [batch][rows][ld] with logical width `cols`; box = box_cols x box_rows x 1.
// Loads read out-of-bounds elements as zero; stores skip them.
bool make_tmap(CUtensorMap* tm, const void* base, int cols, int rows, int batch, int ld,
               int box_cols, int box_rows, CUtensorMapSwizzle swizzle) {
  auto enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2,
                                 static_cast<cuuint64_t>(ld) * 2 * static_cast<cuuint64_t>(rows)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols),
                             static_cast<cuuint32_t>(box_rows), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// GEMM operand tiles: 64 columns (128 bytes) x box_rows, 128-byte swizzle.
bool operand_tmap(CUtensorMap* tm, const void* base, int cols, int rows, int batch, int ld,
                  int box_rows) {
  return make_tmap(tm, base, cols, rows, batch, ld, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Epilogue blocks of 32 rows x 64 columns (128 bytes), 128-byte swizzle.
bool output_tmap(CUtensorMap* tm, const void* base, int cols, int rows, int batch, int ld) {
  return make_tmap(tm, base, cols, rows, batch, ld, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
}

// ------------------------------------------------------------ planning
struct GPlan {
  // caller arrays
  float* p = nullptr;
  const void* g = nullptr;
  float* buf = nullptr;
  __nv_bfloat16* out = nullptr;
  int gdt = 0;
  int batch = 0, r = 0, c = 0;
  float lr_scale = 0.f;
  // derived
  int m = 0, n = 0;
  bool tall = false, small = false;
  int ldx = 0, lda = 0, nparts = 0;
  size_t x0 = 0, x1 = 0, am = 0, bm = 0, parts = 0, xs = 0;  // workspace offsets
  int ctr = 0;  // first per-matrix completion counter (rounds kernel, streamed write)
};

constexpr size_t kStatusBytes = 256;
constexpr int kMaxDim = 65536;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
int round_up(int x, int a) { return (x + a - 1) / a * a; }
int cdiv(int x, int a) { return (x + a - 1) / a; }

bool shape_ok(int batch, int r, int c) {
  return batch >= 0 && batch <= 65535 && r >= 1 && c >= 1 && r <= kMaxDim && c <= kMaxDim;
}

// Fills the derived fields and workspace offsets; returns the total bytes.
// Layout: the status block, the per-matrix completion counters of every
// tensor-core matrix (one u32 each), then each group's buffers.
size_t plan_workspace(std::vector<GPlan>& gs) {
  int counters = 0;
  for (GPlan& g : gs) {
    g.m = std::min(g.r, g.c);
    if (g.batch > 0 && g.m > kSmallMaxM) {
      g.ctr = counters;
      counters += g.batch;
    }
  }
  size_t off = kStatusBytes + (counters ? align256(static_cast<size_t>(counters) * 4) : 0);
  for (GPlan& g : gs) {
    g.tall = g.r > g.c;
    g.m = std::min(g.r, g.c);
    g.n = std::max(g.r, g.c);
    g.small = g.m <= kSmallMaxM;
    if (g.batch == 0) continue;
    const size_t b = static_cast<size_t>(g.batch);
    if (g.small) {
      g.xs = off;
      off += align256(b * g.m * g.n * sizeof(float));
    } else {
      g.ldx = round_up(g.n, 8);
      g.lda = round_up(g.m, 8);
      const size_t xb = align256(b * g.m * static_cast<size_t>(g.ldx) * 2);
      const size_t ab = align256(b * g.m * static_cast<size_t>(g.lda) * 2);
      g.x0 = off; off += xb;
      g.x1 = off; off += xb;
      g.am = off; off += ab;
      g.bm = off; off += ab;
      // ~4 of the prologue's 64x64 tiles per block, at most kMaxParts blocks per matrix
      const int tiles = cdiv(g.r, 64) * cdiv(g.c, 64);
      g.nparts = std::min(std::max(1, cdiv(tiles, 4)), kMaxParts);
      g.parts = off;
      off += align256(b * g.nparts * sizeof(float));
    }
  }
  return off;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool finite(float x) { return std::isfinite(x); }

struct Scalars {
  int mode;  // PrologueMode
  float beta, lr, wd;
  int steps;
  float a, b, c, eps;
};

muon_status check_scalars(const Scalars& s) {
  if (s.steps < 1 || s.steps > 16) return MUON_ERR_INVALID_ARG;
  if (!finite(s.a) || !finite(s.b) || !finite(s.c) || !finite(s.eps) || s.eps < 0.f)
    return MUON_ERR_INVALID_ARG;
  if (s.mode != kPrologueNsOnly) {
    if (!finite(s.beta) || s.beta < 0.f || s.beta > 1.f) return MUON_ERR_INVALID_ARG;
    if (!finite(s.lr) || !finite(s.wd)) return MUON_ERR_INVALID_ARG;
  }
  return MUON_OK;
}

muon_status check_group(const GPlan& g, int mode) {
  if (!shape_ok(g.batch, g.r, g.c)) return MUON_ERR_INVALID_ARG;
  if (g.gdt != MUON_F32 && g.gdt != MUON_BF16) return MUON_ERR_INVALID_ARG;
  if (!finite(g.lr_scale)) return MUON_ERR_INVALID_ARG;
  if (g.batch == 0) return MUON_OK;
  if (!g.g || !aligned16(g.g)) return MUON_ERR_INVALID_ARG;
  if (mode == kPrologueNsOnly) {
    if (!g.out || !aligned16(g.out)) return MUON_ERR_INVALID_ARG;
  } else {
    if (!g.p || !g.buf || !aligned16(g.p) || !aligned16(g.buf)) return MUON_ERR_INVALID_ARG;
  }
  return MUON_OK;
}

// ------------------------------------------------------------ GEMM launch setup
struct StageShape {
  int tiles_m, tiles_n, tiles_per_mat, k_blocks;
};

// Tiles of one stage in units of cluster pairs: two 128-row CTA tiles (rows
// 2p, 2p+1) of one 256-wide column.  Symmetric stages take, for pair row p,
// the columns q >= p (exactly the columns holding entries on or above the
// diagonal for both rows of the pair).
constexpr int kTileN = 256;

StageShape stage_shape(const GPlan& g, int stage) {
  StageShape s{};
  s.tiles_m = cdiv(cdiv(g.m, kTileM), 2);
  if (stage == kStageUpdate) {
    s.tiles_n = cdiv(g.n, kTileN);
    s.tiles_per_mat = s.tiles_m * s.tiles_n;
    s.k_blocks = cdiv(g.m, kTileK);
  } else {
    s.tiles_n = cdiv(g.m, kTileN);  // == tiles_m
    s.tiles_per_mat = 0;
    for (int p = 0; p < s.tiles_m; ++p) s.tiles_per_mat += s.tiles_n - p;
    s.k_blocks = cdiv(stage == kStageGram ? g.n : g.m, kTileK);
  }
  return s;
}

double stage_flops(const GPlan& g, int stage) {
  const double m = g.m, n = g.n, b = g.batch;
  if (stage == kStageGram) return b * n * m * (m + 1);      // m(m+1)/2 entries x 2n
  if (stage == kStagePoly) return b * m * m * (m + 1);      // m(m+1)/2 entries x 2m
  return b * 2.0 * m * m * n;
}

// Builds the launch block of one stage for a chunk of tensor-core groups.
// `cur` selects X0 (0) or X1 (1) as this round's X.
// `signal`: the last round's update, with the parameter write streamed beside
// it: per-matrix completion counters, and O^T for rows > cols matrices.
muon_status build_gemm(GemmLaunch& L, const std::vector<GPlan*>& chunk, int stage,
                       int cur, bool first_round, const Scalars& sc, uint8_t* ws,
                       bool signal) {
  std::memset(&L, 0, sizeof(L));
  // Order of the tile walk.  The update and Poly stages walk the groups by
  // ascending n (matrices ascending); the Gram stage walks the exact reverse,
  // so it reads first the X the previous update wrote last (still in L2), and
  // its heaviest tiles (largest n = longest K) are handed out first.
  std::vector<GPlan*> order(chunk);
  std::stable_sort(order.begin(), order.end(),
                   [](GPlan* x, GPlan* y) { return x->n < y->n; });
  const bool reverse = (stage == kStageGram);
  if (reverse) std::reverse(order.begin(), order.end());
  int tiles = 0;
  for (size_t i = 0; i < order.size(); ++i) {
    const GPlan& g = *order[i];
    GemmProblem& P = L.prob[i];
    const StageShape ss = stage_shape(g, stage);
    P.batch = g.batch;
    P.m = g.m;
    P.n = g.n;
    P.ldx = g.ldx;
    P.lda = g.lda;
    P.tiles_m = ss.tiles_m;
    P.tiles_n = ss.tiles_n;
    P.tiles_per_mat = ss.tiles_per_mat;
    P.k_blocks = ss.k_blocks;
    P.tile_begin = tiles;
    tiles += ss.tiles_per_mat * g.batch;
    const uint8_t* xc = ws + (cur ? g.x1 : g.x0);
    uint8_t* xn = ws + (cur ? g.x0 : g.x1);
    P.a_mat = reinterpret_cast<const __nv_bfloat16*>(ws + g.am);
    P.parts = reinterpret_cast<const float*>(ws + g.parts);
    P.nparts = g.nparts;
    P.first_round = first_round ? 1 : 0;
    P.reverse = reverse ? 1 : 0;
    bool ok = true;
    // (A and B' hold only the 256 x 256 tiles on or above the diagonal; the
    // 64-row maps read the blocks below them at their transposed positions)
    if (stage == kStageGram) {          // A = s^2 X X^T
      ok = operand_tmap(&L.tm_a[i], xc, g.n, g.m, g.batch, g.ldx, kTileM) &&
           operand_tmap(&L.tm_b[i], xc, g.n, g.m, g.batch, g.ldx, kTileM) &&
           output_tmap(&L.tm_out[i], ws + g.am, g.m, g.m, g.batch, g.lda);
    } else if (stage == kStagePoly) {   // B' = a I + b A + c A A
      ok = operand_tmap(&L.tm_a[i], ws + g.am, g.m, g.m, g.batch, g.lda, kTileM) &&
           operand_tmap(&L.tm_b[i], ws + g.am, g.m, g.m, g.batch, g.lda, kTileM) &&
           operand_tmap(&L.tm_at[i], ws + g.am, g.m, g.m, g.batch, g.lda, 64) &&
           operand_tmap(&L.tm_bt[i], ws + g.am, g.m, g.m, g.batch, g.lda, 64) &&
           output_tmap(&L.tm_out[i], ws + g.bm, g.m, g.m, g.batch, g.lda) &&
           output_tmap(&L.tm_in[i], ws + g.am, g.m, g.m, g.batch, g.lda);
    } else {                            // X' = s B' X
      ok = operand_tmap(&L.tm_a[i], ws + g.bm, g.m, g.m, g.batch, g.lda, kTileM) &&
           operand_tmap(&L.tm_at[i], ws + g.bm, g.m, g.m, g.batch, g.lda, 64) &&
           operand_tmap(&L.tm_b[i], xc, g.n, g.m, g.batch, g.ldx, 64) &&
           output_tmap(&L.tm_out[i], xn, g.n, g.m, g.batch, g.ldx);
      if (signal) {
        P.done_begin = g.ctr;
        P.o_pmajor = g.tall ? 1 : 0;
        if (g.tall)
          ok = ok && make_tmap(&L.tm_out_t[i], xn, g.m, g.n, g.batch, g.lda, 32, 64,
                               CU_TENSOR_MAP_SWIZZLE_NONE);
      }
    }
    if (!ok) return MUON_ERR_CUDA;
  }
  L.n_prob = static_cast<int>(order.size());
  L.total_tiles = tiles;
  L.a = sc.a;
  L.b = sc.b;
  L.c = sc.c;
  L.eps = sc.eps;
  L.status = reinterpret_cast<unsigned int*>(ws);
  if (signal) L.done = reinterpret_cast<unsigned int*>(ws + kStatusBytes);
  return MUON_OK;
}

constexpr double kPersistentRoundUs = 400.0;

double round_mma_us(const std::vector<GPlan*>& chunk, int sms) {
  double kblocks = 0;
  for (const GPlan* g : chunk)
    for (int stage = 0; stage < 3; ++stage) {
      const StageShape ss = stage_shape(*g, stage);
      kblocks += static_cast<double>(g->batch) * ss.tiles_per_mat * ss.k_blocks;
    }
  const double pairs = std::max(1, sms / 2);
  return kblocks * 512.0 / pairs / 1.9e3;
}

// Builds the launch block of the persistent rounds kernel for a chunk of
// tensor-core groups: every stage walks the groups by ascending n and each
// group's matrices in order, so a matrix's next stage follows its current one.
muon_status build_rounds(RoundsLaunch& R, const std::vector<GPlan*>& chunk, const Scalars& sc,
                         uint8_t* ws, bool stream) {
  std::memset(&R, 0, sizeof(R));
  std::vector<GPlan*> order(chunk);
  std::stable_sort(order.begin(), order.end(),
                   [](GPlan* x, GPlan* y) { return x->n < y->n; });
  int begin[3] = {0, 0, 0};
  for (size_t i = 0; i < order.size(); ++i) {
    const GPlan& g = *order[i];
    RoundsProblem& P = R.prob[i];
    P.batch = g.batch;
    P.m = g.m;
    P.n = g.n;
    for (int stage = 0; stage < 3; ++stage) {
      const StageShape ss = stage_shape(g, stage);
      P.tiles_m = ss.tiles_m;
      P.tiles_n[stage] = ss.tiles_n;
      P.tiles_per_mat[stage] = ss.tiles_per_mat;
      P.k_blocks[stage] = ss.k_blocks;
      P.tile_begin[stage] = begin[stage];
      begin[stage] += ss.tiles_per_mat * g.batch;
    }
    P.parts = reinterpret_cast<const float*>(ws + g.parts);
    P.nparts = g.nparts;
    P.done_begin = g.ctr;
    // the streamed apply reads O of a rows > cols matrix as O^T (n x m, row
    // stride lda), written by the last round over that matrix's own X slot
    // (the same size: m and n are multiples of 8)
    P.o_pmajor = (stream && g.tall) ? 1 : 0;
    // ... and, likewise, that matrix's X0 is u as the prologue read it (n x m):
    // the first round reads it transposed (no transpose in the prologue)
    P.x0_u = P.o_pmajor;
    bool ok = true;
    if (P.o_pmajor)
      ok = make_tmap(&R.x_out_t[i], ws + ((sc.steps & 1) ? g.x1 : g.x0), g.m, g.n, g.batch, g.lda,
                     32, 64, CU_TENSOR_MAP_SWIZZLE_NONE) &&
           operand_tmap(&R.u_mn[i], ws + g.x0, g.m, g.n, g.batch, g.lda, 64) &&
           operand_tmap(&R.u_k[i], ws + g.x0, g.m, g.n, g.batch, g.lda, kTileM);
    for (int b = 0; b < 2; ++b) {
      uint8_t* xb = ws + (b ? g.x1 : g.x0);
      ok = ok && operand_tmap(&R.x_op[i][b], xb, g.n, g.m, g.batch, g.ldx, kTileM) &&
           operand_tmap(&R.x_mn[i][b], xb, g.n, g.m, g.batch, g.ldx, 64) &&
           output_tmap(&R.x_out[i][b], xb, g.n, g.m, g.batch, g.ldx);
    }
    ok = ok && operand_tmap(&R.a_op[i], ws + g.am, g.m, g.m, g.batch, g.lda, kTileM) &&
         operand_tmap(&R.a_mn[i], ws + g.am, g.m, g.m, g.batch, g.lda, 64) &&
         output_tmap(&R.a_blk[i], ws + g.am, g.m, g.m, g.batch, g.lda) &&
         operand_tmap(&R.b_op[i], ws + g.bm, g.m, g.m, g.batch, g.lda, kTileM) &&
         operand_tmap(&R.b_mn[i], ws + g.bm, g.m, g.m, g.batch, g.lda, 64) &&
         output_tmap(&R.b_out[i], ws + g.bm, g.m, g.m, g.batch, g.lda);
    if (!ok) return MUON_ERR_CUDA;
  }
  R.n_prob = static_cast<int>(order.size());
  R.steps = sc.steps;
  for (int stage = 0; stage < 3; ++stage) R.stage_tiles[stage] = begin[stage];
  R.round_tiles = begin[0] + begin[1] + begin[2];
  R.total_items = sc.steps * R.round_tiles;
  R.done = reinterpret_cast<unsigned int*>(ws + kStatusBytes);
  R.a = sc.a;
  R.b = sc.b;
  R.c = sc.c;
  R.eps = sc.eps;
  R.status = reinterpret_cast<unsigned int*>(ws);
  return MUON_OK;
}

// ------------------------------------------------------------ the step
// clear_status: zero the workspace's sticky error word on `st` once every
// argument has been checked, before the first launch.
muon_status run_step(std::vector<GPlan>& gs, const Scalars& sc, void* workspace,
                     size_t ws_bytes, cudaStream_t st, bool clear_status = false) {
  muon_status s = check_scalars(sc);
  if (s != MUON_OK) return s;
  for (const GPlan& g : gs) {
    s = check_group(g, sc.mode);
    if (s != MUON_OK) return s;
  }
  const size_t need = plan_workspace(gs);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || ws_bytes < need)
    return MUON_ERR_WORKSPACE;
  bool any = false;
  for (const GPlan& g : gs) any |= g.batch > 0;
  if (!any) return MUON_OK;

  int sms = 0;
  s = current_device(&sms);
  if (s != MUON_OK) return s;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (clear_status && cudaMemsetAsync(ws, 0, sizeof(unsigned int), st) != cudaSuccess)
    return MUON_ERR_CUDA;

  // -- small matrices: one fp32 kernel for all of them, launched first; it lets
  //    the grouped prologue below start at once and run beside it
  bool small_launched = false;
  {
    SmallLaunch sl;
    std::memset(&sl, 0, sizeof(sl));
    sl.mode = sc.mode;
    sl.steps = sc.steps;
    sl.beta = sc.beta;
    sl.a = sc.a;
    sl.b = sc.b;
    sl.c = sc.c;
    sl.eps = sc.eps;
    sl.decay = 1.0f - sc.lr * sc.wd;
    sl.status = reinterpret_cast<const unsigned int*>(ws);
    int blocks = 0, max_mn = 0;
    auto flush = [&]() -> muon_status {
      if (sl.n_groups == 0) return MUON_OK;
      double bytes = 0;
      for (int i = 0; i < sl.n_groups; ++i)
        bytes += static_cast<double>(sl.grp[i].batch) * sl.grp[i].r * sl.grp[i].c *
                 (sc.mode == kPrologueNsOnly ? 6.0 : 20.0);
      sl.x_in_smem = max_mn <= kSmallSmemFloats ? 1 : 0;
      const cudaError_t e = tracked_launch(st, {MUON_K_SMALL_NS, -1, 0.0, bytes},
                                           [&] { return launch_small(sl, blocks, max_mn, st); });
      sl.n_groups = 0;
      blocks = 0;
      max_mn = 0;
      small_launched = true;
      return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
    };
    for (GPlan& g : gs) {
      if (!g.small || g.batch == 0) continue;
      SmallGroup& sg = sl.grp[sl.n_groups++];
      sg.g = g.g;
      sg.buf = g.buf;
      sg.param = g.p;
      sg.out = g.out;
      sg.x = reinterpret_cast<float*>(ws + g.xs);
      sg.gdt = g.gdt;
      sg.batch = g.batch;
      sg.r = g.r;
      sg.c = g.c;
      sg.block_begin = blocks;
      const float scale = g.lr_scale > 0.f ? g.lr_scale
                                            : static_cast<float>(std::sqrt(std::max(
                                                  1.0, static_cast<double>(g.r) / g.c)));
      sg.lr_eff = sc.lr * scale;
      blocks += g.batch;
      max_mn = std::max(max_mn, g.m * g.n);
      if (sl.n_groups == kMaxSmallGroups) {
        s = flush();
        if (s != MUON_OK) return s;
      }
    }
    s = flush();
    if (s != MUON_OK) return s;
  }

  // -- matrices with 64 <= m <= 256 and n <= 512 run their NS rounds in one
  //    kernel (after the grouped prologue, before the grouped apply) when no
  //    matrix of the call needs the staged GEMM launches: the fused kernel and
  //    the staged chain run one after the other, and beside a staged chain the
  //    small matrices cost less as extra tiles of its stages
  auto fusable = [](const GPlan& g) {
    return !g.small && g.m <= kFusedMaxM && g.n <= kFusedMaxN;
  };
  bool fuse = g_fused_enabled.load(std::memory_order_relaxed) != 0;
  for (const GPlan& g : gs)
    if (g.batch > 0 && !g.small && !fusable(g)) fuse = false;
  auto is_fused = [&](const GPlan& g) { return fuse && fusable(g); };

  // -- tensor-core matrices: one grouped prologue launch (per kMaxPrologueGroups)
  std::vector<GPlan*> big;
  for (GPlan& g : gs)
    if (!g.small && g.batch > 0) big.push_back(&g);
  std::vector<GPlan*> staged;
  for (GPlan* g : big)
    if (!is_fused(*g)) staged.push_back(g);
  const int rounds_mode = g_rounds_enabled.load(std::memory_order_relaxed);
  // -- the parameter write streams beside the last update (the persistent rounds
  //    kernel, or the last round's update launch) when one such chunk covers
  //    every tensor-core matrix, every parameter row is whole 16-byte segments,
  //    and O^T of a rows > cols matrix fills its X slot exactly
  bool stream = g_stream_apply_enabled.load(std::memory_order_relaxed) != 0 &&
                sc.mode != kPrologueNsOnly && !big.empty() && staged.size() == big.size() &&
                staged.size() <= static_cast<size_t>(kMaxProblems);
  bool stream_rounds = false;  // ... beside the persistent rounds kernel
  if (stream) {
    const double round_us = round_mma_us(staged, sms);
    stream_rounds = rounds_mode == 1 || (rounds_mode == 2 && round_us < kPersistentRoundUs);
    // (the write's waits give up after 2 s: beside the rounds kernel they span
    // all its rounds, beside the last update launch only that launch, which is
    // bounded here by a whole round)
    if ((stream_rounds ? round_us * sc.steps : round_us) >= kStreamMaxUs) stream = false;
    for (const GPlan* g : big)
      if (g->c % 8 != 0 || (g->tall && (g->m % 8 != 0 || g->n % 8 != 0))) stream = false;
  }
  stream_rounds = stream && stream_rounds;
  for (size_t c0 = 0; c0 < big.size(); c0 += kMaxPrologueGroups) {
    PrologueLaunch pl;
    std::memset(&pl, 0, sizeof(pl));
    pl.beta = sc.beta;
    pl.status = reinterpret_cast<const unsigned int*>(ws);
    double bytes = 0;
    int blocks = 0;
    for (size_t k = c0; k < std::min(big.size(), c0 + kMaxPrologueGroups); ++k) {
      const GPlan& g = *big[k];
      PrologueGroup& pg = pl.grp[pl.n_groups++];
      pg.g = g.g;
      pg.buf = g.buf;
      pg.x = reinterpret_cast<__nv_bfloat16*>(ws + g.x0);
      pg.parts = reinterpret_cast<float*>(ws + g.parts);
      pg.gdt = g.gdt;
      pg.batch = g.batch;
      pg.r = g.r;
      pg.c = g.c;
      // a rows > cols matrix that the streamed rounds kernel reads as u: X0 = u
      // as is, row stride lda (== its cols then)
      pg.pmajor = (stream_rounds && g.tall) ? 1 : 0;
      pg.ldx = pg.pmajor ? g.lda : g.ldx;
      pg.nparts = g.nparts;
      pg.block_begin = blocks;
      blocks += g.batch * g.nparts;
      bytes += static_cast<double>(g.batch) * g.r * g.c *
               ((g.gdt == MUON_BF16 ? 2.0 : 4.0) + 2.0 + (sc.mode == kPrologueNsOnly ? 0.0 : 8.0));
    }
    pl.total_blocks = blocks;
    const bool pdl = small_launched && c0 == 0;
    pl.wait_prior = pdl ? 1 : 0;
    if (c0 == 0) {  // the per-matrix completion counters start at zero
      pl.zero = reinterpret_cast<unsigned int*>(ws + kStatusBytes);
      int n = 0;
      for (const GPlan* g : big) n += g->batch;
      pl.n_zero = n;
      // the streamed apply's claim counter: the status block's second word
      if (stream) pl.zero_work = reinterpret_cast<unsigned int*>(ws) + 1;
    }
    const cudaError_t e = tracked_launch(st, {MUON_K_PROLOGUE, -1, 0.0, bytes},
                                         [&] { return launch_prologue(pl, sc.mode, pdl, st); });
    if (e != cudaSuccess) return MUON_ERR_CUDA;
  }

  // fused NS rounds: one CTA per matrix with m <= 128, a CTA pair for larger m
  for (int pair = 0; pair < 2; ++pair) {
    FusedLaunch fl;
    std::memset(&fl, 0, sizeof(fl));
    fl.pair = pair;
    fl.steps = sc.steps;
    fl.a = sc.a;
    fl.b = sc.b;
    fl.c = sc.c;
    fl.eps = sc.eps;
    fl.status = reinterpret_cast<unsigned int*>(ws);
    double flops = 0;
    auto flush = [&]() -> muon_status {
      if (fl.n_groups == 0) return MUON_OK;
      const cudaError_t e = tracked_launch(st, {MUON_K_FUSED_NS, -1, flops, 0.0},
                                           [&] { return launch_fused(fl, st); });
      fl.n_groups = 0;
      fl.total_clusters = 0;
      flops = 0;
      return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
    };
    for (GPlan* gp : big) {
      const GPlan& g = *gp;
      if (!is_fused(g) || (g.m > kTileM) != (pair == 1)) continue;
      const int i = fl.n_groups++;
      FusedGroup& fg = fl.grp[i];
      fg.parts = reinterpret_cast<const float*>(ws + g.parts);
      fg.nparts = g.nparts;
      fg.batch = g.batch;
      fg.m = g.m;
      fg.n = g.n;
      fg.cluster_begin = fl.total_clusters;
      if (!operand_tmap(&fl.tm_x[i][0], ws + g.x0, g.n, g.m, g.batch, g.ldx, kTileM) ||
          !operand_tmap(&fl.tm_x[i][1], ws + g.x1, g.n, g.m, g.batch, g.ldx, kTileM))
        return MUON_ERR_CUDA;
      fl.total_clusters += g.batch;
      const double mm = g.m, nn = g.n;
      flops += static_cast<double>(g.batch) * sc.steps * (4.0 * mm * mm * nn + 2.0 * mm * mm * mm);
      if (fl.n_groups == kMaxFusedGroups) {
        s = flush();
        if (s != MUON_OK) return s;
      }
    }
    s = flush();
    if (s != MUON_OK) return s;
  }

  for (size_t c0 = 0; c0 < staged.size(); c0 += kMaxProblems) {
    std::vector<GPlan*> chunk(staged.begin() + c0,
                              staged.begin() + std::min(staged.size(), c0 + kMaxProblems));
    const bool persistent =
        rounds_mode == 1 || (rounds_mode == 2 && round_mma_us(chunk, sms) < kPersistentRoundUs);
    if (persistent) {
      RoundsLaunch R;
      s = build_rounds(R, chunk, sc, ws, stream_rounds);
      if (s != MUON_OK) return s;
      if (R.total_items == 0) continue;
      double flops = 0;
      for (GPlan* g : chunk)
        for (int stage = 0; stage < 3; ++stage) flops += stage_flops(*g, stage);
      flops *= sc.steps;
      const cudaError_t e = tracked_launch(st, {MUON_K_ROUNDS, -1, flops, 0.0},
                                           [&] { return launch_rounds(R, sms, st); });
      if (e != cudaSuccess) return MUON_ERR_CUDA;
      continue;
    }
    for (int it = 0; it < sc.steps; ++it) {
      const int cur = it & 1;
      const bool first = (it == 0);
      const int stages[3] = {kStageGram, kStagePoly, kStageUpdate};
      for (int stage : stages) {
        GemmLaunch L;
        s = build_gemm(L, chunk, stage, cur, first, sc, ws,
                       stream && it == sc.steps - 1 && stage == kStageUpdate);
        if (s != MUON_OK) return s;
        if (L.total_tiles == 0) continue;
        double flops = 0;
        for (GPlan* g : chunk) flops += stage_flops(*g, stage);
        const int kind = stage == kStageGram   ? MUON_K_GRAM
                         : stage == kStagePoly ? MUON_K_POLY
                                               : MUON_K_UPDATE;
        const cudaError_t e =
            tracked_launch(st, {kind, it, flops, 0.0},
                           [&] { return launch_gemm(L, stage, L.total_tiles, sms, st); });
        if (e != cudaSuccess) return MUON_ERR_CUDA;
      }
    }
  }

  auto lr_eff = [&](const GPlan& g) {
    const float scale = g.lr_scale > 0.f ? g.lr_scale
                                         : static_cast<float>(std::sqrt(std::max(
                                               1.0, static_cast<double>(g.r) / g.c)));
    return sc.lr * scale;
  };
  if (stream) {
    // -- apply, streamed: matrices in the order the last update finishes them
    //    (ascending n, as build_rounds orders its problems and build_gemm walks
    //    the update stage)
    std::vector<GPlan*> order(big);
    std::stable_sort(order.begin(), order.end(),
                     [](GPlan* x, GPlan* y) { return x->n < y->n; });
    ApplyLaunch al;
    std::memset(&al, 0, sizeof(al));
    double bytes = 0;
    int units = 0;
    for (GPlan* gp : order) {
      const GPlan& g = *gp;
      ApplyGroup& ag = al.grp[al.n_groups++];
      ag.o = reinterpret_cast<const __nv_bfloat16*>(ws + ((sc.steps & 1) ? g.x1 : g.x0));
      ag.param = g.p;
      ag.batch = g.batch;
      ag.r = g.r;
      ag.c = g.c;
      ag.ldx = g.tall ? g.lda : g.ldx;  // O^T (n x m) or O = X (m x n)
      ag.lr_eff = lr_eff(g);
      ag.decay = 1.0f - sc.lr * sc.wd;
      ag.done_begin = g.ctr;
      unsigned int per_round = 0;
      for (int stage = 0; stage < 3; ++stage)
        per_round += static_cast<unsigned int>(stage_shape(g, stage).tiles_per_mat);
      // the value the counter ends with: every tile of every round (rounds
      // kernel) or of the last update launch
      ag.done_target = (stream_rounds ? static_cast<unsigned int>(sc.steps) * per_round
                                      : static_cast<unsigned int>(
                                            stage_shape(g, kStageUpdate).tiles_per_mat)) *
                       kRoundsSignalsPerTile;
      ag.unit_rows = std::max(1, 8192 / g.c);
      ag.units_per_mat = cdiv(g.r, ag.unit_rows);
      ag.unit_begin = units;
      units += g.batch * ag.units_per_mat;
      bytes += static_cast<double>(g.batch) * g.r * g.c * 10.0;
    }
    al.total_units = units;
    al.done = reinterpret_cast<const unsigned int*>(ws + kStatusBytes);
    al.work = reinterpret_cast<unsigned int*>(ws) + 1;
    al.status = reinterpret_cast<unsigned int*>(ws);
    const int blocks = std::max(1, std::min(sms * 8, units));
    const cudaError_t e = tracked_launch(st, {MUON_K_APPLY, -1, 0.0, bytes},
                                         [&] { return launch_apply_stream(al, blocks, st); });
    return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
  }

  // -- apply: p <- (1 - lr wd) p - lr rescale O (or O as bf16), one grouped launch;
  //    after round `steps` the result sits in X1 if steps is odd, else in X0
  for (size_t c0 = 0; c0 < big.size(); c0 += kMaxPrologueGroups) {
    ApplyLaunch al;
    std::memset(&al, 0, sizeof(al));
    al.status = reinterpret_cast<unsigned int*>(ws);
    double bytes = 0;
    int blocks = 0;
    const size_t c1 = std::min(big.size(), c0 + kMaxPrologueGroups);
    for (size_t k = c1; k-- > c0;) {  // the last update's final groups first
      const GPlan& g = *big[k];
      ApplyGroup& ag = al.grp[al.n_groups++];
      ag.o = reinterpret_cast<const __nv_bfloat16*>(ws + ((sc.steps & 1) ? g.x1 : g.x0));
      ag.param = g.p;
      ag.out = g.out;
      ag.batch = g.batch;
      ag.r = g.r;
      ag.c = g.c;
      ag.ldx = g.ldx;
      ag.nparts = g.nparts;
      ag.block_begin = blocks;
      ag.lr_eff = lr_eff(g);
      ag.decay = 1.0f - sc.lr * sc.wd;
      blocks += g.batch * g.nparts;
      bytes += static_cast<double>(g.batch) * g.r * g.c *
               (sc.mode == kPrologueNsOnly ? 4.0 : 10.0);
    }
    al.total_blocks = blocks;
    const bool to_param = sc.mode != kPrologueNsOnly;
    const cudaError_t e = tracked_launch(st, {MUON_K_APPLY, -1, 0.0, bytes},
                                         [&] { return launch_apply(al, to_param, st); });
    if (e != cudaSuccess) return MUON_ERR_CUDA;
  }
  return MUON_OK;
}

GPlan make_plan(float* p, const void* g, int gdt, float* buf, __nv_bfloat16* out, int batch,
                int r, int c, float lr_scale) {
  GPlan x;
  x.p = p;
  x.g = g;
  x.gdt = gdt;
  x.buf = buf;
  x.out = out;
  x.batch = batch;
  x.r = r;
  x.c = c;
  x.lr_scale = lr_scale;
  return x;
}

}  // namespace

namespace muon {

muon_status step_clearing_status(float* params, const void* grads, int g_dtype,
                                 float* momentum_buf, int batch, int rows, int cols,
                                 float momentum, int nesterov, float lr, float weight_decay,
                                 float lr_scale, int steps, float a, float b, float c, float eps,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  try {
    std::vector<GPlan> gs{make_plan(params, grads, g_dtype, momentum_buf, nullptr, batch, rows,
                                    cols, lr_scale)};
    const Scalars sc{nesterov ? kPrologueNesterov : kProloguePlain, momentum, lr, weight_decay,
                     steps, a, b, c, eps};
    return run_step(gs, sc, workspace, workspace_bytes, static_cast<cudaStream_t>(stream), true);
  } catch (...) {
    return MUON_ERR_CUDA;
  }
}

}  // namespace muon

// ============================================================ C ABI
extern "C" {

size_t muon_workspace_bytes(int batch, int rows, int cols) {
  if (!shape_ok(batch, rows, cols)) return 0;
  std::vector<GPlan> gs{make_plan(nullptr, nullptr, MUON_BF16, nullptr, nullptr, batch, rows,
                                  cols, 0.f)};
  return plan_workspace(gs);
}

size_t muon_grouped_workspace_bytes(const muon_group* groups, int n_groups) {
  if (n_groups < 0 || (n_groups > 0 && !groups)) return 0;
  std::vector<GPlan> gs;
  for (int i = 0; i < n_groups; ++i) {
    const muon_group& g = groups[i];
    if (!shape_ok(g.batch, g.rows, g.cols)) return 0;
    gs.push_back(make_plan(nullptr, nullptr, g.g_dtype, nullptr, nullptr, g.batch, g.rows,
                           g.cols, g.lr_scale));
  }
  return plan_workspace(gs);
}

muon_status muon_ns5(const void* G, int g_dtype, void* out_bf16, int batch, int rows, int cols,
                     int steps, float a, float b, float c, float eps, void* workspace,
                     size_t workspace_bytes, void* stream) {
  try {
    std::vector<GPlan> gs{make_plan(nullptr, G, g_dtype, nullptr,
                                    static_cast<__nv_bfloat16*>(out_bf16), batch, rows, cols,
                                    0.f)};
    const Scalars sc{kPrologueNsOnly, 0.f, 0.f, 0.f, steps, a, b, c, eps};
    return run_step(gs, sc, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
  } catch (...) {
    return MUON_ERR_CUDA;
  }
}

muon_status muon_step(float* params, const void* grads, int g_dtype, float* momentum_buf,
                      int batch, int rows, int cols, float momentum, int nesterov, float lr,
                      float weight_decay, float lr_scale, int steps, float a, float b, float c,
                      float eps, void* workspace, size_t workspace_bytes, void* stream) {
  try {
    std::vector<GPlan> gs{make_plan(params, grads, g_dtype, momentum_buf, nullptr, batch, rows,
                                    cols, lr_scale)};
    const Scalars sc{nesterov ? kPrologueNesterov : kProloguePlain, momentum, lr, weight_decay,
                     steps, a, b, c, eps};
    return run_step(gs, sc, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
  } catch (...) {
    return MUON_ERR_CUDA;
  }
}

muon_status muon_step_grouped(const muon_group* groups, int n_groups, float momentum,
                              int nesterov, float lr, float weight_decay, int steps, float a,
                              float b, float c, float eps, void* workspace,
                              size_t workspace_bytes, void* stream) {
  try {
    if (n_groups < 0 || (n_groups > 0 && !groups)) return MUON_ERR_INVALID_ARG;
    std::vector<GPlan> gs;
    gs.reserve(n_groups);
    for (int i = 0; i < n_groups; ++i) {
      const muon_group& g = groups[i];
      gs.push_back(make_plan(g.params, g.grads, g.g_dtype, g.momentum_buf, nullptr, g.batch,
                             g.rows, g.cols, g.lr_scale));
    }
    const Scalars sc{nesterov ? kPrologueNesterov : kProloguePlain, momentum, lr, weight_decay,
                     steps, a, b, c, eps};
    return run_step(gs, sc, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
  } catch (...) {
    return MUON_ERR_CUDA;
  }
}

muon_status muon_workspace_status(const void* workspace, size_t workspace_bytes, void* stream,
                                  int clear) {
  if (!workspace || workspace_bytes < kStatusBytes ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MUON_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned int word = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MUON_ERR_CUDA;
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MUON_ERR_CUDA;
  if (clear && cudaMemsetAsync(const_cast<void*>(workspace), 0, sizeof(word), st) != cudaSuccess)
    return MUON_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MUON_ERR_CUDA;
  return word ? MUON_ERR_TIMEOUT : MUON_OK;
}

muon_status muon_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int limit_us,
                                       void* stream) {
  if (limit_us < 1 || limit_us > 100000) return MUON_ERR_INVALID_ARG;
  if (workspace && (workspace_bytes < kStatusBytes ||
                    (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
    return MUON_ERR_WORKSPACE;
  int sms = 0;
  muon_status s = current_device(&sms);
  if (s != MUON_OK) return s;
  if (!workspace) {
    // the built-in scratch of muon_step_noalloc on the current device
    s = noalloc_scratch(&workspace, &workspace_bytes);
    if (s != MUON_OK) return s;
  }
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t e = launch_wait_selftest(static_cast<unsigned int*>(workspace),
                                             1000ull * static_cast<unsigned long long>(limit_us),
                                             st);
  g_launch_count.fetch_add(1, std::memory_order_relaxed);
  return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}

muon_status muon_adam_step(const muon_adam_tensor* tensors, int n_tensors, int step, float lr,
                           float beta1, float beta2, float eps, float weight_decay,
                           void* stream) {
  try {
    if (n_tensors < 0 || (n_tensors > 0 && !tensors) || step < 1) return MUON_ERR_INVALID_ARG;
    if (!(beta1 >= 0.f && beta1 < 1.f) || !(beta2 >= 0.f && beta2 < 1.f) ||
        !(eps >= 0.f && std::isfinite(eps)) || !std::isfinite(lr) ||
        !std::isfinite(weight_decay))
      return MUON_ERR_INVALID_ARG;
    long long work = 0;
    for (int i = 0; i < n_tensors; ++i) {
      const muon_adam_tensor& t = tensors[i];
      if (t.numel < 0) return MUON_ERR_INVALID_ARG;
      if (t.numel == 0) continue;
      work += t.numel;
      if (t.g_dtype != MUON_F32 && t.g_dtype != MUON_BF16) return MUON_ERR_INVALID_ARG;
      if (!t.param || !t.grad || !t.exp_avg || !t.exp_avg_sq || !aligned16(t.param) ||
          !aligned16(t.grad) || !aligned16(t.exp_avg) || !aligned16(t.exp_avg_sq))
        return MUON_ERR_INVALID_ARG;
      if (!(t.lr_scale >= 0.f && std::isfinite(t.lr_scale)) || !std::isfinite(t.wd_scale))
        return MUON_ERR_INVALID_ARG;
    }
    if (work == 0) return MUON_OK;  // nothing to update: nothing is enqueued
    int sms = 0;
    const muon_status ds = current_device(&sms);
    if (ds != MUON_OK) return ds;
    const int per_sm = adam_blocks_per_sm();
    if (per_sm < 1) return MUON_ERR_CUDA;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    // bias corrections in double, as the page computes them in Python floats
    const double bias1 = 1.0 - std::pow(static_cast<double>(beta1), step);
    const double bias2 = 1.0 - std::pow(static_cast<double>(beta2), step);
    AdamLaunch L;
    std::memset(&L, 0, sizeof(L));
    L.beta1 = beta1;
    L.beta2 = beta2;
    L.eps = eps;
    double bytes = 0.0;
    auto flush = [&]() -> muon_status {
      if (L.n_tensors == 0) return MUON_OK;
      const long long blocks = std::min<long long>(L.total_units, 1ll * sms * per_sm);
      const cudaError_t e = tracked_launch(st, {MUON_K_ADAM, -1, 0.0, bytes}, [&] {
        return launch_adam(L, static_cast<int>(blocks), st);
      });
      L.n_tensors = 0;
      L.total_units = 0;
      bytes = 0.0;
      return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
    };
    for (int i = 0; i < n_tensors; ++i) {
      const muon_adam_tensor& t = tensors[i];
      if (t.numel == 0) continue;
      const double lr_eff = static_cast<double>(lr) * t.lr_scale;
      AdamTensor& a = L.t[L.n_tensors++];
      a.p = t.param;
      a.g = t.grad;
      a.m = t.exp_avg;
      a.v = t.exp_avg_sq;
      a.n = t.numel;
      a.unit_begin = L.total_units;
      a.step_size = static_cast<float>(lr_eff * (std::sqrt(bias2) / bias1));
      a.decay = weight_decay != 0.f
                    ? static_cast<float>(1.0 - lr_eff * weight_decay * t.wd_scale)
                    : 1.f;
      a.g_bf16 = t.g_dtype == MUON_BF16;
      L.total_units += (t.numel + kAdamUnit - 1) / kAdamUnit;
      bytes += static_cast<double>(t.numel) * (24 + (a.g_bf16 ? 2 : 4));
      if (L.n_tensors == kMaxAdamTensors) {
        const muon_status fs = flush();
        if (fs != MUON_OK) return fs;
      }
    }
    return flush();
  } catch (...) {
    return MUON_ERR_CUDA;
  }
}

const char* muon_status_string(muon_status status) {
  switch (status) {
    case MUON_OK:
      return "ok";
    case MUON_ERR_INVALID_ARG:
      return "invalid argument";
    case MUON_ERR_UNSUPPORTED:
      return "unsupported device or shape (needs an sm_103a GPU)";
    case MUON_ERR_CUDA:
      return "CUDA error";
    case MUON_ERR_TIMEOUT:
      return "a bounded device-side wait timed out";
    case MUON_ERR_WORKSPACE:
      return "workspace missing, misaligned or too small";
  }
  return "unknown status";
}

int muon_set_persistent_rounds(int enable) {
  if (enable < 0 || enable > 2) return -1;
  return g_rounds_enabled.exchange(enable);
}

int muon_set_streamed_apply(int enable) {
  return g_stream_apply_enabled.exchange(enable ? 1 : 0);
}

int muon_set_fused_ns(int enable) {
  if (enable != 0 && enable != 1) return -1;
  return g_fused_enabled.exchange(enable);
}

unsigned long long muon_kernel_launch_count(void) {
  return g_launch_count.load(std::memory_order_relaxed);
}

muon_status muon_trace_begin(int max_launches) {
  if (max_launches < 0) return MUON_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  for (TraceSlot& t : g_trace) {
    if (t.e0) cudaEventDestroy(t.e0);
    if (t.e1) cudaEventDestroy(t.e1);
  }
  g_trace.clear();
  g_trace.reserve(max_launches);
  g_trace_cap = max_launches;
  g_trace_on = true;
  return MUON_OK;
}

muon_status muon_trace_end(muon_trace_record* out, int max_records, int* count) {
  if (max_records < 0 || (max_records > 0 && !out)) return MUON_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on = false;
  muon_status st = MUON_OK;
  int n = 0;
  for (TraceSlot& t : g_trace) {
    if (n < max_records) {
      float ms = 0.f;
      if (cudaEventSynchronize(t.e1) != cudaSuccess ||
          cudaEventElapsedTime(&ms, t.e0, t.e1) != cudaSuccess)
        st = MUON_ERR_CUDA;
      out[n].kind = t.kind;
      out[n].round = t.round;
      out[n].ms = ms;
      out[n].flops = t.flops;
      out[n].bytes = t.bytes;
      ++n;
    }
    cudaEventDestroy(t.e0);
    cudaEventDestroy(t.e1);
  }
  g_trace.clear();
  if (count) *count = n;
  return st;
}

}  // extern "C"
