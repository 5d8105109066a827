// internal.h -- argument blocks shared by the host planner and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/muon_gb300.h"

namespace muon {

constexpr int kTileM = 128;       // GEMM tile rows (UMMA M)
constexpr int kTileK = 64;        // bf16 elements per 128-byte swizzle row
constexpr int kSmallMaxM = 63;    // min(rows, cols) below 64 takes the fp32 path
constexpr int kMaxParts = 256;    // norm partial sums per matrix
constexpr int kMaxProblems = 8;   // groups per grouped GEMM launch
constexpr int kMaxSmallGroups = 16;
constexpr int kMaxPrologueGroups = 16;
constexpr int kSmallSmemFloats = 40960;  // X of a small matrix kept in shared memory up to 160 KB

// Bits of the sticky device error word (first word of the workspace).
enum DeviceError : unsigned int {
  kErrTimeoutProducer = 1u,
  kErrTimeoutMma = 2u,
  kErrTimeoutEpilogue = 4u,
  kErrTimeoutDrain = 8u,
  kErrTimeoutFused = 16u,
  kErrTimeoutDepend = 32u,
  kErrTimeoutApply = 64u,
};

// What the prologue computes from (g, buf).
enum PrologueMode : int {
  kPrologueNsOnly = 0,       // u = g (muon_ns5)
  kPrologueNesterov = 1,     // buf <- lerp(buf, g, 1-beta); u = lerp(g, buf, beta)
  kProloguePlain = 2,        // buf <- lerp(buf, g, 1-beta); u = buf
};

// One tensor-core group of the grouped prologue launch.
struct PrologueGroup {
  const void* g;          // [batch, r, c] fp32 or bf16
  float* buf;             // [batch, r, c] fp32 (unused in kPrologueNsOnly)
  __nv_bfloat16* x;       // [batch, m, ldx] bf16: u, or u^T when r > c
  float* parts;           // [batch, nparts] partial sums of u^2
  int gdt;
  int batch, r, c, ldx;
  int nparts;             // blocks per matrix (<= kMaxParts)
  int block_begin;        // first block of this group in the launch
  int pmajor;             // rows > cols, but X = u as is (the rounds kernel's first
                          // round reads it transposed), row stride ldx
};

struct PrologueLaunch {
  PrologueGroup grp[kMaxPrologueGroups];
  int n_groups;
  int total_blocks;
  float beta;
  int wait_prior;         // 1: block 0 waits for the preceding grid (PDL) before exiting
  unsigned int* zero;     // counters the launch zeroes (block 0), or null
  int n_zero;
  unsigned int* zero_work;  // the streamed apply's claim counter, zeroed by block 0 (or null)
  const unsigned int* status;  // sticky device error word: set at entry, the launch does nothing
};

// One tensor-core group of the grouped apply launch: the NS result O (bf16,
// [batch, m, ldx], transposed when rows > cols) goes into the parameter,
// p <- decay p - lr_eff O, or into a bf16 output, in the input's orientation.
struct ApplyGroup {
  const __nv_bfloat16* o;
  float* param;
  __nv_bfloat16* out;
  int batch, r, c, ldx;
  int nparts;
  int block_begin;
  float lr_eff, decay;
  // streamed form: O is in the parameter's orientation (r x c, row stride ldx),
  // matrix z may be written once its completion counter done[done_begin + z]
  // reaches done_target; its rows are split into units of unit_rows rows
  int done_begin;
  unsigned int done_target;
  int unit_rows, units_per_mat;
  int unit_begin;         // first work unit of this group
};

struct ApplyLaunch {
  ApplyGroup grp[kMaxPrologueGroups];
  int n_groups;
  int total_blocks;
  // streamed form (apply_stream_kernel), launched beside the persistent rounds
  // kernel: warps claim units in order from *work and wait for their matrix
  const unsigned int* done;
  unsigned int* work;
  unsigned int* status;   // sticky device error word: set at entry, the launch does
                          // nothing; set later, it ends the streamed form's waits
  int total_units;
};

// One group of the fp32 small-matrix path.
struct SmallGroup {
  const void* g;
  float* buf;
  float* param;           // step mode
  __nv_bfloat16* out;     // ns5 mode
  float* x;               // workspace [batch, m, n] fp32
  int gdt;                // muon_dtype
  int batch, r, c;
  int block_begin;        // first block index of this group in the launch
  float lr_eff;           // lr * rescale
};

struct SmallLaunch {
  SmallGroup grp[kMaxSmallGroups];
  int n_groups;
  int x_in_smem;          // 1: X lives in dynamic shared memory (m*n <= kSmallSmemFloats)
  int mode;               // PrologueMode
  int steps;
  float beta, a, b, c, eps, decay;
  const unsigned int* status;  // sticky device error word: set at entry, the launch does nothing
};

struct GemmProblem {
  int batch, m, n;        // X is m x n (m <= n), batch matrices
  int ldx, lda;           // padded leading dimensions (elements) of X and A/B
  int tiles_m;            // pair rows: ceil(ceil(m / 128) / 2)
  int tiles_n;            // 256-wide tile columns of this stage's output
  int tiles_per_mat;      // pair tiles per matrix
  int tile_begin;         // first linear pair-tile index of this problem
  int k_blocks;           // ceil(K / kTileK)
  const __nv_bfloat16* a_mat;   // poly: A (b A term)
  const float* parts;           // norm partials [batch, nparts]
  int nparts;
  int first_round;              // fold s = 1/(||u||_F + eps) in
  int reverse;                  // walk this problem's matrices in descending order
  // last update before a streamed parameter write (GemmLaunch::done set): the
  // problem's first matrix counter, and whether O goes out transposed (tm_out_t)
  int done_begin;
  int o_pmajor;
};

struct GemmLaunch {
  CUtensorMap tm_a[kMaxProblems];   // operand A tiles (box 64 x 128, 128-byte swizzle)
  CUtensorMap tm_b[kMaxProblems];   // operand B half tiles (box 64 x 128, or 64 x 64 for X)
  CUtensorMap tm_at[kMaxProblems];  // symmetric operand A read transposed (box 64 x 64)
  CUtensorMap tm_bt[kMaxProblems];  // Poly: symmetric operand B read transposed (box 64 x 64)
  CUtensorMap tm_out[kMaxProblems]; // output blocks (box 64 x 32 bf16, 128-byte swizzle)
  CUtensorMap tm_in[kMaxProblems];  // Poly: blocks of A for the b A term (box 64 x 32, 128-byte swizzle)
  CUtensorMap tm_out_t[kMaxProblems];  // o_pmajor: O^T blocks of 64 rows x 32 (as x_out_t below)
  GemmProblem prob[kMaxProblems];
  int n_prob;
  int total_tiles;                  // pair tiles
  float a, b, c, eps;
  unsigned int* status;             // sticky device error word
  // update launch of the last round with the parameter write streamed beside it:
  // per-matrix completion counters (zeroed by the prologue), advanced like the
  // rounds kernel's, which the write waits on; null otherwise
  unsigned int* done;
};

enum GemmStage : int { kStageGram = 0, kStagePoly = 1, kStageUpdate = 2 };

// ---- all NS rounds of a chunk of groups in one persistent launch (ns_gemm.cu)
// Work items are the pair tiles of every (round, stage), in round-major, then
// stage, then problem, matrix and tile order; a tile of stage s of round r of a
// matrix starts once every tile of the stages before it (of that matrix) is
// stored, which per-matrix completion counters in the workspace track.
struct RoundsProblem {
  int batch, m, n;
  int tiles_m;            // pair rows: ceil(ceil(m / 128) / 2)
  int tiles_n[3];         // 256-wide tile columns of each stage's output
  int tiles_per_mat[3];   // pair tiles per matrix in each stage
  int tile_begin[3];      // first tile of this problem within each stage
  int k_blocks[3];        // ceil(K / kTileK) per stage
  const float* parts;     // norm partials [batch, nparts]
  int nparts;
  int done_begin;         // this problem's first matrix counter
  int o_pmajor;           // the last round stores O transposed (x_out_t): the parameter's
                          // orientation of a rows > cols matrix, for the streamed apply
  int x0_u;               // X0 of this rows > cols matrix is u as stored (n x m, row stride
                          // round_up(m, 8)): the first round reads it through u_mn / u_k
};

struct RoundsLaunch {
  CUtensorMap x_op[kMaxProblems][2];   // X buffer 0/1 as K-major operand (box 64 x 128)
  CUtensorMap x_mn[kMaxProblems][2];   // X buffer 0/1 as MN-major operand (box 64 x 64)
  CUtensorMap x_out[kMaxProblems][2];  // X buffer 0/1 output blocks (64 x 32, 128-byte swizzle)
  CUtensorMap a_op[kMaxProblems];      // A (box 64 x 128)
  CUtensorMap a_mn[kMaxProblems];      // A read transposed (box 64 x 64)
  CUtensorMap a_blk[kMaxProblems];     // A 64 x 32 blocks (Gram output, Poly b A input)
  CUtensorMap b_op[kMaxProblems];      // B' (box 64 x 128)
  CUtensorMap b_mn[kMaxProblems];      // B' read transposed (box 64 x 64)
  CUtensorMap b_out[kMaxProblems];     // B' 64 x 32 output blocks
  CUtensorMap x_out_t[kMaxProblems];   // o_pmajor: O^T (n x m, row stride round_up(m, 8)) in
                                       // the last round's output buffer, blocks of 64 rows x 32
  CUtensorMap u_mn[kMaxProblems];      // x0_u: u (n x m) as the Gram's MN-major operands (64 x 64)
  CUtensorMap u_k[kMaxProblems];       // x0_u: u as the update's K-major operand B (64 x 128)
  RoundsProblem prob[kMaxProblems];
  int n_prob;
  int steps;
  int stage_tiles[3];     // pair tiles of one stage over all problems
  int round_tiles;        // sum of stage_tiles
  int total_items;        // steps * round_tiles
  unsigned int* done;     // per-matrix completion counters, zeroed by the prologue
  float a, b, c, eps;
  unsigned int* status;   // sticky device error word
};

// ---- fused NS kernel for 64 <= m <= 256, n <= 512 (ns_fused.cu): all rounds
// of one matrix on one CTA pair; X0 and the norm partials come from the
// grouped prologue, the result O goes where the staged path leaves it
constexpr int kFusedMaxM = 256;
constexpr int kFusedMaxN = 512;
constexpr int kMaxFusedGroups = 16;

struct FusedGroup {
  const float* parts;   // [batch, nparts] partial sums of u^2
  int nparts;
  int batch, m, n;
  int cluster_begin;    // first matrix (CTA pair, or CTA) of this group in the launch
};

struct FusedLaunch {
  // bf16 [batch][m][ldx] X buffers 0 and 1 (SW128, 64 x 128 boxes): round it
  // reads buffer it & 1 and writes buffer (it + 1) & 1
  CUtensorMap tm_x[kMaxFusedGroups][2];
  FusedGroup grp[kMaxFusedGroups];
  int n_groups;
  int total_clusters;   // matrices in the launch
  int pair;             // 1: a CTA pair per matrix (m <= 256); 0: one CTA (m <= 128)
  int steps;
  float a, b, c, eps;
  unsigned int* status;
};

// ---- DistAdam update (adam.cu)
constexpr int kAdamUnit = 4096;       // elements per work unit (256 threads x 4 float4)
constexpr int kMaxAdamTensors = 64;   // tensors per launch

struct AdamTensor {
  float* p;
  const void* g;
  float* m;
  float* v;
  long long n;           // elements
  long long unit_begin;  // first unit of this tensor in the launch
  float step_size;       // lr_eff * sqrt(1 - b2^t) / (1 - b1^t)
  float decay;           // 1 - lr_eff * wd * wd_scale (1 when wd == 0)
  int g_bf16;
};

struct AdamLaunch {
  AdamTensor t[kMaxAdamTensors];
  int n_tensors;
  long long total_units;
  float beta1, beta2, eps;
};

// Launchers (defined next to their kernels).  Each returns a cudaError_t from
// the launch; grid sizes come from the caller's SM count.
// The prologue may be launched as a programmatic dependent of the kernel
// before it (pdl = true): it then overlaps that kernel and waits for it only
// before exiting.
cudaError_t launch_prologue(const PrologueLaunch& l, int mode, bool pdl, cudaStream_t s);
cudaError_t launch_small(const SmallLaunch& l, int total_blocks, int max_mn, cudaStream_t s);
cudaError_t launch_apply(const ApplyLaunch& l, bool to_param, cudaStream_t s);
// The streamed parameter write (ApplyLaunch streamed fields), a programmatic
// dependent of the last update launch, `blocks` CTAs of 256 threads.
cudaError_t launch_apply_stream(const ApplyLaunch& l, int blocks, cudaStream_t s);
constexpr unsigned int kRoundsSignalsPerTile = 8;  // completion-counter adds per stored pair tile
// One launch of a GEMM stage over `pair_tiles` cluster tiles (two 128 x 256
// CTA tiles each); the grid is sized from the device's SM count.
cudaError_t launch_gemm(const GemmLaunch& l, int stage, int pair_tiles, int sms, cudaStream_t s);
// All rounds of the problems of `l` in one launch (grid sized from the SM count).
cudaError_t launch_rounds(const RoundsLaunch& l, int sms, cudaStream_t s);
int gemm_smem_bytes();
cudaError_t launch_wait_selftest(unsigned int* status, unsigned long long limit_ns,
                                 cudaStream_t s);
cudaError_t launch_adam(const AdamLaunch& l, int blocks, cudaStream_t s);
// One CTA pair (l.pair) or one CTA per matrix of every group in `l`, launched as a programmatic
// dependent of the kernel before it (the prologue), whose output it reads
// after griddepcontrol.wait.
cudaError_t launch_fused(const FusedLaunch& l, cudaStream_t s);
int adam_blocks_per_sm();  // resident Adam blocks per SM on the current device (0 on error)

// muon_step whose workspace's sticky error word is cleared on the stream after
// the argument checks and before the first kernel (muon_api.cu).
muon_status step_clearing_status(float* params, const void* grads, int g_dtype,
                                 float* momentum_buf, int batch, int rows, int cols,
                                 float momentum, int nesterov, float lr, float weight_decay,
                                 float lr_scale, int steps, float a, float b, float c, float eps,
                                 void* workspace, size_t workspace_bytes, void* stream);
// Device address and size of the built-in scratch of muon_step_noalloc on the
// current device (noalloc.cu).
muon_status noalloc_scratch(void** out, size_t* bytes);

}  // namespace muon
