// ns_gemm.cu -- the three GEMM stages of one quintic Newton-Schulz round on
// sm_103a tensor cores ("parameter-golf train_gpt.py 源码精读", part 1,
// section 核心思想: A = X X^T; B = b A + c A A; X = a X + B X):
//
//   Gram    A = s^2 X X^T      (s = 1/(||u||_F + eps) on the first round, else 1)
//   Poly    B' = a I + b A + c A A
//   Update  X' = s B' X  (= s (a X + B X))
//
// (The parameter write that follows the last round is the elementwise apply
// kernel in prologue.cu.)
// Folding a I into the polynomial's output makes the update a plain GEMM with
// no X operand in its epilogue; rounding a + B_ii to bf16 once was checked to
// cost no accuracy against adding a X in fp32.
//
// X is m x n (m <= n) bf16, row-major with padded leading dimension; A and B
// are m x m bf16.  A and B are symmetric, so Gram and Poly compute and store
// only the 256 x 256 pair tiles on or above the diagonal (diagonal tiles
// whole); nothing is ever written below them.  A consumer that needs a block
// below (rows of pair row p, a K block in pair column q < p) loads the block
// at the transposed position with TMA and hands it to the tensor cores as an
// MN-major operand (the descriptor's major bit per k-block), so the stored
// upper tiles serve both.  For A A the second operand A[k][j] = A[j][k] is read
// the same way; the Update's X operand (contraction over X's rows) is always
// MN-major.
//
// Kernel shape: persistent clusters of two CTAs (a CTA pair), one CTA per SM,
// 192 threads (224 in the rounds kernel, whose warp 6 schedules, below):
//   warp 0      TMA producer (one lane) into a ring of swizzled smem stages
//   warp 1      TMEM allocator; in the even CTA also the tcgen05.mma issuer
//   warps 2..5  epilogue: tcgen05.ld of the fp32 accumulator, fp32 math, 32 x 64
//               blocks staged in shared memory and written by TMA bulk stores
// The pair computes a 256 x 256 tile with cta_group::2 MMAs (M = 256): CTA r
// holds tile rows 2p + r (128 rows of A) and the r-th 128-column half of B in
// its own shared memory, and receives its 128 rows of the result in its own
// TMEM.  Each SM therefore receives 32 KB of operands per 64-deep k-block for
// 128 x 256 x 64 of MMA work.  Both CTAs' copies complete on the even CTA's
// stage barrier; its MMA commits free the slot in both CTAs; both CTAs'
// epilogue warps release the accumulator on the even CTA's barrier.  With
// 256-wide tile columns the two rows of a pair have the same set of
// upper-triangle tiles, so symmetric stages pair up exactly.  The accumulator
// is double buffered in TMEM so the epilogue of one tile overlaps the MMAs of
// the next.
//
// Two kernels share these roles, tile by tile:
//   ns_gemm_kernel<stage>  one stage of one round over a chunk of groups (one
//                          launch per stage, chained by programmatic
//                          dependent launch)
//   ns_rounds_kernel       every stage of every round of a chunk of groups in
//                          one launch: a tile waits for the per-matrix
//                          completion counter of the stages before it, which
//                          the epilogue warps advance once their stores of a
//                          tile are complete, so one matrix's next stage can
//                          start while other matrices still finish the current
//                          one.  A seventh warp (the scheduler) decodes the
//                          tiles and does these waits, and hands ready tiles to
//                          the producer through a small queue, so that the
//                          producer only issues copies.
#include "internal.h"
#include "ptx.cuh"

namespace muon {

// Shared memory per CTA: the operand ring, the epilogue staging slots, barriers.
struct Cfg {
  static constexpr int kBN = 256;                        // pair tile: 256 x 256
  // 5 measured faster than 6 on every workload (GPT-2 124M 1048 -> 1040 us,
  // d=512 241 -> 237 us, d=2048 31.7 -> 31.4 ms) and than 4 on all but d=512
  static constexpr int kStages = 5;
  static constexpr int kABytes = kTileM * kTileK * 2;    // 16 KB: 128 rows x 128 B
  static constexpr int kBBytes = (kBN / 2) * kTileK * 2; // 16 KB: this CTA's half of B
  static constexpr int kStageBytes = kABytes + kBBytes;  // 32 KB
  static constexpr int kTmemCols = 2 * kBN;              // two 128 x 256 fp32 accumulators
  static constexpr int kEpiWarps = 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kRoundsThreads = kThreads + 32;   // + the scheduler warp
  static constexpr int kQueue = 8;                        // ready tiles scheduler -> producer
  static constexpr int kSlots = 2;                       // per epilogue warp
  static constexpr int kSlotBytes = 4096;                // one 32 x 64 bf16 block
  static constexpr int kStagingBytes = kEpiWarps * kSlots * kSlotBytes;
  static constexpr int kBarBytes = 512;
  static constexpr int kSmem = kStages * kStageBytes + kStagingBytes + kBarBytes + 1024;
  // completion-counter increments per stored pair tile: every epilogue warp of both CTAs
  static constexpr unsigned int kSignalsPerTile = 2 * kEpiWarps;
};
static_assert(Cfg::kSignalsPerTile == kRoundsSignalsPerTile, "the host computes the final counts");

// Everything a role needs to know about one pair tile.
struct TileCtx {
  const CUtensorMap* a;    // operand A, K-major boxes of 64 x 128
  const CUtensorMap* at;   // operand A read transposed (symmetric A), boxes of 64 x 64
  const CUtensorMap* b;    // operand B: K-major 64 x 128 (Gram, Poly) or 64 x 64 (Update, X)
  const CUtensorMap* bt;   // Poly: operand B read transposed, 64 x 64
  const CUtensorMap* out;  // output 32 x 64 blocks
  const CUtensorMap* out_t;  // update: O^T in 64 x 32 blocks instead of `out` (or null)
  const CUtensorMap* in;   // Poly: A 32 x 64 blocks (the b A term)
  int mat, pr, tn;         // matrix, pair row (pr >= tiles_m: no rows), tile column
  int m, n, k_blocks;
  const float* parts;      // first round: norm partials of the batch
  int nparts;
  int first_round;
  // first round of a rows > cols matrix whose X0 is u as stored: the Gram reads
  // both operands MN-major through `at`/`bt`, the update operand B K-major
  // through `b`
  int x0_u;
};

struct GemmScalars {
  float a, b, c, eps;
};

// Whether the k-block kb of an operand whose rows lie in pair row `pr` falls
// below the stored upper tiles of a symmetric matrix (its pair column kb / 4 is
// left of the diagonal), so it is read transposed.  Operand A is symmetric in
// Poly (A) and Update (B'); operand B only in Poly.
template <int STAGE>
__device__ __forceinline__ bool a_transposed(int pr, int kb) {
  return STAGE != kStageGram && pr > (kb * kTileK) / 256;
}
template <int STAGE>
__device__ __forceinline__ bool b_transposed(int pr, int kb) {
  return STAGE == kStagePoly && pr > (kb * kTileK) / 256;
}

// Operand majors of k-block kb of a tile.
template <int STAGE>
__device__ __forceinline__ bool a_mn_major(const TileCtx& T, int kb) {
  return STAGE == kStageGram ? T.x0_u != 0 : a_transposed<STAGE>(T.pr, kb);
}
template <int STAGE>
__device__ __forceinline__ bool b_mn_major(const TileCtx& T, int kb) {
  if (STAGE == kStageUpdate) return T.x0_u == 0;
  return STAGE == kStageGram ? T.x0_u != 0 : b_transposed<STAGE>(T.tn, kb);
}

// A diagonal tile of a symmetric stage (Gram X X^T, Poly A A): each CTA's half
// of operand B is the same 128 rows, in the same layout, as its operand A, so
// only A is loaded and the MMAs read it for B too.
template <int STAGE>
__device__ __forceinline__ bool b_is_a(const TileCtx& T) {
  return STAGE != kStageUpdate && T.pr == T.tn;
}

// How a role gives up: the CTA's abort flag (ends every wait of the CTA's
// other roles), the peer CTA's abort flag (shared::cluster address; ends the
// pair's waits at once) and the launch's sticky status word in global memory
// (ends, after a short delay, every wait of every other CTA, and makes later
// kernels on this workspace return at entry).
struct Abort {
  volatile int* flag;
  uint32_t peer_flag;
  unsigned int* status;
};

__device__ __forceinline__ void record_failure(const Abort& ab, unsigned int bit) {
  *ab.flag = 1;
  ptx::st_cluster_u32(ab.peer_flag, 1u);
  atomicOr(ab.status, bit);
}

__device__ __forceinline__ int first_tile() { return blockIdx.x >> 1; }
__device__ __forceinline__ int tile_stride() { return gridDim.x >> 1; }

// ------------------------------------------------------------ producer
struct ProdState {
  int stage = 0;
  uint32_t phase = 0;
  uint32_t armed = 0, armed_parity = 0;  // slots with copies issued, and their phase
};

// Issues the k-blocks of one tile into the ring.  False on a timed-out wait.
template <int STAGE>
__device__ bool produce_tile(const TileCtx& T, uint8_t* smem, uint64_t* full, uint64_t* empty,
                             uint32_t leader_full0, ProdState& ps, const Abort& ab, int rank) {
  using C = Cfg;
  const int tm = 2 * T.pr + rank;  // this CTA's 128-row block
  const bool b_from_a = b_is_a<STAGE>(T);
  for (int kb = 0; kb < T.k_blocks; ++kb) {
    // the pair's MMAs (issued by the even CTA) are done with this slot
    if (!ptx::mbar_wait(&empty[ps.stage], ps.phase ^ 1u, ab.flag, ab.status)) return false;
    uint8_t* sa = smem + ps.stage * C::kStageBytes;
    uint8_t* sb = sa + C::kABytes;
    // both CTAs' copies complete on the even CTA's barrier for this slot
    const uint32_t bar = leader_full0 + ps.stage * 8;
    if (rank == 0)
      ptx::mbar_arrive_expect_tx(&full[ps.stage],
                                 2 * (b_from_a ? C::kABytes : C::kStageBytes));
    // operand A: this CTA's 128 rows x 64 k-columns, or (below the stored
    // tiles) the 64 x 128 block at the transposed position, MN-major
    if (a_mn_major<STAGE>(T, kb)) {
#pragma unroll
      for (int q = 0; q < 2; ++q)
        ptx::tma_load_3d_pair(sa + q * (64 * kTileK * 2), T.at, tm * kTileM + q * 64,
                              kb * kTileK, T.mat, bar);
    } else {
      ptx::tma_load_3d_pair(sa, T.a, kb * kTileK, tm * kTileM, T.mat, bar);
    }
    if (b_from_a) {
      // (the MMAs read operand B from operand A's slot)
    } else if (b_mn_major<STAGE>(T, kb)) {
      // operand B = X[k][j] (update), or the transposed block (Poly below the
      // stored tiles, a first-round Gram of u), MN-major: this CTA's 128
      // columns as 2 slabs of 64 columns x 64 k-rows
      const CUtensorMap* map = STAGE >= kStageUpdate ? T.b : T.bt;
#pragma unroll
      for (int q = 0; q < 2; ++q)
        ptx::tma_load_3d_pair(sb + q * (64 * kTileK * 2), map,
                              T.tn * C::kBN + rank * kTileM + q * 64, kb * kTileK, T.mat, bar);
    } else {
      // operand B: this CTA's 128 of the tile column's 256 rows, K-major
      ptx::tma_load_3d_pair(sb, T.b, kb * kTileK, T.tn * C::kBN + rank * kTileM, T.mat, bar);
    }
    ps.armed |= 1u << ps.stage;
    ps.armed_parity = (ps.armed_parity & ~(1u << ps.stage)) | (ps.phase << ps.stage);
    if (++ps.stage == C::kStages) {
      ps.stage = 0;
      ps.phase ^= 1u;
    }
  }
  return true;
}

// Before exit: the pair's MMAs have released every armed stage, so its copies
// landed and no commit arrival can still be on its way to this CTA.  After a
// failure those releases may never come; the copies themselves land within
// microseconds, so all stages share one bounded window (not one each).
__device__ void drain_producer(const ProdState& ps, uint64_t* empty, const Abort& ab) {
  const uint64_t t0 = ptx::globaltimer();
  for (int s = 0; s < Cfg::kStages; ++s) {
    if (!(ps.armed & (1u << s))) continue;
    const uint64_t spent = ptx::globaltimer() - t0;
    if (spent >= ptx::kWaitTimeoutNs ||
        !ptx::mbar_wait(&empty[s], (ps.armed_parity >> s) & 1u, nullptr, nullptr,
                        ptx::kWaitTimeoutNs - spent)) {
      record_failure(ab, kErrTimeoutDrain);
      return;
    }
  }
}

// ------------------------------------------------------------ MMA issuer
// Runs in the even CTA of the pair only.
struct MmaState {
  int stage = 0;
  uint32_t phase = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
};

template <int STAGE>
__device__ bool mma_tile(const TileCtx& T, uint8_t* smem, uint64_t* full, uint64_t* empty,
                         uint64_t* acc_full, uint64_t* acc_empty, uint32_t tmem_base,
                         MmaState& ms, const Abort& ab) {
  using C = Cfg;
  // both CTAs' epilogues have drained this accumulator
  if (!ptx::mbar_wait(&acc_empty[ms.acc], ms.acc_phase ^ 1u, ab.flag, ab.status)) return false;
  ptx::tc_fence_after();
  const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(ms.acc * C::kBN);
  for (int kb = 0; kb < T.k_blocks; ++kb) {
    // (the barrier orders the TMA writes before these MMA reads; no tcgen05
    // fence is needed here)
    if (!ptx::mbar_wait(&full[ms.stage], ms.phase, ab.flag, ab.status)) return false;
    const uint32_t sa = ptx::smem_u32(smem + ms.stage * C::kStageBytes);
    const bool b_from_a = b_is_a<STAGE>(T);
    const uint32_t sb = b_from_a ? sa : sa + C::kABytes;
    const bool a_mn = a_mn_major<STAGE>(T, kb);
    const bool b_mn = b_from_a ? a_mn : b_mn_major<STAGE>(T, kb);
    const uint32_t idesc = ptx::idesc_bf16(2 * kTileM, C::kBN, b_mn, a_mn);
#pragma unroll
    for (int k = 0; k < kTileK / 16; ++k) {
      // K-major SW128: 8-row groups 1024 B apart; a K=16 slice is 32 B on.
      // MN-major SW128: 64-column slabs (64 x 128 B) apart along M or N,
      // 8-row groups 1024 B apart along K; a K=16 slice is 16 rows = 2048 B on.
      const uint64_t da = a_mn ? ptx::smem_desc_sw128(sa + k * 2048, 64 * kTileK * 2, 1024)
                               : ptx::smem_desc_sw128(sa + k * 32, 16, 1024);
      const uint64_t db = b_mn ? ptx::smem_desc_sw128(sb + k * 2048, 64 * kTileK * 2, 1024)
                               : ptx::smem_desc_sw128(sb + k * 32, 16, 1024);
      ptx::mma_bf16_pair(d_tmem, da, db, idesc, (kb | k) != 0 ? 1u : 0u);
    }
    // frees the slot in both CTAs once these MMAs have read it
    ptx::mma_commit_pair(&empty[ms.stage]);
    if (++ms.stage == C::kStages) {
      ms.stage = 0;
      ms.phase ^= 1u;
    }
  }
  ptx::mma_commit_pair(&acc_full[ms.acc]);
  if (++ms.acc == 2) {
    ms.acc = 0;
    ms.acc_phase ^= 1u;
  }
  return true;
}

// Every MMA issued by this thread completes before TMEM is released.
__device__ void drain_mma(uint64_t* drain, const Abort& ab) {
  ptx::mma_commit_pair(drain, 1);
  if (!ptx::mbar_wait(drain, 0, nullptr)) record_failure(ab, kErrTimeoutDrain);
}

// ------------------------------------------------------------ epilogue helpers
__device__ __forceinline__ float inv_fro_norm(const float* parts, int nparts, float eps,
                                              int lane) {
  float acc = 0.f;
  for (int k = lane; k < nparts; k += 32) acc += parts[k];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return 1.0f / (sqrtf(acc) + eps);
}

// bf16 halves of a packed pair as floats (bf16 is the top half of an fp32).
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b2);
}

// Output staging.  Each epilogue warp owns kSlots 4 KB slots used in turn,
// each holding the warp's 32 x 64 block of the output, bf16, 128-byte rows
// with the 128-byte swizzle TMA expects (16-byte unit u of row r sits at unit
// u ^ (r & 7)), written with 16-byte stores and stored to global memory by one
// TMA bulk store.  Poly first loads its A block into the slot by TMA.  (Blocks
// of 32 x 64 rather than 32 x 32 halve the bulk copies a tile issues.)
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((((c >> 3) ^ r) & 7) << 4) + (c & 7) * 2);
}

// Columns 32 h .. 32 h + 31 of row r.
__device__ __forceinline__ void stage_half_sw128(uint8_t* blk, int r, int h,
                                                 const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 w = make_uint4(pack_bf2(v[8 * q + 0], v[8 * q + 1]),
                               pack_bf2(v[8 * q + 2], v[8 * q + 3]),
                               pack_bf2(v[8 * q + 4], v[8 * q + 5]),
                               pack_bf2(v[8 * q + 6], v[8 * q + 7]));
    *reinterpret_cast<uint4*>(blk + sw128(r, 32 * h + 8 * q)) = w;
  }
}

// ------------------------------------------------------------ epilogue warps
// Warp w (2..5) owns TMEM lanes 32*(w&3).. (32 rows of the 128-row tile) and
// walks the tile's 256 columns in 4 units of 64 (two 32-column TMEM loads each).
struct EpiState {
  int acc = 0;
  uint32_t acc_phase = 0;
  int slot = 0;         // next staging slot (alternating)
  uint32_t in_par = 0;  // Poly: parity of each slot's next input load
};

// One tile.  `dep`/`dep_target` (Poly in the rounds kernel): the counter the
// A blocks of the b A term wait for before lane 0 loads them.  False on a
// timed-out wait.
template <int STAGE>
__device__ bool epilogue_tile(const TileCtx& T, const GemmScalars& k, uint64_t* acc_full,
                              uint64_t* acc_empty, uint64_t* my_in, uint8_t* my_slots,
                              uint32_t tmem_base, EpiState& es, const Abort& ab,
                              int quarter, int lane, int rank, const unsigned int* dep,
                              unsigned int dep_target) {
  using C = Cfg;
  static_assert(C::kSlots == 2, "the staging slots alternate");
  constexpr int kUnits = C::kBN / 64;
  constexpr bool kSym = STAGE <= kStagePoly;
  constexpr bool kPoly = STAGE == kStagePoly;
  __syncwarp();
  float s = 1.f;
  if (STAGE != kStagePoly && T.first_round)
    s = inv_fro_norm(T.parts + static_cast<size_t>(T.mat) * T.nparts, T.nparts, k.eps, lane);
  const int tm = 2 * T.pr + rank;
  const int i0 = tm * kTileM + quarter * 32;  // first row of this warp
  const int ncols = kSym ? T.m : T.n;
  const int jt = T.tn * C::kBN;
  // live units: rows in range, columns in range
  const int u_hi = i0 < T.m ? min(kUnits, (ncols - jt + 63) / 64) : 0;
  // Poly: the first two live units' A blocks into the two slots
  if constexpr (kPoly) {
    int ok = 1;
    if (lane == 0 && u_hi > 0) {
      if (dep != nullptr) {
        if (!ptx::wait_counter(dep, dep_target, ab.flag, ab.status)) ok = 0;
        ptx::fence_proxy_async_global();
      }
      if (ok) {
        // both slots' earlier stores have read their data
        ptx::bulk_wait_read<0>();
        for (int q = 0; q < 2 && q < u_hi; ++q) {
          const int sl = es.slot ^ q;
          ptx::mbar_arrive_expect_tx(&my_in[sl], C::kSlotBytes);
          ptx::tma_load_3d(my_slots + sl * C::kSlotBytes, T.in, jt + 64 * q, i0, T.mat,
                           &my_in[sl]);
        }
      }
    }
    if (__shfl_sync(0xffffffffu, ok, 0) == 0) return false;
  }

  const bool got = ptx::mbar_wait(&acc_full[es.acc], es.acc_phase, ab.flag, ab.status);
  __syncwarp();
  if (!got) return false;
  ptx::tc_fence_after();
  const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                         static_cast<uint32_t>(es.acc * C::kBN);
  bool failed = false;
#pragma unroll 1
  for (int u = 0; u < u_hi; ++u) {
    const int j0 = jt + u * 64;
    uint8_t* blk = my_slots + es.slot * C::kSlotBytes;
    if constexpr (kPoly) {
      const uint32_t par = (es.in_par >> es.slot) & 1u;
      if (!ptx::mbar_wait(&my_in[es.slot], par, ab.flag, ab.status)) failed = true;
      es.in_par ^= 1u << es.slot;
    } else {
      // the slot's previous bulk store (two units ago) has read its data
      if (lane == 0) ptx::bulk_wait_read<C::kSlots - 1>();
    }
    __syncwarp();
    if (STAGE == kStageUpdate && T.out_t != nullptr) {
      // O^T, the parameter's orientation of a rows > cols matrix: the block of
      // rows j0.. (64) and columns i0.. (32), 64-byte rows, lane l writing
      // column l (its TMEM row)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t v[32];
        ptx::tmem_ld32_sync(tbase + static_cast<uint32_t>(u * 64 + h * 32), v);
#pragma unroll
        for (int q = 0; q < 32; ++q)
          *reinterpret_cast<__nv_bfloat16*>(blk + (32 * h + q) * 64 + lane * 2) =
              __float2bfloat16_rn(s * __uint_as_float(v[q]));
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::tma_store_3d(T.out_t, i0, j0, T.mat, blk);
        ptx::bulk_commit();
      }
      es.slot ^= 1;
      continue;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t v[32];
      ptx::tmem_ld32_sync(tbase + static_cast<uint32_t>(u * 64 + h * 32), v);
      float val[32];
      if constexpr (STAGE == kStageGram) {
#pragma unroll
        for (int q = 0; q < 32; ++q) val[q] = __uint_as_float(v[q]) * (s * s);
      } else if constexpr (kPoly) {
        // row `lane`, columns 32 h.. of the A block (each lane reads and then
        // overwrites only its own row)
        uint32_t ev[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 w = *reinterpret_cast<const uint4*>(blk + sw128(lane, 32 * h + 8 * q));
          ev[4 * q + 0] = w.x;
          ev[4 * q + 1] = w.y;
          ev[4 * q + 2] = w.z;
          ev[4 * q + 3] = w.w;
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          val[2 * q] = fmaf(k.c, __uint_as_float(v[2 * q]), k.b * bf_lo(ev[q]));
          val[2 * q + 1] = fmaf(k.c, __uint_as_float(v[2 * q + 1]), k.b * bf_hi(ev[q]));
        }
        // B' = a I + b A + c A A: the update then needs no a X term
        if (j0 + 32 * h == i0) {
#pragma unroll
          for (int q = 0; q < 32; ++q) val[q] += (q == lane) ? k.a : 0.f;
        }
      } else {
#pragma unroll
        for (int q = 0; q < 32; ++q) val[q] = s * __uint_as_float(v[q]);
      }
      stage_half_sw128(blk, lane, h, val);
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      ptx::tma_store_3d(T.out, j0, i0, T.mat, blk);
      ptx::bulk_commit();
      // Poly: the A block two units ahead goes into this slot once the store
      // just issued has read it
      if (kPoly && u + 2 < u_hi) {
        ptx::bulk_wait_read<0>();
        ptx::mbar_arrive_expect_tx(&my_in[es.slot], C::kSlotBytes);
        ptx::tma_load_3d(blk, T.in, j0 + 128, i0, T.mat, &my_in[es.slot]);
      }
    }
    es.slot ^= 1;
  }
  ptx::tc_fence_before();
  __syncwarp();
  // release the accumulator on the even CTA's barrier (the MMA issuer's)
  if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&acc_empty[es.acc]), 0));
  if (++es.acc == 2) {
    es.acc = 0;
    es.acc_phase ^= 1u;
  }
  return !failed;
}

// ------------------------------------------------------------ common setup
struct Smem {
  uint8_t* ring;
  uint8_t* staging;
  uint64_t *full, *empty, *acc_full, *acc_empty, *drain, *in_bar;
  uint64_t *q_full, *q_empty;  // rounds kernel: the ready-tile queue
  uint32_t* tmem_slot;
  volatile int* abort_flag;
};

__device__ __forceinline__ Smem carve_smem(uint8_t* smem_raw) {
  using C = Cfg;
  Smem m;
  // both CTAs of the pair get the same aligned offsets (the pair MMA reads both)
  m.ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  m.staging = m.ring + C::kStages * C::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(m.staging + C::kStagingBytes);
  m.full = bars;
  m.empty = bars + C::kStages;
  m.acc_full = bars + 2 * C::kStages;
  m.acc_empty = m.acc_full + 2;
  m.drain = m.acc_empty + 2;
  m.in_bar = m.drain + 1;  // Poly: one per epilogue warp and slot
  m.q_full = m.in_bar + C::kEpiWarps * C::kSlots;
  m.q_empty = m.q_full + C::kQueue;
  m.tmem_slot = reinterpret_cast<uint32_t*>(m.q_empty + C::kQueue);
  m.abort_flag = reinterpret_cast<volatile int*>(m.tmem_slot + 1);
  return m;
}

// Barriers, TMEM; returns the TMEM base.  Called by every thread of both CTAs.
__device__ __forceinline__ uint32_t setup_cta(const Smem& m, int warp) {
  using C = Cfg;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(&m.full[s], 1);   // the even CTA's expect_tx (+ both CTAs' bytes)
      ptx::mbar_init(&m.empty[s], 1);  // the pair MMA commit
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&m.acc_full[s], 1);
      ptx::mbar_init(&m.acc_empty[s], 2 * C::kEpiWarps);  // both CTAs' epilogue warps
    }
    ptx::mbar_init(m.drain, 1);
    for (int k = 0; k < C::kEpiWarps * C::kSlots; ++k) ptx::mbar_init(&m.in_bar[k], 1);
    for (int k = 0; k < C::kQueue; ++k) {
      ptx::mbar_init(&m.q_full[k], 1);   // the scheduler, entry written
      ptx::mbar_init(&m.q_empty[k], 1);  // the producer, entry read
    }
    *m.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(m.tmem_slot, C::kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  __syncwarp();
  ptx::tc_fence_before();
  // both CTAs' barriers exist before either's copies signal the other's
  ptx::cluster_sync();
  ptx::tc_fence_after();
  return *m.tmem_slot;
}

// The pair's abort context (after setup_cta).
__device__ __forceinline__ Abort pair_abort(const Smem& m, unsigned int* status, int rank) {
  Abort ab;
  ab.flag = m.abort_flag;
  ab.peer_flag = ptx::mapa_shared(ptx::smem_u32((const void*)m.abort_flag),
                                  static_cast<uint32_t>(rank ^ 1));
  ab.status = status;
  return ab;
}

// Called by every thread of both CTAs once the previous grid's output is
// visible (after griddep_wait): true if the status word already records a
// failure (an earlier kernel on this workspace gave up, or a CTA of this
// launch did), in which case the pair does no work at all.  Both CTAs read the
// word and raise both flags, and the cluster barrier makes the decision common
// to the pair, so neither CTA runs roles that wait on roles the other skips.
__device__ __forceinline__ bool skip_at_entry(const Abort& ab) {
  if (threadIdx.x == 0 && ptx::status_set(ab.status)) {
    *ab.flag = 1;
    ptx::st_cluster_u32(ab.peer_flag, 1u);
  }
  ptx::cluster_sync();
  return *ab.flag != 0;
}

__device__ __forceinline__ void teardown_cta(uint32_t tmem_base, int warp) {
  __syncwarp();
  ptx::tc_fence_before();
  // neither CTA exits while the other may still write into its shared memory
  // or arrive on its barriers
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
  }
}

// ============================================================ staged kernel
struct Tile {
  int prob, mat, pr, tn;
};

// Linear pair-tile index -> (problem, matrix, pair row, tile col).
// Symmetric stages enumerate, per pair row p, the tile columns tn >= p.
template <int STAGE>
__device__ __forceinline__ Tile decode_tile(const GemmLaunch& L, int t) {
  int p = 0;
#pragma unroll 1
  while (p + 1 < L.n_prob && t >= L.prob[p + 1].tile_begin) ++p;
  const GemmProblem& P = L.prob[p];
  const int local = t - P.tile_begin;
  Tile r;
  r.prob = p;
  r.mat = local / P.tiles_per_mat;
  int w = local - r.mat * P.tiles_per_mat;
  if (P.reverse) r.mat = P.batch - 1 - r.mat;
  r.pr = P.tiles_m;  // out of range unless found (no stores then)
  r.tn = 0;
  if (STAGE >= kStageUpdate) {
    // column by column: the tiles of one column share their X panel (256
    // columns, all K rows), which L2 can then serve to the pair rows after the
    // first, while B' (m x m) stays in L2 across columns.  On the d=4096 model
    // (4096 x 11008 matrices, 90 MB of X each) an update launch moved 65 GB of
    // DRAM traffic row by row and 56 GB column by column, against 30 GB of
    // operands and results, and the step took 5 % less time.
    r.tn = w / P.tiles_m;
    r.pr = w - r.tn * P.tiles_m;
  } else {
#pragma unroll 1
    for (int q = 0; q < P.tiles_m; ++q) {
      const int cnt = P.tiles_n - q;
      if (w < cnt) {
        r.pr = q;
        r.tn = q + w;
        break;
      }
      w -= cnt;
    }
  }
  return r;
}

__device__ __forceinline__ TileCtx staged_ctx(const GemmLaunch& L, const Tile& tl) {
  const GemmProblem& P = L.prob[tl.prob];
  TileCtx T;
  T.a = &L.tm_a[tl.prob];
  T.at = &L.tm_at[tl.prob];
  T.b = &L.tm_b[tl.prob];
  T.bt = &L.tm_bt[tl.prob];
  T.out = &L.tm_out[tl.prob];
  // (o_pmajor only on the last update before a streamed parameter write)
  T.out_t = P.o_pmajor ? &L.tm_out_t[tl.prob] : nullptr;
  T.in = &L.tm_in[tl.prob];
  T.mat = tl.mat;
  T.pr = tl.pr;
  T.tn = tl.tn;
  T.m = P.m;
  T.n = P.n;
  T.k_blocks = P.k_blocks;
  T.parts = P.parts;
  T.nparts = P.nparts;
  T.first_round = P.first_round;
  T.x0_u = 0;
  return T;
}

template <int STAGE>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    ns_gemm_kernel(const __grid_constant__ GemmLaunch L) {
  extern __shared__ uint8_t smem_raw[];
  const Smem sm = carve_smem(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(ptx::cluster_ctarank());
  // the next stage may be scheduled now; it takes an SM only once this CTA has
  // left it, and waits for this grid to finish before reading its output
  ptx::griddep_launch_dependents();
  const uint32_t tmem_base = setup_cta(sm, warp);
  // setup above overlapped the previous stage's tail; its output is read below
  ptx::griddep_wait();
  const Abort ab = pair_abort(sm, L.status, rank);
  const bool skip = skip_at_entry(ab);

  if (skip) {
    // an earlier failure on this workspace: nothing is read or written
  } else if (warp == 0) {
    if (lane == 0) {
      for (int p = 0; p < L.n_prob; ++p) {
        ptx::prefetch_tmap(&L.tm_a[p]);
        ptx::prefetch_tmap(&L.tm_b[p]);
        if (STAGE != kStageGram) ptx::prefetch_tmap(&L.tm_at[p]);
        if (STAGE == kStagePoly) ptx::prefetch_tmap(&L.tm_bt[p]);
      }
      ProdState ps;
      const uint32_t leader_full0 = ptx::mapa_shared(ptx::smem_u32(sm.full), 0);
      for (int t = first_tile(); t < L.total_tiles; t += tile_stride()) {
        const TileCtx T = staged_ctx(L, decode_tile<STAGE>(L, t));
        if (!produce_tile<STAGE>(T, sm.ring, sm.full, sm.empty, leader_full0, ps, ab, rank)) {
          record_failure(ab, kErrTimeoutProducer);
          break;
        }
      }
      drain_producer(ps, sm.empty, ab);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      MmaState ms;
      for (int t = first_tile(); t < L.total_tiles; t += tile_stride()) {
        const TileCtx T = staged_ctx(L, decode_tile<STAGE>(L, t));
        if (!mma_tile<STAGE>(T, sm.ring, sm.full, sm.empty, sm.acc_full, sm.acc_empty, tmem_base,
                             ms, ab)) {
          record_failure(ab, kErrTimeoutMma);
          break;
        }
      }
      drain_mma(sm.drain, ab);
    }
  } else {
    const int quarter = warp & 3;
    uint8_t* my_slots = sm.staging + quarter * Cfg::kSlots * Cfg::kSlotBytes;
    uint64_t* my_in = sm.in_bar + quarter * Cfg::kSlots;
    const GemmScalars k{L.a, L.b, L.c, L.eps};
    EpiState es;
    for (int t = first_tile(); t < L.total_tiles; t += tile_stride()) {
      const Tile tl = decode_tile<STAGE>(L, t);
      const TileCtx T = staged_ctx(L, tl);
      if (!epilogue_tile<STAGE>(T, k, sm.acc_full, sm.acc_empty, my_in, my_slots, tmem_base, es,
                                ab, quarter, lane, rank, nullptr, 0u)) {
        record_failure(ab, kErrTimeoutEpilogue);
        break;
      }
      // last update before a streamed parameter write: this warp's blocks of
      // the tile are in global memory, count them for the write
      if (STAGE == kStageUpdate && L.done != nullptr) {
        if (lane == 0) {
          ptx::bulk_wait<0>();
          ptx::fence_proxy_async_global();
          ptx::red_release_gpu_add(L.done + L.prob[tl.prob].done_begin + tl.mat, 1u);
        }
        __syncwarp();
      }
    }
    // all bulk copies of this warp are complete before the CTA exits
    if (lane == 0) ptx::bulk_wait<0>();
    __syncwarp();
  }
  teardown_cta(tmem_base, warp);
}

// ============================================================ rounds kernel
struct Item {
  int r, s, p, mat, pr, tn;
};

// Linear item index -> (round, stage, problem, matrix, pair row, tile col).
__device__ __forceinline__ Item decode_item(const RoundsLaunch& L, int item) {
  Item it;
  it.r = item / L.round_tiles;
  int w = item - it.r * L.round_tiles;
  int s = 0;
  while (s < 2 && w >= L.stage_tiles[s]) {
    w -= L.stage_tiles[s];
    ++s;
  }
  int p = 0;
#pragma unroll 1
  while (p + 1 < L.n_prob && w >= L.prob[p + 1].tile_begin[s]) ++p;
  const RoundsProblem& P = L.prob[p];
  const int local = w - P.tile_begin[s];
  it.s = s;
  it.p = p;
  it.mat = local / P.tiles_per_mat[s];
  int q = local - it.mat * P.tiles_per_mat[s];
  it.pr = P.tiles_m;
  it.tn = 0;
  if (s == kStageUpdate) {
    // column by column, as in the per-stage update (GPT-2 124M step 1029 ->
    // 1022 us against row by row)
    it.tn = q / P.tiles_m;
    it.pr = q - it.tn * P.tiles_m;
  } else {
#pragma unroll 1
    for (int row = 0; row < P.tiles_m; ++row) {
      const int cnt = P.tiles_n[s] - row;
      if (q < cnt) {
        it.pr = row;
        it.tn = row + q;
        break;
      }
      q -= cnt;
    }
  }
  return it;
}

// Completion-counter value that every tile of the stages before `it` (for its
// matrix) has stored.
__device__ __forceinline__ unsigned int dep_target(const RoundsLaunch& L, const Item& it) {
  const RoundsProblem& P = L.prob[it.p];
  const unsigned int per_round = static_cast<unsigned int>(
      P.tiles_per_mat[0] + P.tiles_per_mat[1] + P.tiles_per_mat[2]);
  unsigned int tiles = static_cast<unsigned int>(it.r) * per_round;
  if (it.s >= 1) tiles += P.tiles_per_mat[0];
  if (it.s >= 2) tiles += P.tiles_per_mat[1];
  return tiles * Cfg::kSignalsPerTile;
}

__device__ __forceinline__ TileCtx rounds_ctx(const RoundsLaunch& L, const Item& it) {
  const RoundsProblem& P = L.prob[it.p];
  const int cur = it.r & 1;
  TileCtx T;
  T.out_t = nullptr;
  if (it.s == kStageGram) {          // A = s^2 X X^T
    T.a = &L.x_op[it.p][cur];
    T.at = nullptr;
    T.b = &L.x_op[it.p][cur];
    T.bt = nullptr;
    T.out = &L.a_blk[it.p];
    T.in = nullptr;
  } else if (it.s == kStagePoly) {   // B' = a I + b A + c A A
    T.a = &L.a_op[it.p];
    T.at = &L.a_mn[it.p];
    T.b = &L.a_op[it.p];
    T.bt = &L.a_mn[it.p];
    T.out = &L.b_out[it.p];
    T.in = &L.a_blk[it.p];
  } else {                           // X' = s B' X
    T.a = &L.b_op[it.p];
    T.at = &L.b_mn[it.p];
    T.b = &L.x_mn[it.p][cur];
    T.bt = nullptr;
    T.out = &L.x_out[it.p][cur ^ 1];
    T.in = nullptr;
    // the last round of a matrix whose O the streamed apply reads in the
    // parameter's orientation
    if (P.o_pmajor && it.r == L.steps - 1) T.out_t = &L.x_out_t[it.p];
  }
  T.mat = it.mat;
  T.pr = it.pr;
  T.tn = it.tn;
  T.m = P.m;
  T.n = P.n;
  T.k_blocks = P.k_blocks[it.s];
  T.parts = P.parts;
  T.nparts = P.nparts;
  T.first_round = it.r == 0 ? 1 : 0;
  T.x0_u = (it.r == 0 && P.x0_u) ? 1 : 0;
  if (T.x0_u && it.s == kStageGram) {
    T.at = &L.u_mn[it.p];
    T.bt = &L.u_mn[it.p];
  } else if (T.x0_u && it.s == kStageUpdate) {
    T.b = &L.u_k[it.p];
  }
  return T;
}

// Warps: 0 producer, 1 TMEM and MMA issuer, 2..5 epilogue, 6 scheduler.
__global__ void __launch_bounds__(Cfg::kRoundsThreads, 1)
    ns_rounds_kernel(const __grid_constant__ RoundsLaunch L) {
  extern __shared__ uint8_t smem_raw[];
  // ready tiles: round | stage << 8 | problem << 12, matrix, pair row, tile column
  __shared__ int4 queue[Cfg::kQueue];
  const Smem sm = carve_smem(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(ptx::cluster_ctarank());
  const uint32_t tmem_base = setup_cta(sm, warp);
  // X0, the norm partials and the zeroed counters come from the prologue
  ptx::griddep_wait();
  // the dependent (the streamed apply, which waits on this kernel's counters)
  // may start once every CTA of this grid is resident, and after the prologue
  // has completed (it zeroes the apply's claim counter)
  ptx::griddep_launch_dependents();
  const Abort ab = pair_abort(sm, L.status, rank);
  const bool skip = skip_at_entry(ab);

  if (skip) {
    // an earlier failure on this workspace: nothing is read or written (the
    // streamed write, waiting on this kernel's counters, sees the same word)
  } else if (warp == 0) {
    if (lane == 0) {
      for (int p = 0; p < L.n_prob; ++p) {
        ptx::prefetch_tmap(&L.x_op[p][0]);
        ptx::prefetch_tmap(&L.x_op[p][1]);
        ptx::prefetch_tmap(&L.x_mn[p][0]);
        ptx::prefetch_tmap(&L.x_mn[p][1]);
        ptx::prefetch_tmap(&L.a_op[p]);
        ptx::prefetch_tmap(&L.a_mn[p]);
        ptx::prefetch_tmap(&L.b_op[p]);
        ptx::prefetch_tmap(&L.b_mn[p]);
      }
      ProdState ps;
      const uint32_t leader_full0 = ptx::mapa_shared(ptx::smem_u32(sm.full), 0);
      int n = 0;
      for (int i = first_tile(); i < L.total_items; i += tile_stride(), ++n) {
        const int q = n % Cfg::kQueue;
        if (!ptx::mbar_wait(&sm.q_full[q], static_cast<uint32_t>((n / Cfg::kQueue) & 1),
                            ab.flag, ab.status)) {
          record_failure(ab, kErrTimeoutProducer);
          break;
        }
        const int4 e = queue[q];
        ptx::mbar_arrive(&sm.q_empty[q]);
        Item it;
        it.r = e.x & 0xFF;
        it.s = (e.x >> 8) & 0xF;
        it.p = e.x >> 12;
        it.mat = e.y;
        it.pr = e.z;
        it.tn = e.w;
        // the scheduler acquired the counter of the stages before (its queue
        // barrier passes that on); the operands were stored through the async
        // proxy and are read through it
        ptx::fence_proxy_async_global();
        const TileCtx T = rounds_ctx(L, it);
        bool ok;
        if (it.s == kStageGram)
          ok = produce_tile<kStageGram>(T, sm.ring, sm.full, sm.empty, leader_full0, ps, ab, rank);
        else if (it.s == kStagePoly)
          ok = produce_tile<kStagePoly>(T, sm.ring, sm.full, sm.empty, leader_full0, ps, ab, rank);
        else
          ok = produce_tile<kStageUpdate>(T, sm.ring, sm.full, sm.empty, leader_full0, ps, ab, rank);
        if (!ok) {
          record_failure(ab, kErrTimeoutProducer);
          break;
        }
      }
      drain_producer(ps, sm.empty, ab);
    }
  } else if (warp == 2 + Cfg::kEpiWarps) {
    // scheduler: the tiles in order, each once the stages before it (of its
    // matrix) are stored, into the queue
    if (lane == 0) {
      int n = 0;
      for (int i = first_tile(); i < L.total_items; i += tile_stride(), ++n) {
        const int q = n % Cfg::kQueue;
        if (!ptx::mbar_wait(&sm.q_empty[q], static_cast<uint32_t>(((n / Cfg::kQueue) & 1) ^ 1),
                            ab.flag, ab.status)) {
          record_failure(ab, kErrTimeoutProducer);
          break;
        }
        const Item it = decode_item(L, i);
        const unsigned int target = dep_target(L, it);
        if (target > 0 && !ptx::wait_counter(L.done + L.prob[it.p].done_begin + it.mat, target,
                                             ab.flag, ab.status)) {
          record_failure(ab, kErrTimeoutDepend);
          break;
        }
        queue[q] = make_int4(it.r | (it.s << 8) | (it.p << 12), it.mat, it.pr, it.tn);
        ptx::mbar_arrive(&sm.q_full[q]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      MmaState ms;
      for (int i = first_tile(); i < L.total_items; i += tile_stride()) {
        const Item it = decode_item(L, i);
        const TileCtx T = rounds_ctx(L, it);
        bool ok;
        if (it.s == kStageGram)
          ok = mma_tile<kStageGram>(T, sm.ring, sm.full, sm.empty, sm.acc_full, sm.acc_empty,
                                    tmem_base, ms, ab);
        else if (it.s == kStagePoly)
          ok = mma_tile<kStagePoly>(T, sm.ring, sm.full, sm.empty, sm.acc_full, sm.acc_empty,
                                    tmem_base, ms, ab);
        else
          ok = mma_tile<kStageUpdate>(T, sm.ring, sm.full, sm.empty, sm.acc_full, sm.acc_empty,
                                      tmem_base, ms, ab);
        if (!ok) {
          record_failure(ab, kErrTimeoutMma);
          break;
        }
      }
      drain_mma(sm.drain, ab);
    }
  } else {
    const int quarter = warp & 3;
    uint8_t* my_slots = sm.staging + quarter * Cfg::kSlots * Cfg::kSlotBytes;
    uint64_t* my_in = sm.in_bar + quarter * Cfg::kSlots;
    const GemmScalars k{L.a, L.b, L.c, L.eps};
    EpiState es;
    for (int i = first_tile(); i < L.total_items; i += tile_stride()) {
      const Item it = decode_item(L, i);
      const TileCtx T = rounds_ctx(L, it);
      unsigned int* ctr = L.done + L.prob[it.p].done_begin + it.mat;
      bool ok;
      if (it.s == kStageGram)
        ok = epilogue_tile<kStageGram>(T, k, sm.acc_full, sm.acc_empty, my_in, my_slots,
                                       tmem_base, es, ab, quarter, lane, rank,
                                       nullptr, 0u);
      else if (it.s == kStagePoly)
        ok = epilogue_tile<kStagePoly>(T, k, sm.acc_full, sm.acc_empty, my_in, my_slots,
                                       tmem_base, es, ab, quarter, lane, rank, ctr,
                                       dep_target(L, it));
      else
        ok = epilogue_tile<kStageUpdate>(T, k, sm.acc_full, sm.acc_empty, my_in, my_slots,
                                         tmem_base, es, ab, quarter, lane, rank,
                                         nullptr, 0u);
      if (!ok) {
        record_failure(ab, kErrTimeoutEpilogue);
        break;
      }
      // this warp's blocks of the tile are in global memory: count them
      if (lane == 0) {
        ptx::bulk_wait<0>();
        ptx::fence_proxy_async_global();
        ptx::red_release_gpu_add(ctr, 1u);
      }
      __syncwarp();
    }
    // all bulk copies of this warp are complete before the CTA exits
    if (lane == 0) ptx::bulk_wait<0>();
    __syncwarp();
  }
  teardown_cta(tmem_base, warp);
}

// ------------------------------------------------------------ wait self-test
// One thread waits on a barrier that nothing completes, through the same
// bounded wait the GEMM roles use, with a short limit; the timeout is recorded
// in the status word exactly as a GEMM role records one.
__global__ void wait_selftest_kernel(unsigned int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  ptx::mbar_init(&bar, 1);
  abort_flag = 0;
  ptx::fence_mbar_init();
  if (!ptx::mbar_wait(&bar, 0, &abort_flag, nullptr, limit_ns)) atomicOr(status, kErrTimeoutEpilogue);
  // complete the barrier's phase so nothing is left pending
  ptx::mbar_arrive(&bar);
}

cudaError_t launch_wait_selftest(unsigned int* status, unsigned long long limit_ns,
                                 cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

// ------------------------------------------------------------ launchers
// Clusters that fit on the device at once (one CTA per SM), queried once per
// device and kernel.
template <typename K>
static cudaError_t max_clusters(K kernel, int slot, int threads, int sms, int* out) {
  static int cache[4][64] = {{0}};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (cache[slot][dev] == 0) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = Cfg::kSmem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(2 * (sms / 2));
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
    if (e != cudaSuccess) return e;
    cache[slot][dev] = n < 1 ? 1 : n;
  }
  *out = cache[slot][dev];
  return cudaSuccess;
}

template <typename K, typename P>
static cudaError_t launch_pairs(K kernel, const P& params, int threads, int clusters,
                                cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = Cfg::kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cfg.gridDim = dim3(2 * clusters);
  return cudaLaunchKernelEx(&cfg, kernel, params);
}

template <int STAGE>
static cudaError_t launch_instance(const GemmLaunch& l, int pair_tiles, int sms, cudaStream_t s) {
  int n = 0;
  const cudaError_t e = max_clusters(ns_gemm_kernel<STAGE>, STAGE, Cfg::kThreads, sms, &n);
  if (e != cudaSuccess) return e;
  return launch_pairs(ns_gemm_kernel<STAGE>, l, Cfg::kThreads, pair_tiles < n ? pair_tiles : n,
                      s);
}

int gemm_smem_bytes() { return Cfg::kSmem; }

cudaError_t launch_gemm(const GemmLaunch& l, int stage, int pair_tiles, int sms, cudaStream_t s) {
  switch (stage) {
    case kStageGram:
      return launch_instance<kStageGram>(l, pair_tiles, sms, s);
    case kStagePoly:
      return launch_instance<kStagePoly>(l, pair_tiles, sms, s);
    case kStageUpdate:
      return launch_instance<kStageUpdate>(l, pair_tiles, sms, s);
    default:
      return cudaErrorInvalidValue;
  }
}

// Every cluster of the grid must be resident at once: tiles wait for tiles of
// other clusters.  The grid is therefore never larger than what fits.
cudaError_t launch_rounds(const RoundsLaunch& l, int sms, cudaStream_t s) {
  int n = 0;
  const cudaError_t e = max_clusters(ns_rounds_kernel, 3, Cfg::kRoundsThreads, sms, &n);
  if (e != cudaSuccess) return e;
  return launch_pairs(ns_rounds_kernel, l, Cfg::kRoundsThreads,
                      l.total_items < n ? l.total_items : n, s);
}

}  // namespace muon
