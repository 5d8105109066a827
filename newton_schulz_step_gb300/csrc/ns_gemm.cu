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
// 192 threads:
//   warp 0      TMA producer (one lane) into a ring of swizzled smem stages
//   warp 1      TMEM allocator; in the even CTA also the tcgen05.mma issuer
//   warps 2..5  epilogue: tcgen05.ld of the fp32 accumulator, fp32 math, 32 x 32
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
#include "internal.h"
#include "ptx.cuh"

namespace muon {

// Shared memory per CTA: the operand ring, the epilogue staging slots, barriers.
// Poly reads its b A term through TMA into a third slot per warp.
template <int STAGE>
struct GemmCfg {
  static constexpr int kBN = 256;                        // pair tile: 256 x 256
  static constexpr int kStages = 6;
  static constexpr int kABytes = kTileM * kTileK * 2;    // 16 KB: 128 rows x 128 B
  static constexpr int kBBytes = (kBN / 2) * kTileK * 2; // 16 KB: this CTA's half of B
  static constexpr int kStageBytes = kABytes + kBBytes;  // 32 KB
  static constexpr int kTmemCols = 2 * kBN;              // two 128 x 256 fp32 accumulators
  static constexpr int kEpiWarps = 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kSlots = STAGE == kStagePoly ? 3 : 2;  // per epilogue warp
  static constexpr int kSlotBytes = 2048;                // one 32 x 32 bf16 block
  static constexpr int kStagingBytes = kEpiWarps * kSlots * kSlotBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmem = kStages * kStageBytes + kStagingBytes + kBarBytes + 1024;
};

struct Tile {
  int prob, mat, tm, tn;  // tm: this CTA's tile row (2 * pair row + cluster rank)
};

// Linear pair-tile index -> (problem, matrix, tile row of this CTA, tile col).
// Symmetric stages enumerate, per pair row p, the tile columns tn >= p.
template <int STAGE>
__device__ __forceinline__ Tile decode_tile(const GemmLaunch& L, int t, int rank) {
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
  int tp = P.tiles_m;  // out of range unless found (no stores then)
  if (STAGE >= kStageUpdate) {
    tp = w / P.tiles_n;
    r.tn = w - tp * P.tiles_n;
  } else {
    r.tn = 0;
#pragma unroll 1
    for (int q = 0; q < P.tiles_m; ++q) {
      const int cnt = P.tiles_n - q;
      if (w < cnt) {
        tp = q;
        r.tn = q + w;
        break;
      }
      w -= cnt;
    }
  }
  r.tm = 2 * tp + rank;
  return r;
}

__device__ __forceinline__ void record_failure(const GemmLaunch& L, volatile int* abort_flag,
                                               unsigned int bit) {
  *abort_flag = 1;
  atomicOr(L.status, bit);
}

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

__device__ __forceinline__ int first_tile() { return blockIdx.x >> 1; }
__device__ __forceinline__ int tile_stride() { return gridDim.x >> 1; }

// ------------------------------------------------------------ producer
template <int STAGE>
__device__ void run_producer(const GemmLaunch& L, uint8_t* smem, uint64_t* full, uint64_t* empty,
                             volatile int* abort_flag, int rank) {
  using C = GemmCfg<STAGE>;
  for (int p = 0; p < L.n_prob; ++p) {
    ptx::prefetch_tmap(&L.tm_a[p]);
    ptx::prefetch_tmap(&L.tm_b[p]);
    if (STAGE != kStageGram) ptx::prefetch_tmap(&L.tm_at[p]);
    if (STAGE == kStagePoly) ptx::prefetch_tmap(&L.tm_bt[p]);
  }
  int stage = 0;
  uint32_t phase = 0;
  uint32_t armed = 0, armed_parity = 0;
  bool ok = true;
  const uint32_t leader_full0 = ptx::mapa_shared(ptx::smem_u32(full), 0);
  for (int t = first_tile(); ok && t < L.total_tiles; t += tile_stride()) {
    const Tile tl = decode_tile<STAGE>(L, t, rank);
    const GemmProblem& P = L.prob[tl.prob];
    const CUtensorMap* ta = &L.tm_a[tl.prob];
    const CUtensorMap* tb = &L.tm_b[tl.prob];
    const CUtensorMap* tat = &L.tm_at[tl.prob];
    const CUtensorMap* tbt = &L.tm_bt[tl.prob];
    for (int kb = 0; kb < P.k_blocks; ++kb) {
      // the pair's MMAs (issued by the even CTA) are done with this slot
      if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
        record_failure(L, abort_flag, kErrTimeoutProducer);
        ok = false;
        break;
      }
      uint8_t* sa = smem + stage * C::kStageBytes;
      uint8_t* sb = sa + C::kABytes;
      // both CTAs' copies complete on the even CTA's barrier for this slot
      const uint32_t bar = leader_full0 + stage * 8;
      if (rank == 0) ptx::mbar_arrive_expect_tx(&full[stage], 2 * C::kStageBytes);
      // operand A: this CTA's 128 rows x 64 k-columns, or (below the stored
      // tiles) the 64 x 128 block at the transposed position, MN-major
      if (a_transposed<STAGE>(tl.tm >> 1, kb)) {
#pragma unroll
        for (int q = 0; q < 2; ++q)
          ptx::tma_load_3d_pair(sa + q * (64 * kTileK * 2), tat, tl.tm * kTileM + q * 64,
                                kb * kTileK, tl.mat, bar);
      } else {
        ptx::tma_load_3d_pair(sa, ta, kb * kTileK, tl.tm * kTileM, tl.mat, bar);
      }
      if (STAGE >= kStageUpdate) {
        // operand B = X[k][j], MN-major: this CTA's 128 columns as 2 slabs of
        // 64 columns x 64 k-rows
#pragma unroll
        for (int q = 0; q < 2; ++q)
          ptx::tma_load_3d_pair(sb + q * (64 * kTileK * 2), tb, tl.tn * C::kBN + rank * 128 + q * 64,
                                kb * kTileK, tl.mat, bar);
      } else if (b_transposed<STAGE>(tl.tn, kb)) {
        // Poly, below the stored tiles: the transposed block, MN-major
#pragma unroll
        for (int q = 0; q < 2; ++q)
          ptx::tma_load_3d_pair(sb + q * (64 * kTileK * 2), tbt,
                                tl.tn * C::kBN + rank * kTileM + q * 64, kb * kTileK, tl.mat, bar);
      } else {
        // operand B: this CTA's 128 of the tile column's 256 rows, K-major
        ptx::tma_load_3d_pair(sb, tb, kb * kTileK, tl.tn * C::kBN + rank * kTileM, tl.mat, bar);
      }
      armed |= 1u << stage;
      armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == C::kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  // Before exit: the pair's MMAs have released every armed stage, so its copies
  // landed and no commit arrival can still be on its way to this CTA.
  for (int s = 0; s < C::kStages; ++s)
    if (armed & (1u << s))
      if (!ptx::mbar_wait(&empty[s], (armed_parity >> s) & 1u, nullptr))
        record_failure(L, abort_flag, kErrTimeoutDrain);
}

// ------------------------------------------------------------ MMA issuer
// Runs in the even CTA of the pair only.
template <int STAGE>
__device__ void run_mma(const GemmLaunch& L, uint8_t* smem, uint64_t* full, uint64_t* empty,
                        uint64_t* acc_full, uint64_t* acc_empty, uint64_t* drain,
                        uint32_t tmem_base, volatile int* abort_flag) {
  using C = GemmCfg<STAGE>;
  constexpr bool kBmn = (STAGE >= kStageUpdate);
  int stage = 0;
  uint32_t phase = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  bool ok = true;
  for (int t = first_tile(); ok && t < L.total_tiles; t += tile_stride()) {
    const Tile tl = decode_tile<STAGE>(L, t, 0);
    const int kblocks = L.prob[tl.prob].k_blocks;
    // both CTAs' epilogues have drained this accumulator
    if (!ptx::mbar_wait(&acc_empty[acc], acc_phase ^ 1u, abort_flag)) {
      record_failure(L, abort_flag, kErrTimeoutMma);
      break;
    }
    ptx::tc_fence_after();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::kBN);
    for (int kb = 0; kb < kblocks; ++kb) {
      // (the barrier orders the TMA writes before these MMA reads; no tcgen05
      // fence is needed here)
      if (!ptx::mbar_wait(&full[stage], phase, abort_flag)) {
        record_failure(L, abort_flag, kErrTimeoutMma);
        ok = false;
        break;
      }
      const uint32_t sa = ptx::smem_u32(smem + stage * C::kStageBytes);
      const uint32_t sb = sa + C::kABytes;
      const bool a_mn = a_transposed<STAGE>(tl.tm >> 1, kb);
      const bool b_mn = kBmn || b_transposed<STAGE>(tl.tn, kb);
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
      ptx::mma_commit_pair(&empty[stage]);
      if (++stage == C::kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) break;
    ptx::mma_commit_pair(&acc_full[acc]);
    if (++acc == 2) {
      acc = 0;
      acc_phase ^= 1u;
    }
  }
  // Every MMA issued by this thread completes before TMEM is released.
  ptx::mma_commit_pair(drain, 1);
  if (!ptx::mbar_wait(drain, 0, nullptr)) record_failure(L, abort_flag, kErrTimeoutDrain);
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

// 32 consecutive bf16 of a row (zero past `valid`), kept packed.
__device__ __forceinline__ void load_row32(const __nv_bfloat16* src, int valid,
                                           uint32_t (&w)[16]) {
  if (valid >= 32) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = s4[q];
      w[4 * q + 0] = v.x;
      w[4 * q + 1] = v.y;
      w[4 * q + 2] = v.z;
      w[4 * q + 3] = v.w;
    }
  } else {
    const unsigned short* h = reinterpret_cast<const unsigned short*>(src);
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const uint32_t lo = (2 * t < valid) ? h[2 * t] : 0u;
      const uint32_t hi = (2 * t + 1 < valid) ? h[2 * t + 1] : 0u;
      w[t] = lo | (hi << 16);
    }
  }
}

// Output staging.  Each epilogue warp owns two 4 KB slots used in turn:
//   [0, 2 KB)  the warp's 32 x 32 block of the output, bf16, 64-byte rows with
//              the 64-byte swizzle TMA expects (16-byte unit u of row r sits
//              at unit u ^ ((r >> 1) & 3)), written with 16-byte stores;
//   [2, 4 KB)  the mirrored block (entry (i, j) at row j, column i), bf16, no
//              swizzle: lanes hold consecutive i, so its stores are
//              conflict-free.
// Both are stored to global memory by one TMA bulk store each.
__device__ __forceinline__ uint32_t sw64(int r, int c) {
  return static_cast<uint32_t>(r * 64 + ((((c >> 3) ^ (r >> 1)) & 3) << 4) + (c & 7) * 2);
}

__device__ __forceinline__ void stage_row_sw64(uint8_t* blk, int r, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 w = make_uint4(pack_bf2(v[8 * q + 0], v[8 * q + 1]),
                               pack_bf2(v[8 * q + 2], v[8 * q + 3]),
                               pack_bf2(v[8 * q + 4], v[8 * q + 5]),
                               pack_bf2(v[8 * q + 6], v[8 * q + 7]));
    *reinterpret_cast<uint4*>(blk + sw64(r, 8 * q)) = w;
  }
}

// ------------------------------------------------------------ epilogue warps
// Warp w (2..5) owns TMEM lanes 32*(w&3).. (32 rows of the 128-row tile) and
// walks the tile's 256 columns in 8 chunks of 32.
template <int STAGE>
__device__ void run_epilogue(const GemmLaunch& L, uint64_t* acc_full, uint64_t* acc_empty,
                             uint64_t* in_bar, uint32_t tmem_base, uint8_t* staging,
                             volatile int* abort_flag, int warp, int lane, int rank) {
  using C = GemmCfg<STAGE>;
  constexpr int kChunks = C::kBN / 32;
  constexpr bool kSym = STAGE <= kStagePoly;
  constexpr bool kPoly = STAGE == kStagePoly;
  const int quarter = warp & 3;
  uint8_t* my_slots = staging + quarter * C::kSlots * C::kSlotBytes;
  uint64_t* my_in = in_bar + quarter * C::kSlots;
  int acc = 0;
  uint32_t acc_phase = 0;
  int slot = 0;             // next staging slot (ring of kSlots)
  uint32_t in_par = 0;      // Poly: parity of each slot's next input load
  for (int t = first_tile(); t < L.total_tiles; t += tile_stride()) {
    __syncwarp();
    const Tile tl = decode_tile<STAGE>(L, t, rank);
    const GemmProblem& P = L.prob[tl.prob];
    const CUtensorMap* tm_out = &L.tm_out[tl.prob];
    const CUtensorMap* tm_in = &L.tm_in[tl.prob];
    float s = 1.f;
    if (STAGE != kStagePoly && P.first_round)
      s = inv_fro_norm(P.parts + static_cast<size_t>(tl.mat) * P.nparts, P.nparts, L.eps, lane);
    const int i0 = tl.tm * kTileM + quarter * 32;  // first row of this warp
    const int ncols = kSym ? P.m : P.n;
    const int jt = tl.tn * C::kBN;
    // live chunks: c_lo <= ch < c_hi (rows in range, columns in range)
    const int c_lo = 0;
    const int c_hi = i0 < P.m ? min(kChunks, (ncols - jt + 31) / 32) : 0;
    // Poly: the first two live chunks' A blocks into their slots
    if constexpr (kPoly) {
      if (lane == 0) {
        for (int k = 0; k < 2 && c_lo + k < c_hi; ++k) {
          const int sl = (slot + k) % C::kSlots;
          if (k == 0) ptx::bulk_wait_read<2>(); else ptx::bulk_wait_read<1>();
          ptx::mbar_arrive_expect_tx(&my_in[sl], 2048);
          ptx::tma_load_3d(my_slots + sl * C::kSlotBytes, tm_in, jt + 32 * (c_lo + k), i0, tl.mat,
                           &my_in[sl]);
        }
      }
      __syncwarp();
    }

    const bool got = ptx::mbar_wait(&acc_full[acc], acc_phase, abort_flag);
    __syncwarp();
    if (!got) {
      record_failure(L, abort_flag, kErrTimeoutEpilogue);
      break;
    }
    ptx::tc_fence_after();
    const uint32_t tbase =
        tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * C::kBN);
    bool failed = false;
#pragma unroll 1
    for (int ch = c_lo; ch < c_hi; ++ch) {
      const int j0 = jt + ch * 32;
      uint8_t* blk = my_slots + slot * C::kSlotBytes;
      uint32_t ev[16];
      if constexpr (kPoly) {
        const uint32_t par = (in_par >> slot) & 1u;
        if (!ptx::mbar_wait(&my_in[slot], par, abort_flag)) failed = true;
        in_par ^= 1u << slot;
        __syncwarp();
        // row `lane` of the A block, 64-byte swizzled like the output blocks
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 w = *reinterpret_cast<const uint4*>(blk + sw64(lane, 8 * q));
          ev[4 * q + 0] = w.x;
          ev[4 * q + 1] = w.y;
          ev[4 * q + 2] = w.z;
          ev[4 * q + 3] = w.w;
        }
      } else {
        // the slot's previous bulk store (two chunks ago) has read its data
        if (lane == 0) ptx::bulk_wait_read<1>();
      }
      __syncwarp();
      uint32_t v[32];
      ptx::tmem_ld32(tbase + static_cast<uint32_t>(ch * 32), v);
      ptx::tmem_ld_wait();
      float val[32];
      if constexpr (STAGE == kStageGram) {
#pragma unroll
        for (int q = 0; q < 32; ++q) val[q] = __uint_as_float(v[q]) * (s * s);
      } else if constexpr (kPoly) {
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          val[2 * q] = fmaf(L.c, __uint_as_float(v[2 * q]), L.b * bf_lo(ev[q]));
          val[2 * q + 1] = fmaf(L.c, __uint_as_float(v[2 * q + 1]), L.b * bf_hi(ev[q]));
        }
        // B' = a I + b A + c A A: the update then needs no a X term
        if (j0 == i0) {
#pragma unroll
          for (int q = 0; q < 32; ++q) val[q] += (q == lane) ? L.a : 0.f;
        }
      } else {
#pragma unroll
        for (int q = 0; q < 32; ++q) val[q] = s * __uint_as_float(v[q]);
      }

      stage_row_sw64(blk, lane, val);
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::tma_store_3d(tm_out, j0, i0, tl.mat, blk);
        ptx::bulk_commit();
        // Poly: the A block two live chunks ahead goes into the slot whose
        // store was issued one chunk ago
        if (kPoly && ch + 2 < c_hi) {
          const int sl = (slot + 2) % C::kSlots;
          ptx::bulk_wait_read<1>();
          ptx::mbar_arrive_expect_tx(&my_in[sl], 2048);
          ptx::tma_load_3d(my_slots + sl * C::kSlotBytes, tm_in, j0 + 64, i0, tl.mat, &my_in[sl]);
        }
      }
      slot = (slot + 1) % C::kSlots;
    }
    ptx::tc_fence_before();
    __syncwarp();
    // release the accumulator on the even CTA's barrier (the MMA issuer's)
    if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&acc_empty[acc]), 0));
    if (++acc == 2) {
      acc = 0;
      acc_phase ^= 1u;
    }
    if (failed) {
      record_failure(L, abort_flag, kErrTimeoutEpilogue);
      break;
    }
  }
  // all bulk copies of this warp are complete before the CTA exits
  if (lane == 0) ptx::bulk_wait<0>();
  __syncwarp();
}

// ------------------------------------------------------------ kernel
template <int STAGE>
__global__ void __launch_bounds__(GemmCfg<STAGE>::kThreads, 1)
    ns_gemm_kernel(const __grid_constant__ GemmLaunch L) {
  using C = GemmCfg<STAGE>;
  extern __shared__ uint8_t smem_raw[];
  // both CTAs of the pair get the same aligned offsets (the pair MMA reads both)
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* staging = smem + C::kStages * C::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + C::kStagingBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kStages;
  uint64_t* acc_full = bars + 2 * C::kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* in_bar = drain + 1;  // Poly: one per epilogue warp and slot
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(in_bar + C::kEpiWarps * C::kSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(ptx::cluster_ctarank());
  // the next stage may be scheduled now; it takes an SM only once this CTA has
  // left it, and waits for this grid to finish before reading its output
  ptx::griddep_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(&full[s], 1);   // the even CTA's expect_tx (+ both CTAs' bytes)
      ptx::mbar_init(&empty[s], 1);  // the pair MMA commit
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&acc_full[s], 1);
      ptx::mbar_init(&acc_empty[s], 2 * C::kEpiWarps);  // both CTAs' epilogue warps
    }
    ptx::mbar_init(drain, 1);
    for (int k = 0; k < C::kEpiWarps * C::kSlots; ++k) ptx::mbar_init(&in_bar[k], 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_slot, C::kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  __syncwarp();
  ptx::tc_fence_before();
  // both CTAs' barriers exist before either's copies signal the other's
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // setup above overlapped the previous stage's tail; its output is read below
  ptx::griddep_wait();

  if (warp == 0) {
    if (lane == 0) run_producer<STAGE>(L, smem, full, empty, abort_flag, rank);
  } else if (warp == 1) {
    if (lane == 0 && rank == 0)
      run_mma<STAGE>(L, smem, full, empty, acc_full, acc_empty, drain, tmem_base, abort_flag);
  } else {
    run_epilogue<STAGE>(L, acc_full, acc_empty, in_bar, tmem_base, staging, abort_flag, warp,
                        lane, rank);
  }

  __syncwarp();
  ptx::tc_fence_before();
  // neither CTA exits while the other may still write into its shared memory
  // or arrive on its barriers
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, C::kTmemCols);
  }
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
  if (!ptx::mbar_wait(&bar, 0, &abort_flag, limit_ns)) atomicOr(status, kErrTimeoutEpilogue);
  // complete the barrier's phase so nothing is left pending
  ptx::mbar_arrive(&bar);
}

cudaError_t launch_wait_selftest(unsigned int* status, unsigned long long limit_ns,
                                 cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

// ------------------------------------------------------------ launchers
template <int STAGE>
static cudaError_t launch_instance(const GemmLaunch& l, int pair_tiles, int sms, cudaStream_t s) {
  constexpr int kSmem = GemmCfg<STAGE>::kSmem;
  static int max_clusters[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(GemmCfg<STAGE>::kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;  // occupancy query: cluster shape only
  // clusters that fit on the device at once (one CTA per SM), queried once
  int n = dev < 64 ? max_clusters[dev] : 0;
  if (n == 0) {
    e = cudaFuncSetAttribute(ns_gemm_kernel<STAGE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmem);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * (sms / 2));
    e = cudaOccupancyMaxActiveClusters(&n, ns_gemm_kernel<STAGE>, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) n = 1;
    if (dev < 64) max_clusters[dev] = n;
  }
  const int clusters = pair_tiles < n ? pair_tiles : n;
  cfg.gridDim = dim3(2 * clusters);
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, ns_gemm_kernel<STAGE>, l);
}

int gemm_smem_bytes() { return GemmCfg<kStageUpdate>::kSmem; }

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

}  // namespace muon
