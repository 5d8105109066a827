// ns_gemm.cu -- the three GEMM stages of one quintic Newton-Schulz round on
// sm_103a tensor cores ("parameter-golf train_gpt.py 源码精读", part 1,
// section 核心思想: A = X X^T; B = b A + c A A; X = a X + B X):
//
//   Gram    A = s^2 X X^T      (s = 1/(||u||_F + eps) on the first round, else 1)
//   Poly    B = b A + c A A
//   Update  X' = s (a X + B X), or on the last round the parameter write
//           p <- (1 - lr wd) p - lr rescale X'   (or a bf16 copy of X')
//
// X is m x n (m <= n) bf16, row-major with padded leading dimension; A and B
// are m x m bf16.  A and B are symmetric, so Gram and Poly compute only the
// tiles on or above the diagonal and store every entry once directly and once
// mirrored.  For A A the second operand A[k][j] = A[j][k] is then read K-major
// like the first; only the Update's X operand (contraction over X's rows) is
// MN-major.
//
// Kernel shape: persistent, one CTA per SM, 192 threads:
//   warp 0      TMA producer (one lane) into a ring of swizzled smem stages
//   warp 1      TMEM allocator and tcgen05.mma issuer (one lane)
//   warps 2..5  epilogue: tcgen05.ld of the fp32 accumulator, fp32 math,
//               global stores
// The accumulator is double-buffered in TMEM so the epilogue of one tile
// overlaps the MMAs of the next.  Tiles of all problems of the launch form one
// linear list, walked with a stride of gridDim.x.
#include "internal.h"
#include "ptx.cuh"

namespace muon {

template <int BN>
struct GemmCfg {
  static constexpr int kStages = (BN == 256) ? 4 : 6;
  static constexpr int kABytes = kTileM * kTileK * 2;  // 16 KB: 128 rows x 128 B
  static constexpr int kBBytes = BN * kTileK * 2;      // BN rows (or BN/64 slabs) x 128 B
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmem = kStages * kStageBytes + kBarBytes + 1024;
};

struct Tile {
  int prob, mat, tm, tn;
};

// Linear tile index -> (problem, matrix, tile row, tile col).  Symmetric
// stages enumerate, per tile row tm, the tile columns tn >= floor(tm*128/BN).
template <int STAGE, int BN>
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
  if (STAGE == kStageUpdate) {
    r.tm = w / P.tiles_n;
    r.tn = w - r.tm * P.tiles_n;
  } else {
    r.tm = P.tiles_m;  // out of range unless found (no stores then)
    r.tn = 0;
#pragma unroll 1
    for (int tm = 0; tm < P.tiles_m; ++tm) {
      const int first = (tm * kTileM) / BN;
      const int cnt = P.tiles_n - first;
      if (w < cnt) {
        r.tm = tm;
        r.tn = first + w;
        break;
      }
      w -= cnt;
    }
  }
  return r;
}

__device__ __forceinline__ void record_failure(const GemmLaunch& L, volatile int* abort_flag,
                                               unsigned int bit) {
  *abort_flag = 1;
  atomicOr(L.status, bit);
}

// ------------------------------------------------------------ producer
template <int STAGE, int BN>
__device__ void run_producer(const GemmLaunch& L, uint8_t* smem, uint64_t* full, uint64_t* empty,
                             volatile int* abort_flag) {
  using C = GemmCfg<BN>;
  for (int p = 0; p < L.n_prob; ++p) {
    ptx::prefetch_tmap(&L.tm_a[p]);
    ptx::prefetch_tmap(&L.tm_b[p]);
  }
  int stage = 0;
  uint32_t phase = 0;
  uint32_t armed = 0, armed_parity = 0;
  bool ok = true;
  for (int t = blockIdx.x; ok && t < L.total_tiles; t += gridDim.x) {
    const Tile tl = decode_tile<STAGE, BN>(L, t);
    const GemmProblem& P = L.prob[tl.prob];
    const CUtensorMap* ta = &L.tm_a[tl.prob];
    const CUtensorMap* tb = &L.tm_b[tl.prob];
    for (int kb = 0; kb < P.k_blocks; ++kb) {
      if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
        record_failure(L, abort_flag, kErrTimeoutProducer);
        ok = false;
        break;
      }
      uint8_t* sa = smem + stage * C::kStageBytes;
      uint8_t* sb = sa + C::kABytes;
      ptx::mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
      // operand A: 128 rows (tile row tm) x 64 k-columns
      ptx::tma_load_3d(sa, ta, kb * kTileK, tl.tm * kTileM, tl.mat, &full[stage]);
      if (STAGE == kStageUpdate) {
        // operand B = X[k][j], MN-major: BN/64 slabs of 64 columns x 64 k-rows
#pragma unroll
        for (int q = 0; q < BN / 64; ++q)
          ptx::tma_load_3d(sb + q * (64 * kTileK * 2), tb, tl.tn * BN + q * 64, kb * kTileK,
                           tl.mat, &full[stage]);
      } else {
        // operand B: BN rows (tile col tn) x 64 k-columns, K-major
        ptx::tma_load_3d(sb, tb, kb * kTileK, tl.tn * BN, tl.mat, &full[stage]);
      }
      armed |= 1u << stage;
      armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == C::kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  // Every armed stage's copies have landed before the CTA may exit.
  for (int s = 0; s < C::kStages; ++s)
    if (armed & (1u << s))
      if (!ptx::mbar_wait(&full[s], (armed_parity >> s) & 1u, nullptr))
        record_failure(L, abort_flag, kErrTimeoutDrain);
}

// ------------------------------------------------------------ MMA issuer
template <int STAGE, int BN>
__device__ void run_mma(const GemmLaunch& L, uint8_t* smem, uint64_t* full, uint64_t* empty,
                        uint64_t* acc_full, uint64_t* acc_empty, uint64_t* drain,
                        uint32_t tmem_base, volatile int* abort_flag) {
  using C = GemmCfg<BN>;
  constexpr bool kBmn = (STAGE == kStageUpdate);
  constexpr uint32_t kIdesc = ptx::idesc_bf16_m128(BN, kBmn);
  int stage = 0;
  uint32_t phase = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  bool ok = true;
  for (int t = blockIdx.x; ok && t < L.total_tiles; t += gridDim.x) {
    const Tile tl = decode_tile<STAGE, BN>(L, t);
    const int kblocks = L.prob[tl.prob].k_blocks;
    if (!ptx::mbar_wait(&acc_empty[acc], acc_phase ^ 1u, abort_flag)) {
      record_failure(L, abort_flag, kErrTimeoutMma);
      break;
    }
    ptx::tc_fence_after();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
    for (int kb = 0; kb < kblocks; ++kb) {
      if (!ptx::mbar_wait(&full[stage], phase, abort_flag)) {
        record_failure(L, abort_flag, kErrTimeoutMma);
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t sa = ptx::smem_u32(smem + stage * C::kStageBytes);
      const uint32_t sb = sa + C::kABytes;
#pragma unroll
      for (int k = 0; k < kTileK / 16; ++k) {
        // K-major SW128: 8-row groups 1024 B apart; a K=16 slice is 32 B on.
        const uint64_t da = ptx::smem_desc_sw128(sa + k * 32, 16, 1024);
        // MN-major SW128: 64-column slabs (64 x 128 B) apart along N, 8-row
        // groups 1024 B apart along K; a K=16 slice is 16 rows = 2048 B on.
        const uint64_t db = kBmn ? ptx::smem_desc_sw128(sb + k * 2048, 64 * kTileK * 2, 1024)
                                 : ptx::smem_desc_sw128(sb + k * 32, 16, 1024);
        ptx::mma_bf16(d_tmem, da, db, kIdesc, (kb | k) != 0 ? 1u : 0u);
      }
      ptx::mma_commit(&empty[stage]);  // frees the stage once these MMAs finish
      if (++stage == C::kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) break;
    ptx::mma_commit(&acc_full[acc]);
    if (++acc == 2) {
      acc = 0;
      acc_phase ^= 1u;
    }
  }
  // Every MMA issued by this thread completes before TMEM is released.
  ptx::mma_commit(drain);
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

__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, int valid, const float (&f)[32]) {
  if (valid >= 32) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t ws[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(f[q * 8 + 2 * h], f[q * 8 + 2 * h + 1]);
        ws[h] = *reinterpret_cast<uint32_t*>(&b2);
      }
      d4[q] = make_uint4(ws[0], ws[1], ws[2], ws[3]);
    }
  } else {
#pragma unroll
    for (int t = 0; t < 32; ++t)
      if (t < valid) dst[t] = __float2bfloat16_rn(f[t]);
  }
}

// Parameter values the apply epilogue of chunk (i, j0) overwrites.  Not tall:
// p[i][j0..j0+31] of a [m, n] matrix; tall: p[j0+t][i] of an [n, m] matrix
// (lanes hold consecutive i, so each access is coalesced across the warp).
__device__ __forceinline__ void load_params32(const GemmProblem& P, int mat, int i, int j0,
                                              float (&pv)[32]) {
  const int m = P.m, n = P.n;
  const size_t moff = static_cast<size_t>(mat) * m * n;
  const int valid = n - j0;
  if (!P.tall) {
    const float* pr = P.param + moff + static_cast<size_t>(i) * n + j0;
    if (valid >= 32 && (n & 3) == 0) {
      const float4* p4 = reinterpret_cast<const float4*>(pr);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 w = p4[q];
        pv[4 * q + 0] = w.x;
        pv[4 * q + 1] = w.y;
        pv[4 * q + 2] = w.z;
        pv[4 * q + 3] = w.w;
      }
    } else {
#pragma unroll
      for (int t = 0; t < 32; ++t) pv[t] = (t < valid) ? pr[t] : 0.f;
    }
  } else {
    const float* pc = P.param + moff + static_cast<size_t>(j0) * m + i;
#pragma unroll
    for (int t = 0; t < 32; ++t) pv[t] = (t < valid) ? pc[static_cast<size_t>(t) * m] : 0.f;
  }
}

// Final output of chunk (i, j0) in the input's orientation: the parameter
// write p <- decay p - lr_eff x (kOutParam) or a bf16 copy of x (kOutBf16).
__device__ __forceinline__ void store_output32(const GemmProblem& P, int mat, int i, int j0,
                                               const float (&x)[32], const float (&pv)[32]) {
  const int m = P.m, n = P.n;
  const size_t moff = static_cast<size_t>(mat) * m * n;
  const int valid = n - j0;
  float o[32];
  if (P.out_mode == kOutParam) {
#pragma unroll
    for (int t = 0; t < 32; ++t) o[t] = fmaf(-P.lr_eff, x[t], P.decay * pv[t]);
  } else {
#pragma unroll
    for (int t = 0; t < 32; ++t) o[t] = x[t];
  }
  if (!P.tall) {
    const size_t base = moff + static_cast<size_t>(i) * n + j0;
    if (P.out_mode == kOutParam) {
      float* pr = P.param + base;
      if (valid >= 32 && (n & 3) == 0) {
        float4* p4 = reinterpret_cast<float4*>(pr);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          p4[q] = make_float4(o[4 * q + 0], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
      } else {
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (t < valid) pr[t] = o[t];
      }
    } else {
      __nv_bfloat16* orow = P.out + base;
      if (valid >= 32 && (n & 7) == 0) {
        store_row32(orow, 32, o);
      } else {
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (t < valid) orow[t] = __float2bfloat16_rn(o[t]);
      }
    }
  } else {
    const size_t base = moff + static_cast<size_t>(j0) * m + i;
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      if (t < valid) {
        if (P.out_mode == kOutParam)
          P.param[base + static_cast<size_t>(t) * m] = o[t];
        else
          P.out[base + static_cast<size_t>(t) * m] = __float2bfloat16_rn(o[t]);
      }
    }
  }
}

// Gram / Poly chunk: row i, columns j0..j0+31 of the symmetric output; stores
// the entries on/above the diagonal directly and those above it mirrored.
template <int STAGE>
__device__ __forceinline__ void epilogue_sym_chunk(const GemmLaunch& L, const GemmProblem& P,
                                                   int mat, int i, int j0, float scale,
                                                   const uint32_t (&v)[32],
                                                   const uint32_t (&av)[16]) {
  const int m = P.m, ld = P.lda;
  __nv_bfloat16* out = P.sym_out + static_cast<size_t>(mat) * m * ld;
  float val[32];
  if (STAGE == kStageGram) {
#pragma unroll
    for (int t = 0; t < 32; ++t) val[t] = __uint_as_float(v[t]) * scale;
  } else {
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      val[2 * t] = fmaf(L.c, __uint_as_float(v[2 * t]), L.b * bf_lo(av[t]));
      val[2 * t + 1] = fmaf(L.c, __uint_as_float(v[2 * t + 1]), L.b * bf_hi(av[t]));
    }
  }
  __nv_bfloat16* orow = out + static_cast<size_t>(i) * ld + j0;
  if (j0 + 32 <= m && j0 >= i) {
    store_row32(orow, 32, val);
  } else {
#pragma unroll
    for (int t = 0; t < 32; ++t)
      if (j0 + t >= i && j0 + t < m) orow[t] = __float2bfloat16_rn(val[t]);
  }
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    const int j = j0 + t;
    if (j > i && j < m) out[static_cast<size_t>(j) * ld + i] = __float2bfloat16_rn(val[t]);
  }
}

// ------------------------------------------------------------ epilogue warps
// Operands a chunk needs besides the accumulator are loaded one chunk ahead
// (the first chunk before waiting for the accumulator), so their latency
// overlaps the TMEM load and the previous chunk's math and stores.
template <int STAGE, int BN>
__device__ void run_epilogue(const GemmLaunch& L, uint64_t* acc_full, uint64_t* acc_empty,
                             uint32_t tmem_base, volatile int* abort_flag, int warp, int lane) {
  const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
  const int row = quarter * 32 + lane;
  int acc = 0;
  uint32_t acc_phase = 0;
  for (int t = blockIdx.x; t < L.total_tiles; t += gridDim.x) {
    __syncwarp();
    const Tile tl = decode_tile<STAGE, BN>(L, t);
    const GemmProblem& P = L.prob[tl.prob];
    float s = 1.f;
    if (STAGE != kStagePoly && P.first_round)
      s = inv_fro_norm(P.parts + static_cast<size_t>(tl.mat) * P.nparts, P.nparts, L.eps, lane);
    const int i = tl.tm * kTileM + row;
    const bool row_ok = i < P.m;
    const int ncols = (STAGE == kStageUpdate) ? P.n : P.m;
    const bool need_e = (STAGE != kStageGram);
    const bool need_p = (STAGE == kStageUpdate) && P.out_mode == kOutParam;
    const size_t ld = (STAGE == kStageUpdate) ? P.ldx : P.lda;
    const __nv_bfloat16* esrc =
        (STAGE == kStageUpdate ? P.x_cur : P.a_mat) +
        static_cast<size_t>(tl.mat) * P.m * ld + static_cast<size_t>(row_ok ? i : 0) * ld;

    uint32_t e_cur[16], e_nxt[16];
    float p_cur[32], p_nxt[32];
    {
      const int j0 = tl.tn * BN;
      if (row_ok && j0 < ncols) {
        if (need_e) load_row32(esrc + j0, ncols - j0, e_cur);
        if (need_p) load_params32(P, tl.mat, i, j0, p_cur);
      }
    }
    const bool got = ptx::mbar_wait(&acc_full[acc], acc_phase, abort_flag);
    __syncwarp();
    if (!got) {
      record_failure(L, abort_flag, kErrTimeoutEpilogue);
      break;
    }
    ptx::tc_fence_after();
    const uint32_t tbase =
        tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
      const int j0 = tl.tn * BN + ch * 32;
      if (j0 >= ncols) break;  // warp-uniform
      const int jn = j0 + 32;
      if (row_ok && ch + 1 < BN / 32 && jn < ncols) {
        if (need_e) load_row32(esrc + jn, ncols - jn, e_nxt);
        if (need_p) load_params32(P, tl.mat, i, jn, p_nxt);
      }
      __syncwarp();
      uint32_t v[32];
      ptx::tmem_ld32(tbase + static_cast<uint32_t>(ch * 32), v);
      ptx::tmem_ld_wait();
      if (row_ok) {
        if (STAGE == kStageUpdate) {
          float x[32];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            x[2 * q] = s * fmaf(L.a, bf_lo(e_cur[q]), __uint_as_float(v[2 * q]));
            x[2 * q + 1] = s * fmaf(L.a, bf_hi(e_cur[q]), __uint_as_float(v[2 * q + 1]));
          }
          if (P.out_mode == kOutX)
            store_row32(P.x_next + static_cast<size_t>(tl.mat) * P.m * P.ldx +
                            static_cast<size_t>(i) * P.ldx + j0,
                        ncols - j0, x);
          else
            store_output32(P, tl.mat, i, j0, x, p_cur);
        } else {
          epilogue_sym_chunk<STAGE>(L, P, tl.mat, i, j0, s * s, v, e_cur);
        }
      }
#pragma unroll
      for (int q = 0; q < 16; ++q) e_cur[q] = e_nxt[q];
      if (need_p) {
#pragma unroll
        for (int q = 0; q < 32; ++q) p_cur[q] = p_nxt[q];
      }
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&acc_empty[acc]);
    if (++acc == 2) {
      acc = 0;
      acc_phase ^= 1u;
    }
  }
}

// ------------------------------------------------------------ kernel
template <int STAGE, int BN>
__global__ void __launch_bounds__(192, 1) ns_gemm_kernel(const __grid_constant__ GemmLaunch L) {
  using C = GemmCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kStages;
  uint64_t* acc_full = bars + 2 * C::kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&acc_full[s], 1);
      ptx::mbar_init(&acc_empty[s], 4);
    }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) run_producer<STAGE, BN>(L, smem, full, empty, abort_flag);
  } else if (warp == 1) {
    if (lane == 0)
      run_mma<STAGE, BN>(L, smem, full, empty, acc_full, acc_empty, drain, tmem_base, abort_flag);
  } else {
    run_epilogue<STAGE, BN>(L, acc_full, acc_empty, tmem_base, abort_flag, warp, lane);
  }

  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ------------------------------------------------------------ launchers
template <int STAGE, int BN>
static cudaError_t launch_instance(const GemmLaunch& l, int grid, cudaStream_t s) {
  constexpr int kSmem = GemmCfg<BN>::kSmem;
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(ns_gemm_kernel<STAGE, BN>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  ns_gemm_kernel<STAGE, BN><<<grid, 192, kSmem, s>>>(l);
  return cudaGetLastError();
}

int gemm_smem_bytes(int stage, int bn) {
  (void)stage;
  return bn == 256 ? GemmCfg<256>::kSmem : GemmCfg<128>::kSmem;
}

cudaError_t launch_gemm(const GemmLaunch& l, int stage, int bn, int grid, cudaStream_t s) {
  switch (stage) {
    case kStageGram:
      return launch_instance<kStageGram, 128>(l, grid, s);
    case kStagePoly:
      return launch_instance<kStagePoly, 128>(l, grid, s);
    case kStageUpdate:
      return bn == 256 ? launch_instance<kStageUpdate, 256>(l, grid, s)
                       : launch_instance<kStageUpdate, 128>(l, grid, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace muon
