// ns_fused.cu -- every Newton-Schulz round of a matrix with 64 <= m <= 256 and
// n <= 512 (m = min(rows, cols), n = max) in one kernel: one CTA pair per
// matrix, X, A and B' kept in shared memory and TMEM across the rounds.
//
// The rounds are those of the staged path ("Muon Custom Sizing 实战", section
// 2.3; "parameter-golf train_gpt.py 源码精读", section 核心思想): A = X X^T,
// B' = aI + bA + cA^2, X <- B' X, with the first round scaled by
// s = 1 / (||u||_F + eps).  Matrices this small are latency-bound: the staged
// path spends three launches and three HBM round trips per round on them.
// The grouped prologue (momentum, Nesterov blend, bf16 X0 = u or u^T, norm
// partials) runs before this kernel and the grouped apply after it, on all
// SMs; this kernel reads X0 from the workspace and leaves O where the staged
// path leaves it (X buffer `steps & 1`).
//
// Layout.  X is padded to 256 x n_pad (n_pad = n rounded up to 128) with zeros;
// CTA r of the pair holds X rows 128r..128r+127 in up to eight 16 KB slabs of
// 64 columns (128-byte rows, 128-byte swizzle: the tensor cores' K-major
// operand layout, and the layout a 64 x 128 TMA box lands in).  TMA fills rows
// and columns outside the matrix with zeros; zero rows and columns stay zero
// through every round (they meet only zero rows/columns of A and the a*I
// term).  Y (four slabs) holds A, then B', for the CTA's 128 rows.
//
// One round, all MMAs tcgen05.mma.cta_group::2 (M = 256 across the pair)
// issued by one thread of the even CTA:
//   Gram    D0 = X X^T          (N = 256, K = n_pad; both operands = own X rows)
//   epilog  A = s^2 D0  -> bf16 into Y
//   (TMA)   the update reads X MN-major, and with M = 256 across the pair each
//           CTA supplies its half of the N columns for all 256 K rows; the
//           other CTA's rows of that half are loaded from the round's X buffer
//           in global memory (L2) into the slabs the Gram no longer needs,
//           while the polynomial runs
//   Poly    D1 = A A            (N = 256, K = 256; A symmetric: B = own A rows)
//   epilog  B' = a I + b A + c D1 -> bf16 into Y (over A)
//   Update  D = B' X            (up to two MMAs of N <= 256; the epilogue of the
//                                first overlaps the second)
//   epilog  X = s D -> bf16 into the slabs (own rows); TMA store of the slabs
//           the other CTA prefetches next round (all of them, O, at the end)
//           to the next X buffer, by a thread other than the MMA issuer
// Every wait on the tensor cores or TMA is bounded.
#include "internal.h"
#include "ptx.cuh"

namespace muon {
namespace {

constexpr int kFThreads = 256;
constexpr uint32_t kSlab = 16384;          // 128 rows x 128 bytes
constexpr uint32_t kXBytes = 8 * kSlab;    // up to 512 columns
constexpr uint32_t kYBytes = 4 * kSlab;    // 256 columns
constexpr uint32_t kMiscBytes = 256;
constexpr uint32_t kFusedSmem = kXBytes + kYBytes + kMiscBytes + 1024;
constexpr uint32_t kTmemCols = 512;

// byte offset of element (row i, column j) in a region of 128-row slabs
__device__ __forceinline__ uint32_t sw_off(int i, int j) {
  return static_cast<uint32_t>(j >> 6) * kSlab + static_cast<uint32_t>(i) * 128u +
         ((static_cast<uint32_t>((j >> 3) & 7) ^ static_cast<uint32_t>(i & 7)) << 4) +
         (static_cast<uint32_t>(j & 7) << 1);
}

// 32 fp32 values -> bf16 into row `row`, columns col..col+31 (col % 32 == 0)
__device__ __forceinline__ void st_row32(uint8_t* base, int row, int col, const float (&f)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      __nv_bfloat162 b2 = __floats2bfloat162_rn(f[8 * q + 2 * h], f[8 * q + 2 * h + 1]);
      w[h] = *reinterpret_cast<uint32_t*>(&b2);
    }
    *reinterpret_cast<uint4*>(base + sw_off(row, col + 8 * q)) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

struct Ctx {
  int tid, rank;
  int lrow, half;       // TMEM lane (own X row) and column half of this thread
  uint32_t tlane;       // lane field of the TMEM address for this warp
  uint32_t tmem;
  volatile int* bad;
  unsigned int* status;
};

__device__ __forceinline__ void fail(Ctx& x) {
  if (!*x.bad) atomicOr(x.status, kErrTimeoutFused);
  *x.bad = 1;
}

// All threads: wait for the commit of the MMAs with barrier phase `phase` (bounded).
__device__ __forceinline__ void wait_mma(Ctx& x, uint64_t* bar, uint32_t& phase) {
  if (!ptx::mbar_wait(bar, phase, x.bad, x.status)) fail(x);
  phase ^= 1u;
  ptx::tc_fence_after();
}

// Ends an epilogue: the generic shared-memory writes are made visible to the
// tensor cores (of both CTAs of a pair) and every TMEM read is ordered before
// later MMAs.
template <bool kPair>
__device__ __forceinline__ void epilogue_done() {
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  if constexpr (kPair) ptx::cluster_sync();
  else __syncthreads();
}

// kPair: one CTA pair per matrix, MMAs with M = 256 across the pair (m <= 256).
// !kPair: one CTA per matrix, M = 128 (m <= 128): no rows live in another CTA,
// so there is no prefetch and no store before the last round.
template <bool kPair>
__global__ void __launch_bounds__(kFThreads, 1)
    ns_fused_kernel(const __grid_constant__ FusedLaunch L) {
  constexpr int kM = kPair ? 256 : 128;   // MMA M, padded m, Gram N, Poly N and K
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* X = sm;
  uint8_t* Y = sm + kXBytes;
  uint64_t* mma_bar = reinterpret_cast<uint64_t*>(sm + kXBytes + kYBytes);
  uint64_t* ld_bar = mma_bar + 1;
  uint64_t* mma2_bar = ld_bar + 1;                     // second update MMA
  float* s_norm = reinterpret_cast<float*>(mma2_bar + 1);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(s_norm + 1);
  int* bad = reinterpret_cast<int*>(tslot + 1);

  ptx::griddep_launch_dependents();

  Ctx x;
  x.tid = threadIdx.x;
  const int warp = x.tid >> 5;
  x.rank = kPair ? static_cast<int>(ptx::cluster_ctarank()) : 0;
  x.lrow = x.tid & 127;
  x.half = x.tid >> 7;
  x.tlane = static_cast<uint32_t>((warp & 3) * 32) << 16;
  x.bad = bad;
  x.status = L.status;

  // which matrix
  const int unit = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  int gi = 0;
  while (gi + 1 < L.n_groups && unit >= L.grp[gi + 1].cluster_begin) ++gi;
  const FusedGroup& G = L.grp[gi];
  const int mat = unit - G.cluster_begin;
  const int m = G.m, n = G.n;
  const int n_pad = (n + 127) & ~127;
  const int n_slab = n_pad / 64;                        // slabs of own rows
  const int row0 = 128 * x.rank;                        // first X row held here
  const bool rows_here = row0 < m;
  const CUtensorMap* tm[2] = {&L.tm_x[gi][0], &L.tm_x[gi][1]};

  if (x.tid == 0) {
    ptx::mbar_init(mma_bar, 1);
    ptx::mbar_init(ld_bar, 1);
    ptx::mbar_init(mma2_bar, 1);
    *bad = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(tm[0]);
    ptx::prefetch_tmap(tm[1]);
  }
  if (warp == 0) {
    if constexpr (kPair) {
      ptx::tmem_alloc_pair(tslot, kTmemCols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(tslot, kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  x.tmem = *tslot;

  // X0 and the norm partials are written by the prologue, the kernel before
  ptx::griddep_wait();
  // A failure already recorded on this workspace: the CTA issues no copy and
  // no MMA (every later wait returns at once), but still passes every barrier
  // its pair partner passes.
  if (x.tid == 0 && ptx::status_set(L.status)) *bad = 1;
  __syncthreads();
  uint32_t ld_phase = 0, mma_phase = 0, mma2_phase = 0;
  constexpr int kStoreTid = 32;   // issues (and waits for) the X stores
  if (x.tid == 0 && !*bad) {
    ptx::mbar_arrive_expect_tx(ld_bar, n_slab * kSlab);
    for (int q = 0; q < n_slab; ++q)
      ptx::tma_load_3d(X + q * kSlab, tm[0], 64 * q, row0, mat, ld_bar);
  }
  if (warp == 1) {
    // s = 1 / (||u||_F + eps), the partials summed in the staged path's order
    const float* parts = G.parts + static_cast<size_t>(mat) * G.nparts;
    float acc = 0.f;
    for (int k = x.tid & 31; k < G.nparts; k += 32) acc += parts[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((x.tid & 31) == 0) *s_norm = 1.0f / (sqrtf(acc) + L.eps);
  }
  if (!ptx::mbar_wait(ld_bar, ld_phase, x.bad, x.status)) fail(x);
  ld_phase ^= 1u;
  ptx::tc_fence_before();
  if constexpr (kPair) ptx::cluster_sync();   // both CTAs' X0 slabs have landed
  else __syncthreads();
  ptx::tc_fence_after();
  const float s1 = *s_norm;

  const bool leader = x.rank == 0 && x.tid == 0;
  const uint32_t sx = ptx::smem_u32(X), sy = ptx::smem_u32(Y);
  const int n_mma = n_pad > 256 ? 2 : 1;
  auto mma = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    if constexpr (kPair) ptx::mma_bf16_pair(d, a, b, id, acc);
    else ptx::mma_bf16(d, a, b, id, acc);
  };
  auto commit = [&](uint64_t* bar) {
    if constexpr (kPair) ptx::mma_commit_pair(bar);
    else ptx::mma_commit(bar);
  };

  for (int it = 0; it < L.steps; ++it) {
    const float s = it == 0 ? s1 : 1.0f;
    const int cur = it & 1;
    // ------------------------------------------------------------ Gram
    if (leader && !*bad) {
      ptx::tc_fence_after();
      constexpr uint32_t kId = ptx::idesc_bf16(kM, kM, false);
      for (int k = 0; k < n_pad / 16; ++k) {
        const uint64_t d = ptx::smem_desc_sw128(sx + (k >> 2) * kSlab + (k & 3) * 32, 16, 1024);
        mma(x.tmem, d, d, kId, k > 0 ? 1u : 0u);
      }
      commit(mma_bar);
    }
    wait_mma(x, mma_bar, mma_phase);
    {
      const float s2 = s * s;
#pragma unroll 1
      for (int col = (kM / 2) * x.half; col < (kM / 2) * (x.half + 1); col += 64) {
        uint32_t v0[32], v1[32];
        ptx::tmem_ld32x2_sync(x.tmem + x.tlane + col, x.tmem + x.tlane + col + 32, v0, v1);
        float f[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(v0[e]) * s2;
        st_row32(Y, x.lrow, col, f);
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(v1[e]) * s2;
        st_row32(Y, x.lrow, col + 32, f);
      }
    }
    if constexpr (kPair) {
      // the previous round's X stores (read by the prefetch below) are complete
      if (x.tid == kStoreTid) {
        ptx::bulk_wait<0>();
        ptx::fence_proxy_async_global();
      }
    }
    epilogue_done<kPair>();
    // ------------------------------------------------------------ prefetch
    // Update MMA j covers X columns 256j.. (N = min(256, n_pad - 256j)); CTA r
    // supplies its N half, nsl = N / 128 slabs from slab 4j + r*nsl, for all
    // 256 K rows; K block kb (the rows of CTA kb) sits at slabs 4j + kb*nsl.
    // The other CTA's rows go to slabs 4j + (1-r)*nsl + e: those held this
    // CTA's rows of the other half, which only the Gram read.
    if constexpr (kPair) {
      if (x.tid == 0 && !*bad) {
        ptx::fence_proxy_async_global();
        ptx::mbar_arrive_expect_tx(ld_bar, (n_pad / 128) * kSlab);
        for (int j = 0; j < n_mma; ++j) {
          const int nsl = (n_pad - 256 * j) >= 256 ? 2 : 1;
          for (int e = 0; e < nsl; ++e)
            ptx::tma_load_3d(X + (4 * j + (1 - x.rank) * nsl + e) * kSlab, tm[cur],
                             256 * j + 64 * (x.rank * nsl + e), 128 * (1 - x.rank), mat, ld_bar);
        }
      }
    }
    // ------------------------------------------------------------ Poly
    if (leader && !*bad) {
      ptx::tc_fence_after();
      constexpr uint32_t kId = ptx::idesc_bf16(kM, kM, false);
      for (int k = 0; k < kM / 16; ++k) {
        const uint64_t d = ptx::smem_desc_sw128(sy + (k >> 2) * kSlab + (k & 3) * 32, 16, 1024);
        mma(x.tmem + kM, d, d, kId, k > 0 ? 1u : 0u);
      }
      commit(mma_bar);
    }
    wait_mma(x, mma_bar, mma_phase);
    {
      const float s2 = s * s;
      const int grow = row0 + x.lrow;
#pragma unroll 1
      for (int col = (kM / 2) * x.half; col < (kM / 2) * (x.half + 1); col += 32) {
        uint32_t v1[32], v0[32];
        ptx::tmem_ld32x2_sync(x.tmem + x.tlane + kM + col, x.tmem + x.tlane + col, v1, v0);
        float f[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          f[e] = fmaf(L.c, __uint_as_float(v1[e]), L.b * (__uint_as_float(v0[e]) * s2));
          if (grow == col + e) f[e] += L.a;
        }
        st_row32(Y, x.lrow, col, f);
      }
    }
    if constexpr (kPair) {
      // the other CTA's X rows have landed in this CTA's slabs
      if (x.tid == 0 && !*bad && !ptx::mbar_wait(ld_bar, ld_phase, x.bad, x.status)) fail(x);
      ld_phase ^= 1u;
    }
    epilogue_done<kPair>();
    // ------------------------------------------------------------ Update
    if (leader && !*bad) {
      ptx::tc_fence_after();
      for (int j = 0; j < n_mma; ++j) {
        const int nj = min(256, n_pad - 256 * j);
        const uint32_t id = ptx::idesc_bf16(kM, nj, true);
        for (int k = 0; k < kM / 16; ++k) {
          const uint64_t da =
              ptx::smem_desc_sw128(sy + (k >> 2) * kSlab + (k & 3) * 32, 16, 1024);
          uint32_t bslab;
          if constexpr (kPair) bslab = 4 * j + (k >> 3) * (nj / 128);   // K block k / 8
          else bslab = 4 * j;
          const uint64_t db =
              ptx::smem_desc_sw128(sx + bslab * kSlab + (k & 7) * 2048, kSlab, 1024);
          mma(x.tmem + 256 * j, da, db, id, k > 0 ? 1u : 0u);
        }
        commit(j == 0 ? mma_bar : mma2_bar);
      }
    }
#pragma unroll 1
    for (int j = 0; j < n_mma; ++j) {
      if (j == 0) wait_mma(x, mma_bar, mma_phase);
      else wait_mma(x, mma2_bar, mma2_phase);
      // columns of MMA j, split between the two thread halves
      const int per_half = min(256, n_pad - 256 * j) / 2;
      const int c0 = 256 * j + x.half * per_half;
#pragma unroll 1
      for (int col = c0; col < c0 + per_half; col += 64) {
        uint32_t v0[32], v1[32];
        ptx::tmem_ld32x2_sync(x.tmem + x.tlane + col, x.tmem + x.tlane + col + 32, v0, v1);
        float f[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(v0[e]) * s;
        st_row32(X, x.lrow, col, f);
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(v1[e]) * s;
        st_row32(X, x.lrow, col + 32, f);
      }
    }
    if constexpr (kPair) {
      // store this CTA's rows of the new X: the slabs the other CTA prefetches in
      // the next round (its column halves), or all of them after the last round;
      // the storing thread arrives on the cluster barrier first
      ptx::fence_proxy_async_smem();
      __syncthreads();
      ptx::tc_fence_before();
      ptx::cluster_arrive();
      if (x.tid == kStoreTid && rows_here && !*bad) {
        const bool last = it + 1 == L.steps;
        for (int j = 0; j < n_mma; ++j) {
          const int nsl = (n_pad - 256 * j) >= 256 ? 2 : 1;
          for (int e = 0; e < 2 * nsl; ++e) {
            const int q = 4 * j + e;                     // slab = 64 columns from 64q
            const bool theirs = e / nsl == 1 - x.rank;
            if ((last || theirs) && 64 * q < n)
              ptx::tma_store_3d(tm[cur ^ 1], 64 * q, row0, mat, X + q * kSlab);
          }
        }
        ptx::bulk_commit();
      }
      ptx::cluster_wait();
    } else {
      epilogue_done<false>();
      if (it + 1 == L.steps && x.tid == kStoreTid && !*bad) {
        for (int q = 0; q < n_slab && 64 * q < n; ++q)
          ptx::tma_store_3d(tm[cur ^ 1], 64 * q, 0, mat, X + q * kSlab);
        ptx::bulk_commit();
      }
    }
  }

  if (x.tid == kStoreTid) ptx::bulk_wait<0>();   // O is in global memory before the CTA ends
  ptx::tc_fence_before();
  if constexpr (kPair) ptx::cluster_sync();
  else __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    if constexpr (kPair) ptx::tmem_dealloc_pair(x.tmem, kTmemCols);
    else ptx::tmem_dealloc(x.tmem, kTmemCols);
  }
}

template <bool kPair>
cudaError_t launch_variant(const FusedLaunch& l, cudaStream_t s) {
  static int configured[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(
        ns_fused_kernel<kPair>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((kPair ? 2 : 1) * l.total_clusters);
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = kFusedSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kPair ? 2 : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kPair ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, ns_fused_kernel<kPair>, l);
}

}  // namespace

cudaError_t launch_fused(const FusedLaunch& l, cudaStream_t s) {
  return l.pair ? launch_variant<true>(l, s) : launch_variant<false>(l, s);
}

}  // namespace muon
