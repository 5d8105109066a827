// ns_fused.cu -- the whole Muon step of a matrix with 64 <= m <= 256 and n <= 512
// (m = min(rows, cols), n = max) in one kernel: one CTA pair per matrix, with
// X, A and B' kept in shared memory and TMEM for all NS rounds.
//
// The step is the one of the staged path (momentum lerp, Nesterov blend,
// Frobenius norm, quintic Newton-Schulz, rescale, decay, parameter write:
// "Muon Custom Sizing 实战", sections 2.3 and 四; "parameter-golf train_gpt.py
// 源码精读", section 核心思想).  Matrices this small are latency-bound: the staged
// path spends 17 launches and an HBM round trip per stage on them; here the
// intermediate matrices never leave the two SMs.
//
// Layout.  X (m x n, bf16, u^T when rows > cols) is padded to 256 x n_pad
// (n_pad = n rounded up to 128) with zeros; CTA r of the pair holds X rows
// 128r..128r+127 in eight 16 KB slabs of 64 columns (128-byte rows, 128-byte
// swizzle: the K-major operand layout of the tensor cores).  Zero rows and
// columns stay zero through every round (they meet only zero rows/columns of A
// and the a*I term), so the padding needs no masking.
//
// One round, all MMAs tcgen05.mma.cta_group::2 (M = 256 across the pair) issued
// by one thread of the even CTA:
//   Gram    D0 = X X^T          (N = 256, K = n_pad; both operands = own X rows)
//   epilog  A = s^2 D0  -> bf16 into the Y slabs (own rows, K-major)
//   Poly    D1 = A A            (N = 256, K = 256; A symmetric, so B = own A rows)
//   epilog  B' = a I + b A + c D1 -> bf16 into Y (over A)
//   swap    the update needs, in each CTA, every X row for that CTA's half of
//           the N columns; each CTA stages the X slabs the other needs in TMEM
//           and writes them into the other's shared memory (128 B rows)
//   Update  D = B' X            (N = n_pad in up to two MMAs of N <= 256; X read
//                                MN-major straight from the slabs)
//   epilog  X = s D -> bf16 into the X slabs (own rows, all columns)
// s = 1 / (||u||_F + eps) in the first round, 1 after (the norm folded into the
// epilogues, as in the staged path).  Then the parameter write reads X from
// shared memory.  All waits on the tensor cores are bounded.
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

__device__ __forceinline__ float4 ld_g4(const void* g, int gdt, size_t idx) {
  if (gdt == MUON_BF16) {
    const uint2 w = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(g) + idx);
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
  }
  return *reinterpret_cast<const float4*>(static_cast<const float*>(g) + idx);
}
__device__ __forceinline__ float ld_g1(const void* g, int gdt, size_t idx) {
  return gdt == MUON_BF16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(g)[idx])
                          : static_cast<const float*>(g)[idx];
}

// momentum update of one element; returns u, writes the new buffer value to nb
template <int MODE>
__device__ __forceinline__ float mom1(float g, float b, float beta, float& nb) {
  if (MODE == kPrologueNsOnly) return g;
  nb = fmaf(1.0f - beta, g - b, b);
  return MODE == kPrologueNesterov ? fmaf(beta, nb - g, g) : nb;
}

__device__ __forceinline__ void st_x(uint8_t* X, int i, int j, float v) {
  *reinterpret_cast<__nv_bfloat16*>(X + sw_off(i, j)) = __float2bfloat16_rn(v);
}
__device__ __forceinline__ float ld_x(const uint8_t* X, int i, int j) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(X + sw_off(i, j)));
}

// 32 fp32 values -> 32 bf16 of row `row`, columns col..col+31 (col % 32 == 0)
__device__ __forceinline__ void st_row32(uint8_t* base, int row, int col, const float (&f)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      __nv_bfloat162 b2 = __floats2bfloat162_rn(f[8 * q + 2 * h], f[8 * q + 2 * h + 1]);
      w[h] = *reinterpret_cast<uint32_t*>(&b2);
    }
    *reinterpret_cast<uint4*>(base + sw_off(row, col + 8 * q)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

struct Ctx {
  int tid, warp, rank;
  int lrow, half;       // TMEM lane (own X row) and column half of this thread
  uint32_t tlane;       // lane field of the TMEM address for this warp
  uint32_t tmem;
  uint64_t* bar;
  volatile int* bad;
  unsigned int* status;
  uint32_t phase;
};

// All threads: wait for the MMAs committed to `bar` (bounded).
__device__ __forceinline__ void wait_mma(Ctx& x) {
  if (!ptx::mbar_wait(x.bar, x.phase, reinterpret_cast<volatile int*>(x.bad))) {
    if (!*x.bad) atomicOr(x.status, kErrTimeoutFused);
    *x.bad = 1;
  }
  x.phase ^= 1u;
  ptx::tc_fence_after();
}

// Ends an epilogue: the generic shared-memory writes are made visible to the
// tensor cores of both CTAs and every TMEM read is ordered before later MMAs.
__device__ __forceinline__ void epilogue_done() {
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  ptx::cluster_sync();
}

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kFThreads, 1)
    ns_fused_kernel(const __grid_constant__ FusedLaunch L) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* X = sm;
  uint8_t* Y = sm + kXBytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kXBytes + kYBytes);
  float* red = reinterpret_cast<float*>(bar + 1);     // [8] warp sums
  float* norm2 = red + 8;                              // [2] per-CTA sums of u^2
  uint32_t* tslot = reinterpret_cast<uint32_t*>(norm2 + 2);
  int* bad = reinterpret_cast<int*>(tslot + 1);

  ptx::griddep_launch_dependents();

  Ctx x;
  x.tid = threadIdx.x;
  x.warp = x.tid >> 5;
  x.rank = static_cast<int>(ptx::cluster_ctarank());
  x.lrow = x.tid & 127;
  x.half = x.tid >> 7;
  x.tlane = static_cast<uint32_t>((x.warp & 3) * 32) << 16;
  x.bar = bar;
  x.bad = bad;
  x.status = L.status;
  x.phase = 0;

  // which matrix
  const int pair = blockIdx.x >> 1;
  int gi = 0;
  while (gi + 1 < L.n_groups && pair >= L.grp[gi + 1].cluster_begin) ++gi;
  const FusedGroup& G = L.grp[gi];
  const int mat = pair - G.cluster_begin;
  const int r = G.r, c = G.c;
  const bool tall = r > c;
  const int m = tall ? c : r, n = tall ? r : c;
  const int n_pad = (n + 127) & ~127;
  const size_t moff = static_cast<size_t>(mat) * r * c;
  const int row0 = 128 * x.rank;                        // first X row held here
  const int rows_here = max(0, min(128, m - row0));

  if (x.tid == 0) {
    ptx::mbar_init(bar, 1);
    *bad = 0;
    ptx::fence_mbar_init();
  }
  if (x.warp == 0) {
    ptx::tmem_alloc_pair(tslot, kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  // zero X (the padding must read as zero)
  for (int o = x.tid; o < static_cast<int>(kXBytes / 16); o += kFThreads)
    reinterpret_cast<uint4*>(X)[o] = make_uint4(0u, 0u, 0u, 0u);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  x.tmem = *tslot;

  // ---------------------------------------------------------------- prologue
  // u of this CTA's X rows; new momentum buffer; X = bf16(u); sum of u^2
  const float beta = L.beta;
  float ss = 0.f;
  if (!tall) {
    // X row i = matrix row row0 + i
    const size_t base = moff + static_cast<size_t>(row0) * c;
    if ((c & 3) == 0) {
      const int qpr = c >> 2;
      const int total = rows_here * qpr;
      for (int q0 = x.tid; q0 < total; q0 += 4 * kFThreads) {
        float4 gv[4], bv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int q = q0 + u * kFThreads;
          if (q < total) {
            const size_t idx = base + static_cast<size_t>(q) * 4;
            gv[u] = ld_g4(G.g, G.gdt, idx);
            if (MODE != kPrologueNsOnly) bv[u] = *reinterpret_cast<const float4*>(G.buf + idx);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int q = q0 + u * kFThreads;
          if (q >= total) continue;
          const int i = q / qpr, j = (q - i * qpr) * 4;
          const float ga[4] = {gv[u].x, gv[u].y, gv[u].z, gv[u].w};
          float ba[4] = {0.f, 0.f, 0.f, 0.f}, nb[4] = {0.f, 0.f, 0.f, 0.f}, ua[4];
          if (MODE != kPrologueNsOnly) {
            ba[0] = bv[u].x; ba[1] = bv[u].y; ba[2] = bv[u].z; ba[3] = bv[u].w;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            ua[e] = mom1<MODE>(ga[e], ba[e], beta, nb[e]);
            ss = fmaf(ua[e], ua[e], ss);
          }
          if (MODE != kPrologueNsOnly)
            *reinterpret_cast<float4*>(G.buf + base + static_cast<size_t>(q) * 4) =
                make_float4(nb[0], nb[1], nb[2], nb[3]);
          __nv_bfloat162 lo = __floats2bfloat162_rn(ua[0], ua[1]);
          __nv_bfloat162 hi = __floats2bfloat162_rn(ua[2], ua[3]);
          *reinterpret_cast<uint2*>(X + sw_off(i, j)) =
              make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
        }
      }
    } else {
      const int total = rows_here * c;
      for (int e0 = x.tid; e0 < total; e0 += kFThreads) {
        const int i = e0 / c, j = e0 - i * c;
        const size_t idx = base + static_cast<size_t>(e0);
        const float b = MODE != kPrologueNsOnly ? G.buf[idx] : 0.f;
        float nb = 0.f;
        const float u = mom1<MODE>(ld_g1(G.g, G.gdt, idx), b, beta, nb);
        if (MODE != kPrologueNsOnly) G.buf[idx] = nb;
        ss = fmaf(u, u, ss);
        st_x(X, i, j, u);
      }
    }
  } else {
    // X row i = matrix column row0 + i; X column j = matrix row j
    const bool vec = (c & 3) == 0;
    const int qpr = (rows_here + 3) >> 2;
    const int total = n * qpr;
    for (int q = x.tid; q < total; q += kFThreads) {
      const int j = q / qpr, i4 = (q - j * qpr) * 4;
      const size_t idx = moff + static_cast<size_t>(j) * c + row0 + i4;
      const int valid = min(4, rows_here - i4);
      float ga[4] = {0.f, 0.f, 0.f, 0.f}, ba[4] = {0.f, 0.f, 0.f, 0.f};
      if (vec && valid == 4) {
        const float4 g4 = ld_g4(G.g, G.gdt, idx);
        ga[0] = g4.x; ga[1] = g4.y; ga[2] = g4.z; ga[3] = g4.w;
        if (MODE != kPrologueNsOnly) {
          const float4 b4 = *reinterpret_cast<const float4*>(G.buf + idx);
          ba[0] = b4.x; ba[1] = b4.y; ba[2] = b4.z; ba[3] = b4.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (e < valid) {
            ga[e] = ld_g1(G.g, G.gdt, idx + e);
            if (MODE != kPrologueNsOnly) ba[e] = G.buf[idx + e];
          }
      }
      float nb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (e >= valid) continue;
        const float u = mom1<MODE>(ga[e], ba[e], beta, nb[e]);
        ss = fmaf(u, u, ss);
        st_x(X, i4 + e, j, u);
      }
      if (MODE != kPrologueNsOnly) {
        if (vec && valid == 4) {
          *reinterpret_cast<float4*>(G.buf + idx) = make_float4(nb[0], nb[1], nb[2], nb[3]);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (e < valid) G.buf[idx + e] = nb[e];
        }
      }
    }
  }
  // sum of u^2 over the pair, in a fixed order (both CTAs get the same value)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((x.tid & 31) == 0) red[x.warp] = ss;
  __syncthreads();
  if (x.tid == 0) {
    float t = 0.f;
    for (int w = 0; w < kFThreads / 32; ++w) t += red[w];
    norm2[x.rank] = t;
    ptx::st_cluster_f32(ptx::mapa_shared(ptx::smem_u32(&norm2[x.rank]), x.rank ^ 1), t);
  }
  epilogue_done();
  const float s1 = 1.0f / (sqrtf(norm2[0] + norm2[1]) + L.eps);

  const bool leader = x.rank == 0 && x.tid == 0;
  const uint32_t sx = ptx::smem_u32(X), sy = ptx::smem_u32(Y);
  const int n_mma = n_pad > 256 ? 2 : 1;

  for (int it = 0; it < L.steps; ++it) {
    const float s = it == 0 ? s1 : 1.0f;
    // ------------------------------------------------------------ Gram
    if (leader && !*bad) {
      ptx::tc_fence_after();
      constexpr uint32_t kId = ptx::idesc_bf16(256, 256, false);
      for (int k = 0; k < n_pad / 16; ++k) {
        const uint64_t d = ptx::smem_desc_sw128(sx + (k >> 2) * kSlab + (k & 3) * 32, 16, 1024);
        ptx::mma_bf16_pair(x.tmem, d, d, kId, k > 0 ? 1u : 0u);
      }
      ptx::mma_commit_pair(bar);
    }
    wait_mma(x);
    {
      const float s2 = s * s;
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        const int col = 128 * x.half + 32 * ch;
        uint32_t v[32];
        ptx::tmem_ld32_sync(x.tmem + x.tlane + col, v);
        float f[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(v[e]) * s2;
        st_row32(Y, x.lrow, col, f);
      }
    }
    epilogue_done();
    // ------------------------------------------------------------ Poly
    if (leader && !*bad) {
      ptx::tc_fence_after();
      constexpr uint32_t kId = ptx::idesc_bf16(256, 256, false);
      for (int k = 0; k < 16; ++k) {
        const uint64_t d = ptx::smem_desc_sw128(sy + (k >> 2) * kSlab + (k & 3) * 32, 16, 1024);
        ptx::mma_bf16_pair(x.tmem + 256, d, d, kId, k > 0 ? 1u : 0u);
      }
      ptx::mma_commit_pair(bar);
    }
    wait_mma(x);
    {
      const float s2 = s * s;
      const int grow = row0 + x.lrow;
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        const int col = 128 * x.half + 32 * ch;
        uint32_t v1[32], v0[32];
        ptx::tmem_ld32_sync(x.tmem + x.tlane + 256 + col, v1);
        ptx::tmem_ld32_sync(x.tmem + x.tlane + col, v0);
        float f[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          f[e] = fmaf(L.c, __uint_as_float(v1[e]), L.b * (__uint_as_float(v0[e]) * s2));
          if (grow == col + e) f[e] += L.a;
        }
        st_row32(Y, x.lrow, col, f);
      }
    }
    // ------------------------------------------------------------ X swap
    // Update MMA j covers X columns 256j.. (N = min(256, n_pad - 256j)); CTA r
    // supplies its N half, nsl = N / 128 slabs starting at slab 4j + r*nsl, for
    // all 256 K rows (K block kb = the rows of CTA kb).  Outgoing slab o
    // (o < n_pad / 128, j = o / 2, e = o % 2) of CTA r is slab 4j + (1-r)*nsl + e
    // of its own rows (the other CTA's column half); it lands in the other CTA
    // at slab 4j + r*nsl + e, which that CTA has just sent away.  Afterwards
    // both CTAs hold K block kb of MMA j's operand at slabs 4j + kb*nsl + e.
    {
      const int n_out = n_pad / 128;
      for (int o = x.half; o < n_out; o += 2) {
        const int j = o >> 1, e = o & 1;
        const int nsl = (n_pad - 256 * j) >= 256 ? 2 : 1;
        const int src = 4 * j + (1 - x.rank) * nsl + e;
        uint32_t v[32];
        const uint4* line = reinterpret_cast<const uint4*>(X + src * kSlab + x.lrow * 128);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 w = line[q];
          v[4 * q] = w.x; v[4 * q + 1] = w.y; v[4 * q + 2] = w.z; v[4 * q + 3] = w.w;
        }
        ptx::tmem_st32_sync(x.tmem + x.tlane + 32 * o, v);
      }
      epilogue_done();   // (also publishes B' in Y)
      ptx::tc_fence_after();
      for (int o = x.half; o < n_out; o += 2) {
        const int j = o >> 1, e = o & 1;
        const int nsl = (n_pad - 256 * j) >= 256 ? 2 : 1;
        const int dst = 4 * j + x.rank * nsl + e;
        uint32_t v[32];
        ptx::tmem_ld32_sync(x.tmem + x.tlane + 32 * o, v);
        const uint32_t remote = ptx::mapa_shared(sx + dst * kSlab + x.lrow * 128, x.rank ^ 1);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          ptx::st_cluster_v4(remote + 16 * q,
                             make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
      }
      ptx::fence_proxy_async_cluster();
      ptx::tc_fence_before();
      ptx::cluster_sync();
    }
    // ------------------------------------------------------------ Update
    if (leader && !*bad) {
      ptx::tc_fence_after();
      for (int j = 0; j < n_mma; ++j) {
        const int nj = min(256, n_pad - 256 * j);
        const int nsl = nj / 128;
        const uint32_t id = ptx::idesc_bf16(256, nj, true);
        for (int k = 0; k < 16; ++k) {
          const int kb = k >> 3, kk = k & 7;
          const uint64_t da =
              ptx::smem_desc_sw128(sy + (k >> 2) * kSlab + (k & 3) * 32, 16, 1024);
          const uint64_t db =
              ptx::smem_desc_sw128(sx + (4 * j + kb * nsl) * kSlab + kk * 2048, kSlab, 1024);
          ptx::mma_bf16_pair(x.tmem + 256 * j, da, db, id, k > 0 ? 1u : 0u);
        }
      }
      ptx::mma_commit_pair(bar);
    }
    wait_mma(x);
    {
      const int per_half = n_pad / 2;
#pragma unroll 1
      for (int col = x.half * per_half; col < (x.half + 1) * per_half; col += 32) {
        uint32_t v[32];
        ptx::tmem_ld32_sync(x.tmem + x.tlane + col, v);
        float f[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(v[e]) * s;
        st_row32(X, x.lrow, col, f);
      }
    }
    epilogue_done();
  }

  // ---------------------------------------------------------------- apply
  // p <- decay p - lr_eff O, or out <- O (NS only); O = X (transposed back)
  if (!tall) {
    const size_t base = moff + static_cast<size_t>(row0) * c;
    if ((c & 3) == 0) {
      const int qpr = c >> 2;
      const int total = rows_here * qpr;
      for (int q = x.tid; q < total; q += kFThreads) {
        const int i = q / qpr, j = (q - i * qpr) * 4;
        const uint2 w = *reinterpret_cast<const uint2*>(X + sw_off(i, j));
        const size_t idx = base + static_cast<size_t>(q) * 4;
        if (MODE == kPrologueNsOnly) {
          *reinterpret_cast<uint2*>(G.out + idx) = w;
        } else {
          const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
          const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
          float4 p = *reinterpret_cast<const float4*>(G.param + idx);
          p.x = fmaf(-G.lr_eff, lo.x, L.decay * p.x);
          p.y = fmaf(-G.lr_eff, lo.y, L.decay * p.y);
          p.z = fmaf(-G.lr_eff, hi.x, L.decay * p.z);
          p.w = fmaf(-G.lr_eff, hi.y, L.decay * p.w);
          *reinterpret_cast<float4*>(G.param + idx) = p;
        }
      }
    } else {
      const int total = rows_here * c;
      for (int e0 = x.tid; e0 < total; e0 += kFThreads) {
        const int i = e0 / c, j = e0 - i * c;
        const size_t idx = base + static_cast<size_t>(e0);
        const float o = ld_x(X, i, j);
        if (MODE == kPrologueNsOnly) G.out[idx] = __float2bfloat16_rn(o);
        else G.param[idx] = fmaf(-G.lr_eff, o, L.decay * G.param[idx]);
      }
    }
  } else {
    const bool vec = (c & 3) == 0;
    const int qpr = (rows_here + 3) >> 2;
    const int total = n * qpr;
    for (int q = x.tid; q < total; q += kFThreads) {
      const int j = q / qpr, i4 = (q - j * qpr) * 4;
      const size_t idx = moff + static_cast<size_t>(j) * c + row0 + i4;
      const int valid = min(4, rows_here - i4);
      float o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = e < valid ? ld_x(X, i4 + e, j) : 0.f;
      if (MODE == kPrologueNsOnly) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (e < valid) G.out[idx + e] = __float2bfloat16_rn(o[e]);
      } else if (vec && valid == 4) {
        float4 p = *reinterpret_cast<const float4*>(G.param + idx);
        p.x = fmaf(-G.lr_eff, o[0], L.decay * p.x);
        p.y = fmaf(-G.lr_eff, o[1], L.decay * p.y);
        p.z = fmaf(-G.lr_eff, o[2], L.decay * p.z);
        p.w = fmaf(-G.lr_eff, o[3], L.decay * p.w);
        *reinterpret_cast<float4*>(G.param + idx) = p;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (e < valid) G.param[idx + e] = fmaf(-G.lr_eff, o[e], L.decay * G.param[idx + e]);
      }
    }
  }

  // a programmatic dependent of the kernel before: finish only after it
  ptx::griddep_wait();
  ptx::tc_fence_before();
  ptx::cluster_sync();
  if (x.warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(x.tmem, kTmemCols);
  }
}

template <int MODE>
cudaError_t launch_mode(const FusedLaunch& l, bool pdl, cudaStream_t s) {
  static int configured[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(
        ns_fused_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * l.total_clusters);
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = kFusedSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, ns_fused_kernel<MODE>, l);
}

}  // namespace

cudaError_t launch_fused(const FusedLaunch& l, bool pdl, cudaStream_t s) {
  switch (l.mode) {
    case kPrologueNsOnly:
      return launch_mode<kPrologueNsOnly>(l, pdl, s);
    case kPrologueNesterov:
      return launch_mode<kPrologueNesterov>(l, pdl, s);
    case kProloguePlain:
      return launch_mode<kProloguePlain>(l, pdl, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace muon
