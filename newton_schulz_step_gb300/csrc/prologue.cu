// prologue.cu -- the elementwise head of the Muon step, one pass over HBM:
//
//   buf <- buf + (1 - beta) (g - buf)        momentum buffer moved towards g
//   u   <- g + beta (buf - g)                Nesterov blend
//                                            (or u = buf without Nesterov, u = g for NS only)
//   X   <- bf16(u), or bf16(u^T) when rows > cols (padded leading dimension)
//   partial sums of u^2 for the Frobenius norm, one per block
//
// ("Muon Custom Sizing 实战", section 四, second pass; the norm is the Frobenius norm
// of "parameter-golf train_gpt.py 源码精读", section 核心思想.)  The division by
// ||u||_F + eps is folded into the first Gram and update epilogues, which sum
// the partials in a fixed order, so the result is deterministic.
//
// One launch covers every tensor-core group: block b of the launch belongs to
// group g, matrix z, part q, and walks the 64x64 tiles q, q + nparts, ... of
// that matrix (nparts is chosen per group so each block gets ~4 tiles).  Each
// thread moves 2 x 8 consecutive elements of a tile row with 16-byte accesses;
// rows > cols tiles are transposed through shared memory so the X stores stay
// coalesced.  Launched as a programmatic dependent of the small-matrix kernel,
// it overlaps that kernel; one of its blocks waits for it before exiting.
#include "internal.h"

namespace muon {

namespace {

__device__ __forceinline__ void load_g8(const void* g, int gdt, size_t idx, bool vec, int valid,
                                        float (&out)[8]) {
  if (gdt == MUON_BF16) {
    const __nv_bfloat16* gp = static_cast<const __nv_bfloat16*>(g) + idx;
    if (vec) {
      const uint4 w = *reinterpret_cast<const uint4*>(gp);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[h]));
        out[2 * h] = f.x;
        out[2 * h + 1] = f.y;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) out[e] = (e < valid) ? __bfloat162float(gp[e]) : 0.f;
    }
  } else {
    const float* gp = static_cast<const float*>(g) + idx;
    if (vec) {
      const float4 a = *reinterpret_cast<const float4*>(gp);
      const float4 b = *reinterpret_cast<const float4*>(gp + 4);
      out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
      out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) out[e] = (e < valid) ? gp[e] : 0.f;
    }
  }
}

__device__ __forceinline__ void load_f8(const float* p, bool vec, int valid, float (&out)[8]) {
  if (vec) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
    out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) out[e] = (e < valid) ? p[e] : 0.f;
  }
}

__device__ __forceinline__ void store_f8(float* p, bool vec, int valid, const float (&v)[8]) {
  if (vec) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (e < valid) p[e] = v[e];
  }
}

__device__ __forceinline__ void store_bf8(__nv_bfloat16* p, bool vec, int valid,
                                          const float (&v)[8]) {
  if (vec) {
    uint32_t ws[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * h], v[2 * h + 1]);
      ws[h] = *reinterpret_cast<uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(ws[0], ws[1], ws[2], ws[3]);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (e < valid) p[e] = __float2bfloat16_rn(v[e]);
  }
}

template <int MODE>
__global__ void __launch_bounds__(256) prologue_kernel(const __grid_constant__ PrologueLaunch L) {
  __shared__ float stage_tile[64][65];
  __shared__ float red[8];
  // the first Gram stage may be scheduled once every block here has started
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // a failure already recorded on this workspace: this call changes nothing
  // (block 0 still keeps the completion chain, below)
  if (*reinterpret_cast<const volatile unsigned int*>(L.status) != 0u) {
    if (L.wait_prior && blockIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
    return;
  }
  // per-matrix completion counters of the GEMMs, which read them only
  // after this grid has completed
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < L.n_zero; i += blockDim.x) L.zero[i] = 0u;
    if (threadIdx.x == 0 && L.zero_work != nullptr) *L.zero_work = 0u;
  }
  int gi = 0;
  while (gi + 1 < L.n_groups && static_cast<int>(blockIdx.x) >= L.grp[gi + 1].block_begin) ++gi;
  const PrologueGroup& A = L.grp[gi];
  const int local = blockIdx.x - A.block_begin;
  const int mat = local / A.nparts;
  const int part = local - mat * A.nparts;
  const int r = A.r, c = A.c;
  const bool tall = r > c && !A.pmajor;  // X = u^T, transposed here
  const int tiles_c = (c + 63) / 64;
  const int ntiles = ((r + 63) / 64) * tiles_c;
  const size_t moff = static_cast<size_t>(mat) * r * c;
  const int m = tall ? c : r;
  __nv_bfloat16* xm = A.x + static_cast<size_t>(mat) * m * A.ldx;
  const int tid = threadIdx.x;
  const int ty = tid >> 3;        // tile row within a 32-row half
  const int tx = (tid & 7) * 8;   // first of 8 tile columns
  const bool cvec = (c & 7) == 0; // rows start 16-byte aligned
  const float beta = L.beta;
  float sumsq = 0.f;

  for (int tile = part; tile < ntiles; tile += A.nparts) {
    const int tr = tile / tiles_c;
    const int tc = tile - tr * tiles_c;
    const int cc = tc * 64 + tx;
    const int valid = max(0, min(8, c - cc));
    float gv[2][8], bv[2][8];
    // all loads of the tile first, so both halves are in flight together
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int rr = tr * 64 + ty + 32 * h;
      const bool in = rr < r && valid > 0;
      const size_t idx = moff + static_cast<size_t>(rr) * c + cc;
      if (in) {
        load_g8(A.g, A.gdt, idx, cvec && valid == 8, valid, gv[h]);
        if (MODE != kPrologueNsOnly) load_f8(A.buf + idx, cvec && valid == 8, valid, bv[h]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) gv[h][e] = bv[h][e] = 0.f;
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int rr = tr * 64 + ty + 32 * h;
      const bool in = rr < r && valid > 0;
      const size_t idx = moff + static_cast<size_t>(rr) * c + cc;
      float u[8];
      if (MODE == kPrologueNsOnly) {
#pragma unroll
        for (int e = 0; e < 8; ++e) u[e] = gv[h][e];
      } else {
        float nb[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          nb[e] = fmaf(1.0f - beta, gv[h][e] - bv[h][e], bv[h][e]);
          u[e] = (MODE == kPrologueNesterov) ? fmaf(beta, nb[e] - gv[h][e], gv[h][e]) : nb[e];
        }
        if (in) store_f8(A.buf + idx, cvec && valid == 8, valid, nb);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) sumsq = fmaf(u[e], u[e], sumsq);
      if (!tall) {
        if (in) store_bf8(xm + static_cast<size_t>(rr) * A.ldx + cc, valid == 8, valid, u);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) stage_tile[ty + 32 * h][tx + e] = u[e];
      }
    }
    if (tall) {
      // X = u^T: X row (original column) tc*64 + ..., X columns tr*64 + ...
      __syncthreads();
      const int xc = tr * 64 + tx;                 // X column = original row
      const int xvalid = max(0, min(8, r - xc));
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int xr = tc * 64 + ty + 32 * h;      // X row = original column
        if (xr < c && xvalid > 0) {
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = stage_tile[tx + e][ty + 32 * h];
          store_bf8(xm + static_cast<size_t>(xr) * A.ldx + xc, xvalid == 8, xvalid, v);
        }
      }
      __syncthreads();
    }
  }

  // deterministic block reduction of sum(u^2)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sumsq += __shfl_xor_sync(0xffffffffu, sumsq, o);
  if ((tid & 31) == 0) red[tid >> 5] = sumsq;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += red[w];
    A.parts[static_cast<size_t>(mat) * A.nparts + part] = t;
  }
  // Programmatic dependent of the small-matrix kernel: the grid finishes only
  // after it.  One block waiting is enough for that (the grid completes when its
  // last block exits); if every block waited, the first wave would hold its SMs
  // until the small kernel ended and the rest of the prologue could not start.
  if (L.wait_prior && blockIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------------ apply
// The tail of the Muon step ("Muon Custom Sizing 实战", section 四: decay
// lr*wd on the parameter, then the NS result added with alpha = -lr * rescale;
// "parameter-golf train_gpt.py 源码精读", section 分布式细节: the rescale
// max(1, m/n)^0.5):  p <- (1 - lr wd) p - lr_eff O, with O the bf16 NS result
// transposed back when rows > cols.  Same block layout as the prologue.
template <bool TO_PARAM>
__global__ void __launch_bounds__(256) apply_kernel(const __grid_constant__ ApplyLaunch L) {
  __shared__ float stage_tile[64][65];
  // launched as a programmatic dependent of the last update: its output is O
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // a failure recorded on this workspace (by this call's NS or an earlier
  // call): O is not valid, nothing is written
  if (*reinterpret_cast<const volatile unsigned int*>(L.status) != 0u) return;
  int gi = 0;
  while (gi + 1 < L.n_groups && static_cast<int>(blockIdx.x) >= L.grp[gi + 1].block_begin) ++gi;
  const ApplyGroup& A = L.grp[gi];
  const int local = blockIdx.x - A.block_begin;
  const int mat = local / A.nparts;
  const int part = local - mat * A.nparts;
  const int r = A.r, c = A.c;
  const bool tall = r > c;
  const int tiles_c = (c + 63) / 64;
  const int ntiles = ((r + 63) / 64) * tiles_c;
  const size_t moff = static_cast<size_t>(mat) * r * c;
  const int m = tall ? c : r;
  const __nv_bfloat16* om = A.o + static_cast<size_t>(mat) * m * A.ldx;
  const int tid = threadIdx.x;
  const int ty = tid >> 3;
  const int tx = (tid & 7) * 8;
  const bool cvec = (c & 7) == 0;

  for (int tile = part; tile < ntiles; tile += A.nparts) {
    const int tr = tile / tiles_c;
    const int tc = tile - tr * tiles_c;
    const int cc = tc * 64 + tx;
    const int valid = max(0, min(8, c - cc));
    float pv[2][8], ov[2][8];
    if (TO_PARAM) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int rr = tr * 64 + ty + 32 * h;
        if (rr < r && valid > 0)
          load_f8(A.param + moff + static_cast<size_t>(rr) * c + cc, cvec && valid == 8, valid,
                  pv[h]);
      }
    }
    if (!tall) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int rr = tr * 64 + ty + 32 * h;
        if (rr < r && valid > 0)
          load_g8(om + static_cast<size_t>(rr) * A.ldx + cc, MUON_BF16, 0, valid == 8, valid,
                  ov[h]);
      }
    } else {
      // O row = original column, O column = original row: transpose the tile
      const int xc = tr * 64 + tx;
      const int xvalid = max(0, min(8, r - xc));
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int xr = tc * 64 + ty + 32 * h;
        float v[8];
        if (xr < c && xvalid > 0)
          load_g8(om + static_cast<size_t>(xr) * A.ldx + xc, MUON_BF16, 0, xvalid == 8, xvalid, v);
        else
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) stage_tile[ty + 32 * h][tx + e] = v[e];
      }
      __syncthreads();
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) ov[h][e] = stage_tile[tx + e][ty + 32 * h];
      __syncthreads();
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int rr = tr * 64 + ty + 32 * h;
      if (rr < r && valid > 0) {
        const size_t idx = moff + static_cast<size_t>(rr) * c + cc;
        if (TO_PARAM) {
          float nv[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) nv[e] = fmaf(-A.lr_eff, ov[h][e], A.decay * pv[h][e]);
          store_f8(A.param + idx, cvec && valid == 8, valid, nv);
        } else {
          store_bf8(A.out + idx, cvec && valid == 8, valid, ov[h]);
        }
      }
    }
  }
}

// ------------------------------------------------------------ streamed apply
// The same parameter write, p <- (1 - lr wd) p - lr_eff O, launched as a
// programmatic dependent of the last update (the persistent rounds kernel, or
// the last round's update launch) so that it runs beside it: each block claims
// work units (a few rows of one matrix, ~8192 elements) in the order that
// update finishes matrices, waits until the matrix's completion counter shows
// its last update stored, and streams the rows.  O is already in the
// parameter's orientation (the last update of a rows > cols matrix stores
// O^T), so every access is a coalesced row access and the kernel needs almost
// no shared memory: one of its blocks fits on an SM beside a GEMM CTA.
// Requires cols % 8 == 0 (16-byte row segments).
constexpr int kStreamSeg = 8;    // elements per thread access (16 B of O, 32 B of p)
constexpr int kStreamDepth = 2;  // row segments per thread in flight

// Counter wait of the streamed apply: acquire, bounded, ended early by a set
// status word.  One thread per block polls, with a backoff from 1 to 8 us:
// the counters are the GEMM's own, which its epilogues update (and the rounds
// kernel's scheduler warps poll), so these waits must not crowd their L2 lines.
__device__ __forceinline__ bool wait_done(const unsigned int* p, unsigned int target,
                                          const unsigned int* status) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  if (v >= target) return true;
  unsigned long long t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  unsigned int sleep_ns = 1000;
  while (true) {
    __nanosleep(sleep_ns);
    if (sleep_ns < 8000) sleep_ns *= 2;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= target) return true;
    if (*reinterpret_cast<const volatile unsigned int*>(status) != 0u) return false;
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > 2000000000ull) return false;
  }
}

// (at most 64 registers: four blocks per SM once the GEMM CTAs have left,
// one beside a GEMM CTA; measured faster than deeper, fewer blocks)
__global__ void __launch_bounds__(256, 4) apply_stream_kernel(const __grid_constant__ ApplyLaunch L) {
  __shared__ int s_unit;
  // thread 0 claims the block's next unit while the block works on the current
  // one; with a failure already recorded on this workspace it claims nothing
  unsigned int next = 0;
  if (threadIdx.x == 0)
    next = *reinterpret_cast<const volatile unsigned int*>(L.status) != 0u
               ? static_cast<unsigned int>(L.total_units)
               : atomicAdd(L.work, 1u);
  while (true) {
    if (threadIdx.x == 0) {
      int u = static_cast<int>(next);
      if (u < L.total_units) {
        int gi = 0;
        while (gi + 1 < L.n_groups && u >= L.grp[gi + 1].unit_begin) ++gi;
        const ApplyGroup& A = L.grp[gi];
        const int mat = (u - A.unit_begin) / A.units_per_mat;
        if (!wait_done(L.done + A.done_begin + mat, A.done_target, L.status)) {
          atomicOr(L.status, kErrTimeoutApply);
          u = L.total_units;
        }
      }
      s_unit = u;
    }
    // (thread 0's acquire of the counter and this barrier order the last
    // update's stores of O before every thread's loads of it)
    __syncthreads();
    const int u = s_unit;
    __syncthreads();  // s_unit is rewritten by the next claim only after every thread read it
    if (u >= L.total_units) break;
    if (threadIdx.x == 0) next = atomicAdd(L.work, 1u);
    int gi = 0;
    while (gi + 1 < L.n_groups && u >= L.grp[gi + 1].unit_begin) ++gi;
    const ApplyGroup& A = L.grp[gi];
    const int local = u - A.unit_begin;
    const int mat = local / A.units_per_mat;
    const int r0 = (local - mat * A.units_per_mat) * A.unit_rows;
    const int r1 = min(A.r, r0 + A.unit_rows);
    const size_t poff = static_cast<size_t>(mat) * A.r * A.c;
    const size_t ooff = static_cast<size_t>(mat) * A.r * A.ldx;
    const int segs_row = A.c / kStreamSeg;
    const int segs = (r1 - r0) * segs_row;
    for (int g0 = threadIdx.x; g0 < segs; g0 += blockDim.x * kStreamDepth) {
      float4 pa[kStreamDepth], pb[kStreamDepth];
      uint4 ow[kStreamDepth];
      size_t pi[kStreamDepth];
      bool in[kStreamDepth];
#pragma unroll
      for (int d = 0; d < kStreamDepth; ++d) {
        const int g = g0 + static_cast<int>(blockDim.x) * d;
        in[d] = g < segs;
        const int row = r0 + (in[d] ? g / segs_row : 0);
        const int col = in[d] ? (g - (row - r0) * segs_row) * kStreamSeg : 0;
        pi[d] = poff + static_cast<size_t>(row) * A.c + col;
        if (in[d]) {
          pa[d] = __ldcs(reinterpret_cast<const float4*>(A.param + pi[d]));
          pb[d] = __ldcs(reinterpret_cast<const float4*>(A.param + pi[d] + 4));
          ow[d] = __ldcg(reinterpret_cast<const uint4*>(
              A.o + ooff + static_cast<size_t>(row) * A.ldx + col));
        }
      }
#pragma unroll
      for (int d = 0; d < kStreamDepth; ++d) {
        if (!in[d]) continue;
        const uint32_t ws[4] = {ow[d].x, ow[d].y, ow[d].z, ow[d].w};
        float o[kStreamSeg];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[h]));
          o[2 * h] = f.x;
          o[2 * h + 1] = f.y;
        }
        const float k = -A.lr_eff, dec = A.decay;
        __stcs(reinterpret_cast<float4*>(A.param + pi[d]),
               make_float4(fmaf(k, o[0], dec * pa[d].x), fmaf(k, o[1], dec * pa[d].y),
                           fmaf(k, o[2], dec * pa[d].z), fmaf(k, o[3], dec * pa[d].w)));
        __stcs(reinterpret_cast<float4*>(A.param + pi[d] + 4),
               make_float4(fmaf(k, o[4], dec * pb[d].x), fmaf(k, o[5], dec * pb[d].y),
                           fmaf(k, o[6], dec * pb[d].z), fmaf(k, o[7], dec * pb[d].w)));
      }
    }
  }
  // Programmatic dependent of the last update: the grid completes only after
  // it (and so after everything before it in the stream)
  if (blockIdx.x == 0 && threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int MODE>
cudaError_t launch_mode(const PrologueLaunch& l, bool pdl, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(l.total_blocks);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, prologue_kernel<MODE>, l);
}

}  // namespace

cudaError_t launch_apply(const ApplyLaunch& l, bool to_param, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(l.total_blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return to_param ? cudaLaunchKernelEx(&cfg, apply_kernel<true>, l)
                  : cudaLaunchKernelEx(&cfg, apply_kernel<false>, l);
}

cudaError_t launch_apply_stream(const ApplyLaunch& l, int blocks, cudaStream_t s) {
  // shared memory is preferred over L1 (this kernel uses none) so that its
  // blocks can share an SM with a rounds CTA configured for 227 KB
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(apply_stream_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, apply_stream_kernel, l);
}

cudaError_t launch_prologue(const PrologueLaunch& l, int mode, bool pdl, cudaStream_t s) {
  switch (mode) {
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
