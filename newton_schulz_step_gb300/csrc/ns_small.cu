// ns_small.cu -- the whole Muon step for matrices with min(rows, cols) < 64
// (e.g. the 1x12 smear gate and 12x768 attention gates of the d=768 GPT-2
// model in "Muon Custom Sizing 实战", section 2.1), one CTA per matrix, fp32
// on the CUDA cores.  At these sizes the tensor cores have nothing to do, and
// bf16 rounding of a 1 x n matrix's single singular value moves the result by
// several percent, so the iteration runs in fp32 throughout.
//
// Steps (same arithmetic as the tensor-core path, different precision):
//   buf <- buf + (1 - beta)(g - buf);  u <- g + beta (buf - g)  (or buf, or g)
//   X = u (u^T if rows > cols) / (||u||_F + eps)                (m x n, fp32, workspace)
//   steps x:  A = X X^T;  B = b A + c A A;  X = a X + B X       (A, B in shared memory)
//   p <- (1 - lr wd) p - lr_eff X^(T)   or   out <- bf16(X^(T))
//
// X stays in dynamic shared memory when every small matrix of the launch fits
// (m n <= kSmallSmemFloats), else in the fp32 workspace.  The kernel lets the
// next grid in the stream (the grouped prologue) start at once: the two are
// independent and run side by side.
#include "internal.h"

namespace muon {

namespace {

constexpr int kSmallThreads = 256;
constexpr int kBatch = 8;  // elements per thread in flight in the elementwise passes
constexpr int kSmallLd = 64;  // shared A, B are 64 x 64 with zero padding

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  for (int k = 0; k < kSmallThreads / 32; ++k) t += red[k];
  __syncthreads();
  return t;
}

// X = a X + B X for the columns owned by this thread; MP >= m bounds the
// unrolled register column (B is zero-padded past m).
template <int MP>
__device__ __forceinline__ void update_columns(float* X, const float* Bs, int m, int n, float a) {
  for (int k = threadIdx.x; k < n; k += kSmallThreads) {
    float xv[MP];
#pragma unroll
    for (int l = 0; l < MP; ++l) xv[l] = (l < m) ? X[static_cast<size_t>(l) * n + k] : 0.f;
    for (int i = 0; i < m; ++i) {
      float acc = 0.f;
#pragma unroll
      for (int l = 0; l < MP; ++l) acc = fmaf(Bs[i * kSmallLd + l], xv[l], acc);
      float* xi = X + static_cast<size_t>(i) * n + k;
      *xi = fmaf(a, *xi, acc);
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(kSmallThreads) small_ns_kernel(
    const __grid_constant__ SmallLaunch L) {
  __shared__ float As[kSmallLd * kSmallLd];
  __shared__ float Bs[kSmallLd * kSmallLd];
  __shared__ float red[kSmallThreads / 32];
  extern __shared__ float xs_dyn[];

  // the next grid (independent work) may start right away
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // a failure already recorded on this workspace: this call changes nothing
  if (*reinterpret_cast<const volatile unsigned int*>(L.status) != 0u) return;

  int gi = 0;
  while (gi + 1 < L.n_groups && static_cast<int>(blockIdx.x) >= L.grp[gi + 1].block_begin) ++gi;
  const SmallGroup& G = L.grp[gi];
  const int mat = blockIdx.x - G.block_begin;
  const int r = G.r, c = G.c;
  const bool tall = r > c;
  const int m = tall ? c : r;
  const int n = tall ? r : c;
  const size_t moff = static_cast<size_t>(mat) * r * c;
  const int total = r * c;
  float* X = L.x_in_smem ? xs_dyn : G.x + moff;  // m x n, row-major
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const float beta = L.beta;

  // 1. momentum, Nesterov blend, X = u (transposed when tall), sum(u^2); the
  //    loads of kBatch elements per thread are issued before any use, so the
  //    pass costs a few memory latencies rather than one per element
  float ss = 0.f;
  for (int e0 = tid; e0 < total; e0 += kSmallThreads * kBatch) {
    float gv[kBatch], bv[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int e = e0 + k * kSmallThreads;
      gv[k] = bv[k] = 0.f;
      if (e < total) {
        gv[k] = (G.gdt == MUON_BF16)
                    ? __bfloat162float(static_cast<const __nv_bfloat16*>(G.g)[moff + e])
                    : static_cast<const float*>(G.g)[moff + e];
        if (MODE != kPrologueNsOnly) bv[k] = G.buf[moff + e];
      }
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int e = e0 + k * kSmallThreads;
      if (e >= total) break;
      const int ri = e / c, ci = e - ri * c;
      float u = gv[k];
      if (MODE != kPrologueNsOnly) {
        const float nb = fmaf(1.0f - beta, gv[k] - bv[k], bv[k]);
        G.buf[moff + e] = nb;
        u = (MODE == kPrologueNesterov) ? fmaf(beta, nb - gv[k], gv[k]) : nb;
      }
      X[tall ? static_cast<size_t>(ci) * n + ri : static_cast<size_t>(ri) * n + ci] = u;
      ss = fmaf(u, u, ss);
    }
  }
  for (int e = tid; e < kSmallLd * kSmallLd; e += kSmallThreads) {
    As[e] = 0.f;
    Bs[e] = 0.f;
  }
  const float s = 1.0f / (sqrtf(block_sum(ss, red)) + L.eps);
  for (int e = tid; e < total; e += kSmallThreads) X[e] *= s;
  __syncthreads();

  for (int it = 0; it < L.steps; ++it) {
    // A = X X^T: one warp per (i, j >= i) entry, lanes stride over the row
    for (int pr = warp; pr < m * m; pr += kSmallThreads / 32) {
      const int i = pr / m, j = pr - (pr / m) * m;
      if (j < i) continue;
      const float* xi = X + static_cast<size_t>(i) * n;
      const float* xj = X + static_cast<size_t>(j) * n;
      float d = 0.f;
      for (int k = lane; k < n; k += 32) d = fmaf(xi[k], xj[k], d);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      if (lane == 0) {
        As[i * kSmallLd + j] = d;
        As[j * kSmallLd + i] = d;
      }
    }
    __syncthreads();
    // B = b A + c A A
    for (int e = tid; e < m * m; e += kSmallThreads) {
      const int i = e / m, j = e - (e / m) * m;
      float acc = 0.f;
      for (int l = 0; l < m; ++l) acc = fmaf(As[i * kSmallLd + l], As[l * kSmallLd + j], acc);
      Bs[i * kSmallLd + j] = fmaf(L.c, acc, L.b * As[i * kSmallLd + j]);
    }
    __syncthreads();
    // X = a X + B X, one column of X per thread (columns are independent)
    if (m <= 16)
      update_columns<16>(X, Bs, m, n, L.a);
    else if (m <= 32)
      update_columns<32>(X, Bs, m, n, L.a);
    else
      update_columns<64>(X, Bs, m, n, L.a);
    __syncthreads();
  }

  // apply (or write the bf16 result), in the input's orientation, kBatch
  // parameter loads per thread in flight
  for (int e0 = tid; e0 < total; e0 += kSmallThreads * kBatch) {
    float pv[kBatch];
    if (MODE != kPrologueNsOnly) {
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int e = e0 + k * kSmallThreads;
        pv[k] = e < total ? G.param[moff + e] : 0.f;
      }
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int e = e0 + k * kSmallThreads;
      if (e >= total) break;
      const int ri = e / c, ci = e - ri * c;
      const float o =
          X[tall ? static_cast<size_t>(ci) * n + ri : static_cast<size_t>(ri) * n + ci];
      if (MODE == kPrologueNsOnly)
        G.out[moff + e] = __float2bfloat16_rn(o);
      else
        G.param[moff + e] = fmaf(-G.lr_eff, o, L.decay * pv[k]);
    }
  }
}

}  // namespace

cudaError_t launch_small(const SmallLaunch& l, int total_blocks, int max_mn, cudaStream_t s) {
  const size_t smem = l.x_in_smem ? static_cast<size_t>(max_mn) * sizeof(float) : 0;
  // static A, B (32 KB) plus up to 160 KB of X: above the 48 KB default, so
  // the limit is raised once per device and kernel instance
  static int configured[3][64] = {{0}};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  auto run = [&](auto kern, int which) -> cudaError_t {
    if (dev >= 64 || !configured[which][dev]) {
      const cudaError_t ea =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kSmallSmemFloats * sizeof(float)));
      if (ea != cudaSuccess) return ea;
      if (dev < 64) configured[which][dev] = 1;
    }
    kern<<<total_blocks, kSmallThreads, smem, s>>>(l);
    return cudaGetLastError();
  };
  switch (l.mode) {
    case kPrologueNsOnly:
      return run(small_ns_kernel<kPrologueNsOnly>, 0);
    case kPrologueNesterov:
      return run(small_ns_kernel<kPrologueNesterov>, 1);
    case kProloguePlain:
      return run(small_ns_kernel<kProloguePlain>, 2);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace muon
