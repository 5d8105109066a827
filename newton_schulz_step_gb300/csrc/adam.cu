// adam.cu -- the DistAdam update of the parameters Muon does not take
// (embeddings, output head, scalars), as one fused HBM-streaming kernel.
//
// Per element, in the order of the DistAdam step() printed in "将 Adam 梯度同步
// （Reduce-Scatter）移入反向 Hook…", section 改动二:
//   p <- p * (1 - lr wd)                 (decoupled decay, skipped when wd == 0)
//   m <- b1 m + (1 - b1) g
//   v <- b2 v + (1 - b2) g^2
//   p <- p - step_size * m / (sqrt(v) + eps),  step_size = lr sqrt(1-b2^t)/(1-b1^t)
// The host folds lr, wd and the bias corrections into two floats per tensor
// (step_size, decay), so the kernel is three fp32 streams in, one gradient
// stream in, three fp32 streams out: 26 bytes per element with bf16 gradients,
// 28 with fp32.  Nothing is reused, so the bound is HBM bandwidth.
//
// Layout of the work: each tensor is cut into units of kAdamUnit elements;
// a persistent grid of 256-thread blocks walks the units of all tensors of the
// launch.  A thread owns four float4 lanes of a unit, spaced one block-width
// apart, so every warp instruction touches 512 contiguous bytes; all loads of a
// unit are issued before any arithmetic (16 independent 16-byte loads per
// thread in flight).  The last unit of a tensor may be ragged: whole vectors go
// the vector path, the final 1-3 elements a scalar path.
#include <mutex>

#include "internal.h"

namespace muon {
namespace {

constexpr int kAdamThreads = 256;
constexpr int kAdamVecs = 4;  // float4 lanes per thread per unit

struct Vals {
  float4 p, m, v, g;
};

__device__ __forceinline__ float4 load_grad4(const void* g, bool bf16, long long e) {
  if (bf16) {
    const uint2 raw = __ldcs(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(g) + e));
    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
    const float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
    return make_float4(a.x, a.y, b.x, b.y);
  }
  return __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(g) + e));
}

__device__ __forceinline__ float load_grad1(const void* g, bool bf16, long long e) {
  return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(g)[e])
              : static_cast<const float*>(g)[e];
}

struct Coef {
  float b1, omb1, b2, omb2, eps, step_size, decay;
};

// One element of the update; p, m, v in/out.
__device__ __forceinline__ void adam_elem(float& p, float& m, float& v, float g, const Coef& k) {
  p = p * k.decay;
  m = k.b1 * m + k.omb1 * g;
  v = k.b2 * v + k.omb2 * (g * g);
  const float denom = sqrtf(v) + k.eps;
  p = p - (m / denom) * k.step_size;
}

__global__ void __launch_bounds__(kAdamThreads) adam_kernel(const __grid_constant__ AdamLaunch L) {
  for (long long u = blockIdx.x; u < L.total_units; u += gridDim.x) {
    // tensor owning unit u: last i with unit_begin <= u
    int lo = 0, hi = L.n_tensors - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (L.t[mid].unit_begin <= u) lo = mid;
      else hi = mid - 1;
    }
    const AdamTensor& T = L.t[lo];
    const Coef k{L.beta1, 1.f - L.beta1, L.beta2, 1.f - L.beta2, L.eps, T.step_size, T.decay};
    const long long base = (u - T.unit_begin) * kAdamUnit;
    const bool bf16 = T.g_bf16 != 0;

    if (base + kAdamUnit <= T.n) {
      // full unit: all loads first, then arithmetic, then stores
      Vals x[kAdamVecs];
#pragma unroll
      for (int j = 0; j < kAdamVecs; ++j) {
        const long long e = base + 4ll * (j * kAdamThreads + threadIdx.x);
        x[j].p = __ldcs(reinterpret_cast<const float4*>(T.p + e));
        x[j].m = __ldcs(reinterpret_cast<const float4*>(T.m + e));
        x[j].v = __ldcs(reinterpret_cast<const float4*>(T.v + e));
        x[j].g = load_grad4(T.g, bf16, e);
      }
#pragma unroll
      for (int j = 0; j < kAdamVecs; ++j) {
        adam_elem(x[j].p.x, x[j].m.x, x[j].v.x, x[j].g.x, k);
        adam_elem(x[j].p.y, x[j].m.y, x[j].v.y, x[j].g.y, k);
        adam_elem(x[j].p.z, x[j].m.z, x[j].v.z, x[j].g.z, k);
        adam_elem(x[j].p.w, x[j].m.w, x[j].v.w, x[j].g.w, k);
      }
#pragma unroll
      for (int j = 0; j < kAdamVecs; ++j) {
        const long long e = base + 4ll * (j * kAdamThreads + threadIdx.x);
        __stcs(reinterpret_cast<float4*>(T.p + e), x[j].p);
        __stcs(reinterpret_cast<float4*>(T.m + e), x[j].m);
        __stcs(reinterpret_cast<float4*>(T.v + e), x[j].v);
      }
    } else {
      // ragged last unit of a tensor
      for (int j = 0; j < kAdamVecs; ++j) {
        const long long e = base + 4ll * (j * kAdamThreads + threadIdx.x);
        if (e + 4 <= T.n) {
          float4 p = *reinterpret_cast<const float4*>(T.p + e);
          float4 m = *reinterpret_cast<const float4*>(T.m + e);
          float4 v = *reinterpret_cast<const float4*>(T.v + e);
          const float4 g = load_grad4(T.g, bf16, e);
          adam_elem(p.x, m.x, v.x, g.x, k);
          adam_elem(p.y, m.y, v.y, g.y, k);
          adam_elem(p.z, m.z, v.z, g.z, k);
          adam_elem(p.w, m.w, v.w, g.w, k);
          *reinterpret_cast<float4*>(T.p + e) = p;
          *reinterpret_cast<float4*>(T.m + e) = m;
          *reinterpret_cast<float4*>(T.v + e) = v;
        } else {
          for (long long i = e; i < T.n && i < e + 4; ++i) {
            float p = T.p[i], m = T.m[i], v = T.v[i];
            adam_elem(p, m, v, load_grad1(T.g, bf16, i), k);
            T.p[i] = p;
            T.m[i] = m;
            T.v[i] = v;
          }
        }
      }
    }
  }
}

}  // namespace

int adam_blocks_per_sm() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (!cached[dev]) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, adam_kernel, kAdamThreads, 0) !=
        cudaSuccess)
      return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

cudaError_t launch_adam(const AdamLaunch& l, int blocks, cudaStream_t s) {
  adam_kernel<<<blocks, kAdamThreads, 0, s>>>(l);
  return cudaGetLastError();
}

}  // namespace muon
