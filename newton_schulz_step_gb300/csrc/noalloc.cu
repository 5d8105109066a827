// noalloc.cu -- muon_step_noalloc: muon_step for callers that cannot allocate
// device memory, e.g. code running under an allocator that has reserved the
// whole GPU, plug-ins that may only touch memory handed to them, or loops where
// any allocation after start-up is forbidden.  Its scratch is a fixed array
// inside this library instead of a caller-provided workspace.
//
// In host code the array below is only a host-side stand-in: the device address
// returned by cudaGetSymbolAddress is what reaches the kernels.  That address is
// looked up once per device, with the device current, on the first call made
// on that device (so that first call should come before any stream capture).
// Every call then passes it to muon_step, which runs the usual kernels on it.
// All calls on a device share the one array: calls that overlap on the GPU
// (different streams, or different host threads) race on it.
//
// The array starts with the sticky device error word that every workspace
// carries.  Each call clears that word on its stream (after its argument
// checks, before its first kernel), so the word always describes the latest
// call on the device; muon_noalloc_status reads it.
#include <mutex>

#include "internal.h"

namespace {

// 64 MiB per device: enough for muon_workspace_bytes() of, e.g., four 768x3072
// weights or one 2048x2048 weight.  It is held by every GPU that loads this
// library until the process exits.
constexpr size_t kNoAllocScratchBytes = 64ull << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {nullptr};

}  // namespace

namespace muon {

// Device address and size of the scratch on the current device (the address
// is looked up once per device).
muon_status noalloc_scratch(void** out, size_t* bytes) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MUON_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MUON_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  *bytes = kNoAllocScratchBytes;
  return MUON_OK;
}

}  // namespace muon

extern "C" muon_status muon_step_noalloc(float* params, const void* grads, int g_dtype,
                                         float* momentum_buf, int batch, int rows, int cols,
                                         float momentum, int nesterov, float lr,
                                         float weight_decay, float lr_scale, int steps, float a,
                                         float b, float c, float eps, void* stream) {
  const size_t need = muon_workspace_bytes(batch, rows, cols);
  if (need == 0) return MUON_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return MUON_ERR_WORKSPACE;  // beyond the built-in scratch
  void* scratch = nullptr;
  size_t bytes = 0;
  const muon_status s = muon::noalloc_scratch(&scratch, &bytes);
  if (s != MUON_OK) return s;
  // The scratch keeps the previous call's contents.  Everything a call reads
  // was written earlier in the same call, except the sticky error word at its
  // start: a word left set by an earlier call would make every kernel of this
  // one return at entry, so the step clears it first.
  return muon::step_clearing_status(params, grads, g_dtype, momentum_buf, batch, rows, cols,
                                    momentum, nesterov, lr, weight_decay, lr_scale, steps, a, b,
                                    c, eps, scratch, bytes, stream);
}

extern "C" muon_status muon_noalloc_status(void* stream, int clear) {
  void* scratch = nullptr;
  size_t bytes = 0;
  const muon_status s = muon::noalloc_scratch(&scratch, &bytes);
  if (s != MUON_OK) return s;
  return muon_workspace_status(scratch, bytes, stream, clear);
}
