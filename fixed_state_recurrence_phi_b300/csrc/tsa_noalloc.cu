// tsa_noalloc.cu -- tsa_prefill_noalloc: the prefill for callers that cannot
// allocate device memory.
//
// tsa_prefill takes its span-state scratch from a stream-ordered memory pool
// the library owns. Some callers cannot let a library allocate: processes that
// hand their whole device-memory budget to their own allocator at start-up,
// serving loops that must not allocate once they are running, and GPUs where
// the stream-ordered allocator is not available (some virtualised setups).
// This entry point instead uses one fixed array in device memory, declared
// below, that exists on every GPU that loads the library until the process
// exits. It calls no cudaMalloc, cudaMallocAsync, cudaFree or other allocating
// routine.
#include <cuda_runtime.h>

#include <mutex>

#include "tsa_internal.h"

namespace tsa {
namespace {

// Largest scratch the call can use: 16 MiB (the span states of e.g. 8 heads x
// 32 spans at d_k=16, d_v=64, n=3 take 10.4 MB).
constexpr size_t kNoAllocScratchBytes = 16u << 20;

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

std::mutex g_mu;
float* g_addr[64];
bool g_ready[64];

// Device address of g_noalloc_scratch on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device, with that device current, and cached for the life of the
// process (a cudaDeviceReset reloads the module and leaves the cached address
// stale; the header tells callers not to reset a device they use this on).
tsa_status scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(TSA_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_ready[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
    g_addr[dev] = static_cast<float*>(p);
    g_ready[dev] = true;
  }
  *out = g_addr[dev];
  return TSA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace tsa

using namespace tsa;

extern "C" tsa_status tsa_prefill_noalloc(const tsa_config* c, int64_t N, const void* q, const void* k,
                                          const void* v, void* out, float* states, unsigned flags,
                                          void* stream) {
  NvtxRange nvtx_range("tsa_prefill_noalloc");
  tsa_status st = check_config(c);
  if (st != TSA_OK) return st;
  if (N < 0) return fail(TSA_ERR_INVALID, "N must be >= 0 (got %lld)", (long long)N);
  if (flags & ~TSA_PREFILL_ACCUMULATE) return fail(TSA_ERR_INVALID, "unknown flags 0x%x", flags);
  if (!states) return fail(TSA_ERR_INVALID, "states is NULL");
  if (!aligned16(states)) return fail(TSA_ERR_INVALID, "states not 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool acc = (flags & TSA_PREFILL_ACCUMULATE) != 0;
  if (N == 0) {
    if (!acc) {
      cudaError_t e = cudaMemsetAsync(states, 0, tsa_state_bytes(c), s);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(states)");
    }
    return TSA_OK;
  }
  if (!q || !k || !v || !out) return fail(TSA_ERR_INVALID, "q, k, v and out must be non-NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(TSA_ERR_INVALID, "q, k, v and out must be 16-byte aligned");
  const int sms = device_sm_count();
  if (sms <= 0) return fail(TSA_ERR_CUDA, "no CUDA device");
  tsa_plan pl;
  // only span counts whose scratch fits the fixed array (fewer spans per head
  // where tsa_prefill would use more)
  st = make_plan(c, (long long)N, sms, &pl, kNoAllocScratchBytes);
  if (st != TSA_OK) return st;
  if (pl.scratch_bytes > kNoAllocScratchBytes)   // not reached: one span needs no scratch
    return fail(TSA_ERR_UNSUPPORTED, "tsa_prefill_noalloc: plan needs %zu bytes of scratch (> %zu)",
                pl.scratch_bytes, kNoAllocScratchBytes);
  PrefillParams p;
  p.q = q; p.k = k; p.v = v; p.out = out; p.states = states; p.scratch = nullptr;
  p.N = N; p.heads = c->B * c->H; p.dv = c->d_v; p.n_slices = pl.n_slices;
  p.n_spans = pl.n_spans; p.chunks_per_span = pl.chunks_per_span; p.accumulate = acc ? 1 : 0;
  if (pl.scratch_bytes) {
    // Every element of the scratch that is read is first written by the span
    // pass of the same call, so nothing needs clearing.
    st = scratch_address(&p.scratch);
    if (st != TSA_OK) return st;
  }
  return launch_prefill(c, pl, p, s);
}
