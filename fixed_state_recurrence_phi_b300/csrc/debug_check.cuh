// debug_check.cuh -- device-side checks of the library's debug build.
//
// Compiled with -DTSA_DEBUG (libtsa_debug.so), the tensor-core wrappers
// (tc_ptx.cuh) and the kernels check, before each access:
//   - TMEM: the columns an access or accumulator touches lie inside the 512
//     columns every tensor-core kernel allocates, and a warp's tcgen05.ld/st
//     stays in its own 32-lane quarter (warp index mod 4);
//   - MMA operands in shared memory: the bytes a no-swizzle descriptor spans
//     (rows / 8 core-matrix groups SBO apart, two core matrices LBO apart
//     along K = 16) lie inside the CTA's dynamic shared memory;
//   - TMA: the innermost coordinate of a tiled copy is a multiple of 8
//     elements (every map this library encodes starts its boxes at x = 0) and
//     a tiled store starts at no negative coordinate; a bulk copy has 16-byte
//     aligned addresses and size and ends inside shared memory;
//   - state and work indices: a CTA's (head, span) lies inside the launch, a
//     state element lies inside its head's state.
// A failed check records what failed and two values in a report word of its
// translation unit (the first failure wins), skips the access (a load returns
// zeros, an MMA or copy is not issued) and lets the kernel run on: a skipped
// copy leaves its barrier short, so the bounded wait for it gives up. There is
// no trap. tsa_sync_status collects the reports of every translation unit and
// returns TSA_ERR_DEVICE_CHECK with the first one in tsa_last_error.
//
// Without TSA_DEBUG every check is the constant true: the release library is
// unchanged.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace tsa {
namespace dbg {

enum : uint32_t {
  kTmemColumns = 1,   // a = first column, b = columns
  kTmemLanes = 2,     // a = lane field of the address, b = the warp's quarter
  kSmemOperand = 3,   // a = shared-memory start << 32 | first byte, b = end << 32 | one past the last byte
  kTmaCoord = 4,      // a = coordinate index (0 = innermost), b = its value
  kBulkCopy = 5,      // a = shared-memory start << 32 | address, b = end << 32 | bytes
  kStateIndex = 6,    // a = element index, b = elements of the state
  kWorkUnit = 7,      // a = index, b = count
};

#ifdef TSA_DEBUG
constexpr bool kEnabled = true;
// [0] what failed (0 = nothing), [1] a, [2] b, [3] block << 32 | thread
static __device__ unsigned long long g_report[4];

static __device__ __noinline__ void record(uint32_t what, long long a, long long b) {
  if (atomicCAS(&g_report[0], 0ull, (unsigned long long)what) == 0ull) {
    g_report[1] = (unsigned long long)a;
    g_report[2] = (unsigned long long)b;
    const unsigned long long block = blockIdx.x + (unsigned long long)blockIdx.y * gridDim.x;
    g_report[3] = (block << 32) | threadIdx.x;
    __threadfence();
  }
}
#define TSA_DCHECK(cond, what, a, b) \
  ((cond) ? true : (::tsa::dbg::record((what), (long long)(a), (long long)(b)), false))
#else
constexpr bool kEnabled = false;
__host__ __device__ constexpr bool pass() { return true; }
#define TSA_DCHECK(cond, what, a, b) ::tsa::dbg::pass()
#endif
// n elements from index idx lie inside a state (or state area) of `elems`
#define TSA_DCHECK_STATE(idx, n, elems) \
  TSA_DCHECK((size_t)(idx) + (size_t)(n) <= (size_t)(elems), ::tsa::dbg::kStateIndex, (idx), (elems))

}  // namespace dbg
}  // namespace tsa

// The host side of one translation unit's report: copy it out (4 words) and
// clear it. Returns the CUDA error of the copies. Without TSA_DEBUG it reports
// nothing.
#ifdef TSA_DEBUG
#define TSA_DEBUG_REPORT_READER(fn)                                                    \
  cudaError_t fn(unsigned long long* out) {                                           \
    cudaError_t e = cudaMemcpyFromSymbol(out, ::tsa::dbg::g_report, 4 * sizeof(unsigned long long)); \
    if (e != cudaSuccess || out[0] == 0) return e;                                     \
    const unsigned long long zero[4] = {0, 0, 0, 0};                                   \
    return cudaMemcpyToSymbol(::tsa::dbg::g_report, zero, sizeof(zero));               \
  }
#else
#define TSA_DEBUG_REPORT_READER(fn)                     \
  cudaError_t fn(unsigned long long* out) {            \
    out[0] = out[1] = out[2] = out[3] = 0;             \
    return cudaSuccess;                                 \
  }
#endif
