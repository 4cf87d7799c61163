// tsa_internal.h -- host helpers shared by the translation units of libtsa.so.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include "../../include/tsa.h"
#include "prefill_params.h"

namespace tsa {
// An NVTX range over one ABI call (named after the call), so that a profiler
// timeline shows which launches each call made. Header-only NVTX: without an
// attached tool the push and pop are no-ops.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
tsa_status fail(tsa_status s, const char* fmt, ...);
tsa_status cuda_fail(cudaError_t e, const char* what);
tsa_status check_config(const tsa_config* c);
size_t state_floats_per_head(const tsa_config* c);
int device_sm_count();
// Raise a kernel's dynamic shared-memory limit to `smem` bytes once per device
// (the attribute call costs microseconds of host time per prefill otherwise).
cudaError_t set_smem_once(const void* kernel, int smem);
// max_scratch: only span counts whose scratch fits are considered (one span
// needs none, so a plan always exists)
tsa_status make_plan(const tsa_config* c, long long N, int num_sms, tsa_plan* pl,
                     size_t max_scratch = SIZE_MAX);
tsa_status launch_prefill(const tsa_config* c, const tsa_plan& pl, PrefillParams p, cudaStream_t s);

// Tensor-core prefill (prefill_tc.cu).
struct TcSlicing {
  int nb, nmax, n_slices, ring;
  int c0[4], w[4];
  size_t smem;
};
bool tc_supported(int dk, int nt);
bool tc_slicing(int dk, int nt, int dv, TcSlicing* ts);
tsa_status launch_prefill_tc(const tsa_config* c, const tsa_plan& pl, const PrefillParams& p, cudaStream_t s);
// The span-state pass and scan of a multi-span bf16 plan (value-sliced).
tsa_status launch_span_states_tc(int dk, int nt, const tsa_plan& pl, const PrefillParams& p, cudaStream_t s);
// bf16 prefill with the head state shared by a cluster of CTAs
// (prefill_pair.cu): whether a layout exists, its CTAs per (head, span) and
// its shared memory.
bool pair_fits(int dk, int nt, int dv, int* cs, size_t* smem);
tsa_status launch_prefill_pair(const tsa_config* c, const tsa_plan& pl, const PrefillParams& p, cudaStream_t s);
tsa_status device_error_word(int** out);
// The testing hooks' current settings: the bound of each wait and whether
// the fp32 output pass withholds its first publication.
void tc_debug_params(unsigned long long* wait_ns, int* withhold);
// fp32 tensor-core prefill with split-bf16 operands (prefill_tc32.cu).
bool tc32_fits(int dk, int nt, int dv);
size_t tc32_smem(int dk, int nt, int dv);
tsa_status launch_prefill_tc32(const tsa_config* c, const tsa_plan& pl, const PrefillParams& p, cudaStream_t s);
// The final state only: the fp32 span pass and the scan.
tsa_status launch_states_tc32(const tsa_config* c, const tsa_plan& pl, const PrefillParams& p, cudaStream_t s);
// Plan and launches of tsa_prefill_states (tsa_abi.cu).
tsa_status make_states_plan(const tsa_config* c, long long N, int num_sms, tsa_plan* pl);
tsa_status launch_states(const tsa_config* c, const tsa_plan& pl, PrefillParams p, cudaStream_t s);
tsa_status take_device_error();
bool tc_append_fits(int dk, int nt, int dv, size_t* smem);
// The device-check reports of the translation units with kernels (debug
// build; each copies out and clears its own report, debug_check.cuh).
cudaError_t debug_report_abi(unsigned long long* out);
cudaError_t debug_report_tc(unsigned long long* out);
cudaError_t debug_report_tc32(unsigned long long* out);
cudaError_t debug_report_pair(unsigned long long* out);
cudaError_t debug_report_short(unsigned long long* out);
// Short-segment prefill, state resident in shared memory (prefill_short.cu).
bool short_supported(int dk, int nt, int dv);
size_t short_smem(int dk, int nt, int dv);
tsa_status launch_prefill_short(const tsa_config* c, const PrefillParams& p, cudaStream_t s);
}  // namespace tsa
