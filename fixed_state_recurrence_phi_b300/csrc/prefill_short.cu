// prefill_short.cu -- host side of the short-segment prefill (state resident
// in shared memory): which shapes it serves, and the launch.
#include <cuda_runtime.h>

#include "tsa_internal.h"
#include "prefill_short.cuh"

namespace tsa {

// This translation unit's device-check report (debug build; debug_check.cuh).
TSA_DEBUG_REPORT_READER(debug_report_short)
namespace {

template <typename T, int DK, int NT, int DV>
tsa_status launch_short_t(const PrefillParams& p, int* err, cudaStream_t s) {
  if constexpr (!short_fits(DK, NT, DV)) {
    return fail(TSA_ERR_UNSUPPORTED, "short-segment prefill does not fit d_k=%d n=%d d_v=%d", DK, NT, DV);
  } else {
    using L = ShortLayout<DK, NT, DV>;
    cudaError_t e = set_smem_once((const void*)short_prefill_kernel<T, DK, NT, DV>, (int)L::bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(short_prefill)");
    ShortParams sp;
    sp.q = p.q;
    sp.k = p.k;
    sp.v = p.v;
    sp.out = p.out;
    sp.states = p.states;
    sp.err = err;
    sp.N = p.N;
    sp.heads = p.heads;
    sp.accumulate = p.accumulate;
    short_prefill_kernel<T, DK, NT, DV><<<(unsigned)p.heads, 256, L::bytes, s>>>(sp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "launch short_prefill");
    return TSA_OK;
  }
}

template <typename T, int DK, int NT>
tsa_status launch_short_dv(int dv, const PrefillParams& p, int* err, cudaStream_t s) {
  switch (dv) {
    case 32: return launch_short_t<T, DK, NT, 32>(p, err, s);
    case 64: return launch_short_t<T, DK, NT, 64>(p, err, s);
    case 128: return launch_short_t<T, DK, NT, 128>(p, err, s);
    default: return fail(TSA_ERR_UNSUPPORTED, "d_v=%d", dv);
  }
}

template <typename T>
tsa_status launch_short(const tsa_config* c, const PrefillParams& p, int* err, cudaStream_t s) {
#define TSA_SH_CASE(DK, NT) \
  if (c->d_k == DK && c->n_terms == NT) return launch_short_dv<T, DK, NT>(c->d_v, p, err, s);
  TSA_SH_CASE(16, 1) TSA_SH_CASE(16, 2) TSA_SH_CASE(16, 3) TSA_SH_CASE(32, 1) TSA_SH_CASE(32, 2)
#undef TSA_SH_CASE
  return fail(TSA_ERR_UNSUPPORTED, "no short-segment prefill for d_k=%d n=%d", c->d_k, c->n_terms);
}

}  // namespace

bool short_supported(int dk, int nt, int dv) {
  const bool built = (dk == 16 && nt >= 1 && nt <= 3) || (dk == 32 && nt >= 1 && nt <= 2);
  return built && short_fits(dk, nt, dv);
}

size_t short_smem(int dk, int nt, int dv) { return short_smem_bytes(dk, nt, dv); }

tsa_status launch_prefill_short(const tsa_config* c, const PrefillParams& p, cudaStream_t s) {
  int* err = nullptr;
  tsa_status st = device_error_word(&err);
  if (st != TSA_OK) return st;
  return (c->dtype == TSA_F32) ? launch_short<float>(c, p, err, s)
                               : launch_short<__nv_bfloat16>(c, p, err, s);
}

}  // namespace tsa
