// prefill_tc32.cu -- host side of the fp32 tensor-core prefill (split-bf16
// operands): when it applies, its fp32 staging tensor maps, and the launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "tsa_internal.h"
#include "prefill_tc32.cuh"
#include "prefill_simt.cuh"

namespace tsa {

// This translation unit's device-check report (debug build; debug_check.cuh).
TSA_DEBUG_REPORT_READER(debug_report_tc32)
namespace {

constexpr size_t kSmemLimit = 227 * 1024;

template <int DK, int NT>
size_t smem_tc32(int dv, int ring) {
  using S = Tc32Shape<DK, NT>;
  return Tc32Smem(DK, dv, dv + 16, S::ROWS, ring).total;
}
// the span pass's own layout (no q staging, q/k tiles or state copies)
template <int DK, int NT>
size_t smem_tc32_span(int dv, int ring) {
  using S = Tc32Shape<DK, NT>;
  return Tc32Smem(DK, dv, dv + 16, S::ROWS, ring, true).total;
}

size_t smem_for(int dk, int nt, int dv, int ring) {
#define TSA_T32_CASE(DK, NT) \
  if (dk == DK && nt == NT) return smem_tc32<DK, NT>(dv, ring);
  TSA_T32_CASE(16, 1) TSA_T32_CASE(16, 2) TSA_T32_CASE(16, 3) TSA_T32_CASE(16, 4)
  TSA_T32_CASE(32, 1) TSA_T32_CASE(32, 2) TSA_T32_CASE(32, 3)
#undef TSA_T32_CASE
  return 0;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static std::mutex mu;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [heads][N][inner] fp32 as 4-D (4, N, inner/4, heads); a box (4, rows,
// cols/4, 1) is a [col/4][token][4] fp32 tile in shared memory.
tsa_status make_tmap32(CUtensorMap* m, const void* base, int inner, long long N, int heads, int cols,
                       int rows = TC_C) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return fail(TSA_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
  cuuint64_t dims[4] = {4, (cuuint64_t)N, (cuuint64_t)(inner / 4), (cuuint64_t)heads};
  cuuint64_t strides[3] = {(cuuint64_t)inner * 4, 16, (cuuint64_t)N * inner * 4};
  cuuint32_t box[4] = {4, (cuuint32_t)rows, (cuuint32_t)(cols / 4), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TSA_ERR_CUDA, "cuTensorMapEncodeTiled (fp32) failed (%d)", (int)r);
  return TSA_OK;
}

// The span pass (each span's state sum into the scratch) and the exclusive
// scan over spans, which also writes the final state. The pass takes its own
// layout (three ring slots where that fits), or the output pass's (`smem`)
// where its own does not fit.
template <int DK, int NT>
tsa_status span_pass32(const tsa_plan& pl, const PrefillParams& pp, const TcParams& p, int smem,
                       const CUtensorMap& mk, const CUtensorMap& mv, cudaStream_t s) {
  using S = Tc32Shape<DK, NT>;
  const unsigned grid = (unsigned)((long long)pp.heads * pl.n_spans);
  TcParams ps = p;
  int smem_s = smem;
  if (smem_tc32_span<DK, NT>(pp.dv, 2) <= kSmemLimit) {
    ps.span_layout = 1;
    ps.ring = (smem_tc32_span<DK, NT>(pp.dv, 3) <= kSmemLimit) ? 3 : 2;
    smem_s = (int)smem_tc32_span<DK, NT>(pp.dv, ps.ring);
  }
  cudaError_t e = set_smem_once((const void*)span_state_tc32_kernel<DK, NT>, smem_s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(span_state_tc32)");
  span_state_tc32_kernel<DK, NT><<<grid, TC_THREADS, smem_s, s>>>(ps, mk, mv);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch span_state_tc32");
  const int elems4 = (int)(round_up(S::D, 4) * (pp.dv + 1) / 4);
  e = launch_span_scan(pp.states, pp.scratch, pp.heads, pl.n_spans, elems4, pp.accumulate, s);
  if (e != cudaSuccess) return cuda_fail(e, "launch span_scan");
  return TSA_OK;
}

// The final state only (tsa_prefill_states): span pass and scan, any number
// of spans.
template <int DK, int NT>
tsa_status states32(const tsa_plan& pl, const PrefillParams& pp, cudaStream_t s) {
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.states = pp.states; p.scratch = pp.scratch;
  p.N = pp.N; p.heads = pp.heads; p.dv = pp.dv; p.n_spans = pl.n_spans;
  p.chunks_per_span = pl.chunks_per_span; p.accumulate = pp.accumulate;
  p.n_slices = 1; p.nmax = pp.dv + 16;
  p.slice_c0[0] = 0; p.slice_w[0] = pp.dv;
  p.ring = (smem_tc32<DK, NT>(pp.dv, 3) <= kSmemLimit) ? 3 : 2;
  const int smem = (int)smem_tc32<DK, NT>(pp.dv, p.ring);
  tc_debug_params(&p.wait_ns, &p.dbg_withhold);
  p.dbg_withhold = (p.dbg_withhold == 1);   // hook 1: this pass's first O
  tsa_status st = device_error_word(&p.err);
  if (st != TSA_OK) return st;
  CUtensorMap mk, mv;
  if ((st = make_tmap32(&mk, pp.k, DK, pp.N, pp.heads, DK)) != TSA_OK) return st;
  if ((st = make_tmap32(&mv, pp.v, pp.dv, pp.N, pp.heads, pp.dv)) != TSA_OK) return st;
  return span_pass32<DK, NT>(pl, pp, p, smem, mk, mv, s);
}

template <int DK, int NT>
tsa_status launch32(const tsa_plan& pl, const PrefillParams& pp, cudaStream_t s) {
  using S = Tc32Shape<DK, NT>;
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.out = pp.out; p.states = pp.states; p.scratch = pp.scratch;
  p.N = pp.N; p.heads = pp.heads; p.dv = pp.dv; p.n_spans = pl.n_spans;
  p.chunks_per_span = pl.chunks_per_span; p.accumulate = pp.accumulate;
  p.n_slices = 1; p.nmax = pp.dv + 16;
  p.slice_c0[0] = 0; p.slice_w[0] = pp.dv;
  p.ring = (smem_tc32<DK, NT>(pp.dv, 3) <= kSmemLimit) ? 3 : 2;
  const int smem = (int)smem_tc32<DK, NT>(pp.dv, p.ring);
  tc_debug_params(&p.wait_ns, &p.dbg_withhold);
  p.dbg_withhold = (p.dbg_withhold == 1);   // hook 1: this pass's first O
  tsa_status st = device_error_word(&p.err);
  if (st != TSA_OK) return st;
  CUtensorMap mq, mk, mv, mo;
  if ((st = make_tmap32(&mq, pp.q, DK, pp.N, pp.heads, DK)) != TSA_OK) return st;
  if ((st = make_tmap32(&mk, pp.k, DK, pp.N, pp.heads, DK)) != TSA_OK) return st;
  if ((st = make_tmap32(&mv, pp.v, pp.dv, pp.N, pp.heads, pp.dv)) != TSA_OK) return st;
  // output stores: one 32-token x dv/2 box per worker warp
  memset(&mo, 0, sizeof(mo));
  if (tc32_out_tma(S::ROWS, pp.dv + 16, pp.dv) &&
      (st = make_tmap32(&mo, pp.out, pp.dv, pp.N, pp.heads, pp.dv / 2, 32)) != TSA_OK)
    return st;
  const unsigned grid = (unsigned)((long long)pp.heads * pl.n_spans);
  cudaError_t e;
  if (pl.n_spans > 1 && (st = span_pass32<DK, NT>(pl, pp, p, smem, mk, mv, s)) != TSA_OK) return st;
  e = set_smem_once((const void*)span_output_tc32_kernel<DK, NT>, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(span_output_tc32)");
  // after the scan: launched with a programmatic dependency, so that its
  // set-up and first input loads overlap the scan (it waits for the scan
  // before reading the prefixes)
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(TC32_OUT_THREADS);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &at;
  cfg.numAttrs = pl.n_spans > 1 ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, span_output_tc32_kernel<DK, NT>, p, mq, mk, mv, mo);
  if (e != cudaSuccess) return cuda_fail(e, "launch span_output_tc32");
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch span_output_tc32");
  return TSA_OK;
}

}  // namespace

// fp32 inputs take the split-bf16 tensor-core path when one CTA can hold the
// whole head: the TMEM state (NB blocks x (d_v + 16) columns) plus the A/O
// accumulator in 512 columns, and the shared memory below the limit.
bool tc32_fits(int dk, int nt, int dv) {
  if (!tc_supported(dk, nt) || dv % 16 != 0) return false;
  const int D = feat_dim(dk, nt), nb = (D + 127) / 128, nm = dv + 16;
  // state, O, A and at least one readout feature tile in separate TMEM columns
  if (tc32_ro_bufs(nb, nm) == 0) return false;
  const size_t sm = smem_for(dk, nt, dv, 2);
  return sm > 0 && sm <= kSmemLimit;
}

size_t tc32_smem(int dk, int nt, int dv) {
  const size_t s3 = smem_for(dk, nt, dv, 3);
  return (s3 > 0 && s3 <= kSmemLimit) ? s3 : smem_for(dk, nt, dv, 2);
}

tsa_status launch_states_tc32(const tsa_config* c, const tsa_plan& pl, const PrefillParams& p, cudaStream_t s) {
#define TSA_S32_CASE(DK, NT) \
  if (c->d_k == DK && c->n_terms == NT) return states32<DK, NT>(pl, p, s);
  TSA_S32_CASE(16, 1) TSA_S32_CASE(16, 2) TSA_S32_CASE(16, 3) TSA_S32_CASE(16, 4)
  TSA_S32_CASE(32, 1) TSA_S32_CASE(32, 2) TSA_S32_CASE(32, 3)
#undef TSA_S32_CASE
  return fail(TSA_ERR_UNSUPPORTED, "no fp32 tensor-core span pass for d_k=%d n=%d", c->d_k, c->n_terms);
}

tsa_status launch_prefill_tc32(const tsa_config* c, const tsa_plan& pl, const PrefillParams& p, cudaStream_t s) {
#define TSA_T32_CASE(DK, NT) \
  if (c->d_k == DK && c->n_terms == NT) return launch32<DK, NT>(pl, p, s);
  TSA_T32_CASE(16, 1) TSA_T32_CASE(16, 2) TSA_T32_CASE(16, 3) TSA_T32_CASE(16, 4)
  TSA_T32_CASE(32, 1) TSA_T32_CASE(32, 2) TSA_T32_CASE(32, 3)
#undef TSA_T32_CASE
  return fail(TSA_ERR_UNSUPPORTED, "no fp32 tensor-core prefill for d_k=%d n=%d", c->d_k, c->n_terms);
}

}  // namespace tsa
