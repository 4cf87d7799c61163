// prefill_tc.cu -- host side of the tensor-core prefill: value-column slicing
// under the TMEM budget, TMA tensor maps, launches, and the device error word
// that bounded waits set on time-out.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>
#include <atomic>
#include <mutex>

#include "tsa_internal.h"
#include "prefill_tc.cuh"
#include "prefill_append.cuh"
#include "prefill_simt.cuh"

namespace tsa {

// This translation unit's device-check report (debug build; debug_check.cuh).
TSA_DEBUG_REPORT_READER(debug_report_tc)
namespace {

// Set by a kernel whose bounded wait gave up; read and cleared by
// tsa_sync_status.
__device__ int g_tsa_err;

std::mutex g_mu;
int* g_err_addr[64];
bool g_err_ready[64];

constexpr size_t kSmemLimit = 227 * 1024;
constexpr size_t kSmemPerSm = 228 * 1024;
constexpr int kTmemCols = 512;

// Testing hooks (tsa_debug_set_wait_limit, tsa_debug_withhold_publication).
std::atomic<unsigned long long> g_wait_ns{TC_WAIT_NS};
std::atomic<int> g_withhold{0};

}  // namespace

void tc_debug_params(unsigned long long* wait_ns, int* withhold) {
  *wait_ns = g_wait_ns.load();
  *withhold = g_withhold.load();
}

tsa_status device_error_word(int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(TSA_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ready[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_tsa_err);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    g_err_addr[dev] = static_cast<int*>(p);
    g_err_ready[dev] = true;
  }
  *out = g_err_addr[dev];
  return TSA_OK;
}

tsa_status take_device_error() {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_tsa_err, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_tsa_err, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clear error word");
    return fail(TSA_ERR_TIMEOUT, "a device-side wait timed out (error word %d)", v);
  }
  return TSA_OK;
}

// Split d_v into slices whose TMEM footprint fits: each slice holds the state
// (NB blocks of 128 rows x (W + 16) fp32 columns, the 16 being the normaliser
// group) plus the A/O accumulator (max(128, W + 16) columns). Widths are
// multiples of 16 and as equal as possible.
bool tc_slicing(int dk, int nt, int dv, TcSlicing* ts) {
  memset(ts, 0, sizeof(*ts));
  if (dv % 16 != 0) return false;
  const int D = feat_dim(dk, nt);
  const int nb = (D + 127) / 128;
  int nmax = std::min(dv + 16, (384 / nb) / 16 * 16);
  if (nmax < 32) return false;
  const int wmax = nmax - 16;
  const int units = dv / 16;
  const int s = (dv + wmax - 1) / wmax;
  if (s > TC_MAX_SLICES) return false;
  int c0 = 0, wbig = 0;
  for (int k = 0; k < s; ++k) {
    const int u = units / s + (k < units % s ? 1 : 0);
    ts->w[k] = 16 * u;
    ts->c0[k] = c0;
    c0 += ts->w[k];
    wbig = std::max(wbig, ts->w[k]);
    const int nm = ts->w[k] + 16;
    if (nb * nm + std::max(128, nm) > kTmemCols) return false;
  }
  ts->nb = nb;
  ts->n_slices = s;
  ts->nmax = wbig + 16;
  // three ring slots hide the issuer <-> worker round trip; two if they do not fit
  ts->ring = TC_MAX_RING;
  ts->smem = TcSmem(dk, ts->nmax, nb, ts->ring).total;
  if (ts->smem > kSmemLimit) {
    ts->ring = 2;
    ts->smem = TcSmem(dk, ts->nmax, nb, ts->ring).total;
  }
  return ts->smem <= kSmemLimit;
}

// The append form (append_tc_kernel): one chunk of at most 64 tokens, the
// fp32 state outside TMEM (128 columns per CTA), three CTAs per SM; d_v <= 64
// and at most two feature blocks, the second with at most 64 rows of value
// loads per thread pair.
bool tc_append_fits(int dk, int nt, int dv, size_t* smem) {
  if (!tc_supported(dk, nt) || dv % 16 != 0 || dv < 16 || dv > 64) return false;
  const int D = feat_dim(dk, nt);
  if (D > 256) return false;
  const AppSmem L(dk, dv, D);
  if (L.k1 * (dv / 8) > 2 * TC_WORKERS) return false;
  if (L.total + 1024 > kSmemPerSm / 3) return false;
  if (smem) *smem = L.total;
  return true;
}

bool tc_supported(int dk, int nt) {
  return (dk == 16 && nt >= 1 && nt <= 4) || (dk == 32 && nt >= 1 && nt <= 3);
}

namespace {

// cuTensorMapEncodeTiled, looked up through the runtime so that the library
// carries no link-time dependency on the driver library.
tsa_status encode_fn(PFN_cuTensorMapEncodeTiled_v12000* out) {
  static std::mutex mu;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p)
      return fail(TSA_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  *out = fn;
  return TSA_OK;
}

// [heads][N][inner] bf16 viewed as 4-D (8, N, inner/8, heads) so that a box
// (8, 128, groups, 1) lands in shared memory as [group][token][8] -- the
// core-matrix layout of the MMA operands.
tsa_status make_tmap(CUtensorMap* m, const void* base, int inner, long long N, int heads, int groups,
                     int rows = TC_C) {
  cuuint64_t dims[4] = {8, (cuuint64_t)N, (cuuint64_t)(inner / 8), (cuuint64_t)heads};
  cuuint64_t strides[3] = {(cuuint64_t)inner * 2, 16, (cuuint64_t)N * inner * 2};
  cuuint32_t box[4] = {8, (cuuint32_t)rows, (cuuint32_t)groups, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  tsa_status st = encode_fn(&enc);
  if (st != TSA_OK) return st;
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                                      strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                      CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TSA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return TSA_OK;
}

// The fp32 value rows of each head's state ([heads][DPAD*(dv+1)], rows of dv
// floats) viewed as 4-D (4, D, dv/4, heads), so that a box (4, rows, dv/4, 1)
// lands in shared memory as [c/4][a][4]: the 16 bytes of a row's column
// group are contiguous across rows.
tsa_status make_state_tmap(CUtensorMap* m, const float* states, int D, int dv, int heads, int rows) {
  const size_t per_head = (size_t)round_up(D, 4) * (dv + 1) * 4;
  cuuint64_t dims[4] = {4, (cuuint64_t)D, (cuuint64_t)(dv / 4), (cuuint64_t)heads};
  cuuint64_t strides[3] = {(cuuint64_t)dv * 4, 16, (cuuint64_t)per_head};
  cuuint32_t box[4] = {4, (cuuint32_t)rows, (cuuint32_t)(dv / 4), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  tsa_status st = encode_fn(&enc);
  if (st != TSA_OK) return st;
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(states), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TSA_ERR_CUDA, "cuTensorMapEncodeTiled (states) failed (%d)", (int)r);
  return TSA_OK;
}

template <typename Kern>
cudaError_t set_smem(Kern kernel, int smem) {
  return set_smem_once((const void*)kernel, smem);
}

template <int DK, int NT>
void fill_tc_params(TcParams* p, const tsa_plan& pl, const TcSlicing& ts, const PrefillParams& pp) {
  memset(p, 0, sizeof(*p));
  p->out = pp.out; p->states = pp.states; p->scratch = pp.scratch;
  p->N = pp.N; p->heads = pp.heads; p->dv = pp.dv; p->n_spans = pl.n_spans;
  p->chunks_per_span = pl.chunks_per_span; p->accumulate = pp.accumulate;
  p->n_slices = ts.n_slices; p->nmax = ts.nmax; p->ring = ts.ring;
  for (int k = 0; k < ts.n_slices; ++k) { p->slice_c0[k] = ts.c0[k]; p->slice_w[k] = ts.w[k]; }
  tc_debug_params(&p->wait_ns, &p->dbg_withhold);
  p->dbg_withhold = 0;   // no withheld publication in these kernels
}

// The span-state pass of a multi-span plan (each span's state sum into the
// scratch, value slices as the TMEM budget allows) and the exclusive scan
// over spans.
template <int DK, int NT>
tsa_status launch_span_tc(const tsa_plan& pl, const TcSlicing& ts, const PrefillParams& pp, cudaStream_t s) {
  TcParams p;
  fill_tc_params<DK, NT>(&p, pl, ts, pp);
  tsa_status st = device_error_word(&p.err);
  if (st != TSA_OK) return st;
  CUtensorMap mk, mv;
  if ((st = make_tmap(&mk, pp.k, DK, pp.N, pp.heads, DK / 8)) != TSA_OK) return st;
  if ((st = make_tmap(&mv, pp.v, pp.dv, pp.N, pp.heads, 2)) != TSA_OK) return st;
  const unsigned grid = (unsigned)((long long)pp.heads * ts.n_slices * pl.n_spans);
  const int smem = (int)ts.smem;
  cudaError_t e = set_smem(span_state_tc_kernel<DK, NT>, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(span_state_tc)");
  span_state_tc_kernel<DK, NT><<<grid, TC_THREADS, smem, s>>>(p, mk, mv);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch span_state_tc");
  const int elems4 = (int)(round_up(feat_dim(DK, NT), 4) * (pp.dv + 1) / 4);
  e = launch_span_scan(pp.states, pp.scratch, pp.heads, pl.n_spans, elems4, pp.accumulate, s);
  if (e != cudaSuccess) return cuda_fail(e, "launch span_scan");
  return TSA_OK;
}

template <int DK, int NT>
tsa_status launch_tc(const tsa_plan& pl, const TcSlicing& ts, const PrefillParams& pp, cudaStream_t s) {
  tsa_status st;
  if (pl.n_spans > 1 && (st = launch_span_tc<DK, NT>(pl, ts, pp, s)) != TSA_OK) return st;
  TcParams p;
  fill_tc_params<DK, NT>(&p, pl, ts, pp);
  if ((st = device_error_word(&p.err)) != TSA_OK) return st;
  CUtensorMap mq, mk, mv;
  if ((st = make_tmap(&mq, pp.q, DK, pp.N, pp.heads, DK / 8)) != TSA_OK) return st;
  if ((st = make_tmap(&mk, pp.k, DK, pp.N, pp.heads, DK / 8)) != TSA_OK) return st;
  if ((st = make_tmap(&mv, pp.v, pp.dv, pp.N, pp.heads, 2)) != TSA_OK) return st;
  const unsigned grid = (unsigned)((long long)pp.heads * ts.n_slices * pl.n_spans);
  if constexpr (FeatConst<DK, NT>::NB <= 2) {
    if (pl.ctas_per_sm == 3) {   // the append form (tc_append_fits)
      size_t asmem = 0;
      if (pl.n_spans != 1 || pp.N > APP_KEYS || !tc_append_fits(DK, NT, pp.dv, &asmem))
        return fail(TSA_ERR_UNSUPPORTED, "three CTAs per SM only for one chunk of up to 64 tokens");
      constexpr int D = FeatConst<DK, NT>::D;
      {   // testing hook 3: the append form withholds O's completion
        unsigned long long wn;
        int wh;
        tc_debug_params(&wn, &wh);
        p.dbg_withhold = (wh == 3);
      }
      CUtensorMap ak, av, as;
      if ((st = make_tmap(&ak, pp.k, DK, pp.N, pp.heads, DK / 8, APP_KEYS)) != TSA_OK) return st;
      if ((st = make_tmap(&av, pp.v, pp.dv, pp.N, pp.heads, 2, APP_KEYS)) != TSA_OK) return st;
      if ((st = make_state_tmap(&as, pp.states, D, pp.dv, pp.heads, D < 128 ? D : 128)) != TSA_OK) return st;
      cudaError_t e = set_smem(append_tc_kernel<DK, NT>, (int)asmem);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(append_tc)");
      append_tc_kernel<DK, NT><<<(unsigned)pp.heads, TC_THREADS, asmem, s>>>(p, mq, ak, av, as);
      e = cudaGetLastError();
      if (e != cudaSuccess) return cuda_fail(e, "launch append_tc");
      return TSA_OK;
    }
  }
  if (pl.ctas_per_sm != 1) return fail(TSA_ERR_UNSUPPORTED, "no append form for d_k=%d n=%d", DK, NT);
  const int smem = (int)ts.smem;
  cudaError_t e = set_smem(span_output_tc_kernel<__nv_bfloat16, DK, NT>, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(span_output_tc)");
  span_output_tc_kernel<__nv_bfloat16, DK, NT><<<grid, TC_THREADS, smem, s>>>(p, mq, mk, mv);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch span_output_tc");
  return TSA_OK;
}

}  // namespace

tsa_status launch_span_states_tc(int dk, int nt, const tsa_plan& pl, const PrefillParams& p, cudaStream_t s) {
  TcSlicing ts;
  if (!tc_slicing(dk, nt, p.dv, &ts))
    return fail(TSA_ERR_UNSUPPORTED, "no tensor-core slicing for d_k=%d d_v=%d n=%d", dk, p.dv, nt);
#define TSA_TCS_CASE(DK, NT) \
  if (dk == DK && nt == NT) return launch_span_tc<DK, NT>(pl, ts, p, s);
  TSA_TCS_CASE(16, 1) TSA_TCS_CASE(16, 2) TSA_TCS_CASE(16, 3) TSA_TCS_CASE(16, 4)
  TSA_TCS_CASE(32, 1) TSA_TCS_CASE(32, 2) TSA_TCS_CASE(32, 3)
#undef TSA_TCS_CASE
  return fail(TSA_ERR_UNSUPPORTED, "no tensor-core span pass for d_k=%d n=%d", dk, nt);
}

tsa_status launch_prefill_tc(const tsa_config* c, const tsa_plan& pl, const PrefillParams& p, cudaStream_t s) {
  TcSlicing ts;
  if (!tc_slicing(c->d_k, c->n_terms, c->d_v, &ts))
    return fail(TSA_ERR_UNSUPPORTED, "no tensor-core slicing for d_k=%d d_v=%d n=%d", c->d_k, c->d_v, c->n_terms);
#define TSA_TC_CASE(DK, NT) \
  if (c->d_k == DK && c->n_terms == NT) return launch_tc<DK, NT>(pl, ts, p, s);
  TSA_TC_CASE(16, 1) TSA_TC_CASE(16, 2) TSA_TC_CASE(16, 3) TSA_TC_CASE(16, 4)
  TSA_TC_CASE(32, 1) TSA_TC_CASE(32, 2) TSA_TC_CASE(32, 3)
#undef TSA_TC_CASE
  return fail(TSA_ERR_UNSUPPORTED, "no tensor-core prefill for d_k=%d n=%d", c->d_k, c->n_terms);
}

}  // namespace tsa

extern "C" tsa_status tsa_debug_set_wait_limit(uint64_t ns) {
  tsa::g_wait_ns.store(ns == 0 ? tsa::TC_WAIT_NS : (unsigned long long)ns);
  return TSA_OK;
}

extern "C" tsa_status tsa_debug_withhold_publication(int what) {
  if (what < 0 || what > 3) return tsa::fail(TSA_ERR_INVALID, "withhold must be 0..3 (got %d)", what);
  tsa::g_withhold.store(what);
  return TSA_OK;
}
