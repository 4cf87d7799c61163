// tsa_abi.cu -- host side of libtsa.so: argument validation, planning, scratch
// from a library-owned stream-ordered memory pool, and kernel dispatch.
// The C declarations and their contracts are in include/tsa.h.
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <climits>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>

#include "../../include/tsa.h"
#include "tsa_internal.h"
#include "common.cuh"
#include "tc_ptx.cuh"
#include "prefill_simt.cuh"
#include "decode.cuh"

namespace tsa {

static thread_local std::string g_last_error;

tsa_status fail(tsa_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

tsa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(TSA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

// This translation unit's device-check report (debug build; debug_check.cuh).
TSA_DEBUG_REPORT_READER(debug_report_abi)

// What a failed device check was about.
static const char* check_name(unsigned long long what) {
  switch (what) {
    case dbg::kTmemColumns: return "TMEM columns beyond the allocation (first column, columns)";
    case dbg::kTmemLanes: return "TMEM lanes outside the warp's quarter (lane, quarter)";
    case dbg::kSmemOperand:
      return "MMA operand outside the dynamic shared memory (shared-memory start << 32 | first byte, end << 32 | "
             "one past the last byte)";
    case dbg::kTmaCoord: return "TMA coordinate (index, value)";
    case dbg::kBulkCopy:
      return "bulk copy address, size or extent (shared-memory start << 32 | address, end << 32 | bytes)";
    case dbg::kStateIndex: return "state element index (index, elements)";
    case dbg::kWorkUnit: return "work unit beyond the launch (index, count)";
  }
  return "unknown check";
}

// Collect and clear the device-check reports of every translation unit; the
// first one found is returned as TSA_ERR_DEVICE_CHECK. Release build: TSA_OK.
tsa_status take_debug_reports() {
  using Reader = cudaError_t (*)(unsigned long long*);
  const Reader readers[] = {debug_report_abi, debug_report_tc, debug_report_tc32, debug_report_pair,
                            debug_report_short};
  unsigned long long first[4] = {0, 0, 0, 0};
  for (Reader rd : readers) {
    unsigned long long rep[4];
    const cudaError_t e = rd(rep);
    if (e != cudaSuccess) return cuda_fail(e, "read device-check report");
    if (rep[0] != 0 && first[0] == 0) memcpy(first, rep, sizeof(first));
  }
  if (first[0] == 0) return TSA_OK;
  return fail(TSA_ERR_DEVICE_CHECK, "device check failed: %s = (%lld, %lld) [0x%llx, 0x%llx] in block %llu, thread %llu",
              check_name(first[0]), (long long)first[1], (long long)first[2], first[1], first[2], first[3] >> 32,
              first[3] & 0xFFFFFFFFull);
}

// Runs the wrappers' TMEM-column check on 16 columns from `col` without any
// TMEM access (nothing is allocated): with col > 496 it fails, which tests
// the debug build's report path end to end.
__global__ void debug_selftest_kernel(uint32_t col) {
  if (threadIdx.x == 0) tc::chk_tmem_cols(col, 16u);
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape check shared by every call. Returns TSA_OK or the error.
tsa_status check_config(const tsa_config* c) {
  if (!c) return fail(TSA_ERR_INVALID, "config is NULL");
  if (c->B < 1 || c->H < 1) return fail(TSA_ERR_INVALID, "B and H must be >= 1 (got %d, %d)", c->B, c->H);
  if ((long long)c->B * c->H > (1LL << 30)) return fail(TSA_ERR_INVALID, "B*H too large");
  if (c->d_k < 1 || c->d_v < 1 || c->n_terms < 1)
    return fail(TSA_ERR_INVALID, "d_k, d_v and n_terms must be >= 1");
  if (c->dtype != TSA_F32 && c->dtype != TSA_BF16) return fail(TSA_ERR_INVALID, "unknown dtype %d", (int)c->dtype);
  if (c->chunk < 0) return fail(TSA_ERR_INVALID, "chunk must be >= 0");
  if (c->d_k != 16 && c->d_k != 32) return fail(TSA_ERR_UNSUPPORTED, "d_k=%d not built (16, 32)", c->d_k);
  if (c->d_v != 32 && c->d_v != 64 && c->d_v != 128)
    return fail(TSA_ERR_UNSUPPORTED, "d_v=%d not built (32, 64, 128)", c->d_v);
  if (c->n_terms > kMaxTerms) return fail(TSA_ERR_UNSUPPORTED, "n_terms=%d not built (1..5)", c->n_terms);
  // up to 1,024 features (8 blocks of 128) on every path; the order-4 state of
  // d_k = 16 (4,845 features) on the CUDA cores with the state in global memory
  const bool wide_built = c->d_k == 16 && c->n_terms == 5;
  if (feat_dim(c->d_k, c->n_terms) > 1024 && !wide_built)
    return fail(TSA_ERR_UNSUPPORTED, "feature dim %d > 1024 (d_k=%d, n=%d)",
                feat_dim(c->d_k, c->n_terms), c->d_k, c->n_terms);
  if (wide_built && c->d_v != 32 && c->d_v != 64)
    return fail(TSA_ERR_UNSUPPORTED, "n_terms=5 is built for d_v = 32 or 64 (one value slice), not %d", c->d_v);
  return TSA_OK;
}

size_t state_floats_per_head(const tsa_config* c) {
  return (size_t)round_up(feat_dim(c->d_k, c->n_terms), 4) * (size_t)(c->d_v + 1);
}

// ---------------------------------------------------------------------------
// Scratch: one stream-ordered pool per device, kept warm (release threshold at
// max) so steady-state calls do not reach the driver.
// ---------------------------------------------------------------------------
static std::mutex g_pool_mu;
static cudaMemPool_t g_pools[64];
static bool g_pool_ok[64];

tsa_status scratch_alloc(void** p, size_t bytes, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(TSA_ERR_CUDA, "device index %d out of range", dev);
  {
    std::lock_guard<std::mutex> lk(g_pool_mu);
    if (!g_pool_ok[dev]) {
      cudaMemPoolProps props;
      memset(&props, 0, sizeof(props));
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      e = cudaMemPoolCreate(&g_pools[dev], &props);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolCreate");
      uint64_t thr = ~0ull;
      e = cudaMemPoolSetAttribute(g_pools[dev], cudaMemPoolAttrReleaseThreshold, &thr);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolSetAttribute");
      g_pool_ok[dev] = true;
    }
  }
  e = cudaMallocFromPoolAsync(p, bytes, g_pools[dev], s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMallocFromPoolAsync");
  return TSA_OK;
}

tsa_status scratch_free(void* p, cudaStream_t s) {
  cudaError_t e = cudaFreeAsync(p, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync");
  return TSA_OK;
}

cudaError_t set_smem_once(const void* kernel, int smem) {
  static std::mutex mu;
  static std::unordered_map<const void*, int> done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  auto it = done[dev].find(kernel);
  if (it != done[dev].end() && it->second >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) done[dev][kernel] = smem;
  return e;
}

// The preferred shared-memory carveout of a kernel, set once per device (the
// attribute is per device: a second GPU needs its own call).
cudaError_t set_carveout_once(const void* kernel, int carveout) {
  static std::mutex mu;
  static std::unordered_map<const void*, int> done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  auto it = done[dev].find(kernel);
  if (it != done[dev].end() && it->second == carveout) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, carveout);
  if (e == cudaSuccess) done[dev][kernel] = carveout;
  return e;
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// ---------------------------------------------------------------------------
// Planning (host only; exported through tsa_prefill_plan for inspection).
// ---------------------------------------------------------------------------
static size_t simt_smem_bytes(int dk, int nt, int W) {
#define TSA_SMEM_CASE(DK, NT)                                              \
  if (dk == DK && nt == NT)                                                \
    return W == 64 ? SimtLayout<DK, NT, 64>::bytes : SimtLayout<DK, NT, 32>::bytes;
  TSA_SMEM_CASE(16, 1) TSA_SMEM_CASE(16, 2) TSA_SMEM_CASE(16, 3) TSA_SMEM_CASE(16, 4)
  TSA_SMEM_CASE(16, 5) TSA_SMEM_CASE(32, 1) TSA_SMEM_CASE(32, 2) TSA_SMEM_CASE(32, 3)
#undef TSA_SMEM_CASE
  return 0;
}

static constexpr size_t kSmemLimit = 227 * 1024;

// The CUDA-core slice width: 64 where d_v allows and the layout fits, else
// 32. The layouts that keep the state slice in global memory (n = 5; n = 4
// with W = 64) take one slice, W = d_v.
static int simt_width(const tsa_config* c) {
  if (c->n_terms >= 5 || (c->n_terms == 4 && c->d_v == 64)) return c->d_v;
  if (c->n_terms == 4) return 32;
  return (c->d_v % 64 == 0 && simt_smem_bytes(c->d_k, c->n_terms, 64) <= kSmemLimit) ? 64 : 32;
}
static constexpr size_t kSmemPerSm = 228 * 1024;

// Tensor-core plan (bf16 inputs): chunks of 128 tokens, d_v sliced under the
// TMEM budget, one CTA per SM. A span-state chunk costs about half an output
// chunk (phi(K) and the update only).
static tsa_status make_plan_tc(const tsa_config* c, long long N, int num_sms, const TcSlicing& ts,
                               tsa_plan* pl, int path, size_t max_scratch) {
  const int chunk = 128;
  const long long heads = (long long)c->B * c->H;
  const long long n_chunks = (N + chunk - 1) / chunk;
  const long long units = heads * ts.n_slices;
  const long long slots = std::max(1, num_sms);
  int best_s = 1;
  double best_cost = 1e300;
  const long long s_max = std::min<long long>(n_chunks, 1024);
  for (long long s = 1; s <= std::max<long long>(1, s_max); ++s) {
    const long long cps = (n_chunks + s - 1) / s;
    const long long s_eff = cps > 0 ? (n_chunks + cps - 1) / cps : 1;
    if (s_eff != s) continue;
    const long long waves = (units * s_eff + slots - 1) / slots;
    // span states go to scratch and back four times (span pass, scan read and
    // write, prefix read): charged at ~6 TB/s against ~4 us per chunk step
    const double scratch_bytes = (double)heads * s_eff * state_floats_per_head(c) * 4.0;
    const double scratch_cost = s_eff > 1 ? 2.0 + 4.0 * scratch_bytes / 6e12 / 4e-6 : 0.0;
    if (s_eff > 1 && (scratch_bytes > (double)(1ull << 30) || scratch_bytes > (double)max_scratch)) continue;
    const double cost = (double)waves * cps * (s_eff > 1 ? 1.5 : 1.0) + scratch_cost;
    if (cost < best_cost - 1e-9) { best_cost = cost; best_s = (int)s_eff; }
  }
  int wmax = 0;
  for (int k = 0; k < ts.n_slices; ++k) wmax = std::max(wmax, ts.w[k]);
  pl->chunk = chunk;
  pl->slice_width = wmax;
  pl->n_slices = ts.n_slices;
  pl->n_spans = best_s;
  pl->chunks_per_span = n_chunks > 0 ? (int)((n_chunks + best_s - 1) / best_s) : 0;
  pl->smem_bytes = ts.smem;
  pl->ctas_per_sm = 1;
  pl->scratch_bytes = best_s > 1 ? (size_t)heads * best_s * state_floats_per_head(c) * 4 : 0;
  pl->launches = best_s > 1 ? 3 : 1;
  pl->path = path;
  pl->cluster = 1;
  return TSA_OK;
}

// Segments up to this length go to the short-segment prefill when the library
// chooses (chunk = 0): 16 tokens where the tensor-core append form takes the
// shape (bf16 inputs; it is faster from 17 tokens on 1,024 heads), 32
// otherwise; chunk = 16 asks for it at any length.
static constexpr long long kShortAutoMaxN = 32;
static constexpr long long kShortAutoMaxNAppend = 16;
// Token coordinates of the TMA tensor copies and of the kernels'
// chunk indexing are 32-bit: one call takes at most 2^31 - 1 tokens.
static constexpr long long kMaxTokens = INT_MAX;

tsa_status make_plan(const tsa_config* c, long long N, int num_sms, tsa_plan* pl, size_t max_scratch) {
  memset(pl, 0, sizeof(*pl));
  if (N > kMaxTokens) return fail(TSA_ERR_INVALID, "N = %lld exceeds 2^31 - 1 tokens a call", N);
  const bool append_ok = c->dtype == TSA_BF16 && tc_supported(c->d_k, c->n_terms) &&
                         tc_append_fits(c->d_k, c->n_terms, c->d_v, nullptr);
  const long long short_max = append_ok ? kShortAutoMaxNAppend : kShortAutoMaxN;
  // Short segments: each head's state stays in shared memory for the whole
  // segment (read once, written once), 16-token blocks on the CUDA cores.
  if (short_supported(c->d_k, c->n_terms, c->d_v) &&
      (c->chunk == 16 || (c->chunk == 0 && N <= short_max))) {
    const size_t smem = short_smem(c->d_k, c->n_terms, c->d_v);
    pl->chunk = 16;
    pl->slice_width = c->d_v;
    pl->n_slices = 1;
    pl->n_spans = 1;
    pl->chunks_per_span = (int)std::max<long long>(1, std::min<long long>((N + 15) / 16, INT_MAX));
    pl->smem_bytes = smem;
    pl->ctas_per_sm = std::max(1, std::min(2, (int)(kSmemPerSm / (smem + 1024))));   // 2: registers
    pl->scratch_bytes = 0;
    pl->launches = 1;
    pl->path = TSA_PATH_SHORT;
    pl->cluster = 1;
    return TSA_OK;
  }
  if (c->dtype == TSA_BF16 && tc_supported(c->d_k, c->n_terms)) {
    TcSlicing ts;
    if (tc_slicing(c->d_k, c->n_terms, c->d_v, &ts)) {
      if (c->chunk != 0 && c->chunk != 128)
        return fail(TSA_ERR_UNSUPPORTED, "chunk=%d not built for bf16 (0 or 128)", c->chunk);
      // a state that one CTA holds only in value slices: a CTA pair holds it
      // whole, each CTA half of its feature blocks (prefill_pair.cuh)
      int cs = 1;
      size_t psmem = 0;
      if (ts.n_slices > 1 && pair_fits(c->d_k, c->n_terms, c->d_v, &cs, &psmem) && cs == 2) {
        TcSlicing tp = ts;
        tp.n_slices = cs;   // CTAs per (head, span), for the cost of the plan
        tp.w[0] = c->d_v;
        tp.smem = psmem;
        tsa_status st = make_plan_tc(c, N, num_sms, tp, pl, TSA_PATH_TC, max_scratch);
        pl->n_slices = 1;
        pl->slice_width = c->d_v;
        pl->cluster = cs;
        return st;
      }
      tsa_status st = make_plan_tc(c, N, num_sms, ts, pl, TSA_PATH_TC, max_scratch);
      // one chunk of at most 64 tokens (a short append) of a state of at
      // most two feature blocks: the append form, three CTAs per SM
      size_t asmem = 0;
      if (st == TSA_OK && N <= 64 && pl->n_spans == 1 && tc_append_fits(c->d_k, c->n_terms, c->d_v, &asmem)) {
        pl->ctas_per_sm = 3;
        pl->smem_bytes = asmem;
      }
      return st;
    }
  }
  if (c->dtype == TSA_F32 && tc32_fits(c->d_k, c->n_terms, c->d_v) && (c->chunk == 0 || c->chunk == 128)) {
    TcSlicing ts;
    memset(&ts, 0, sizeof(ts));
    ts.nb = (feat_dim(c->d_k, c->n_terms) + 127) / 128;
    ts.n_slices = 1;
    ts.w[0] = c->d_v;
    ts.nmax = c->d_v + 16;
    ts.smem = tc32_smem(c->d_k, c->n_terms, c->d_v);
    return make_plan_tc(c, N, num_sms, ts, pl, TSA_PATH_TC_F32, max_scratch);
  }
  const int chunk = 64;
  if (c->chunk != 0 && c->chunk != chunk)
    return fail(TSA_ERR_UNSUPPORTED, "chunk=%d not built (0 or 64)", c->chunk);
  const int W = simt_width(c);
  const size_t smem = simt_smem_bytes(c->d_k, c->n_terms, W);
  if (smem == 0 || smem > kSmemLimit) return fail(TSA_ERR_UNSUPPORTED, "no kernel fits shared memory");
  const int occ = std::max(1, std::min(2, (int)(kSmemPerSm / (smem + 1024))));
  const long long heads = (long long)c->B * c->H;
  const int n_slices = c->d_v / W;
  const long long n_chunks = (N + chunk - 1) / chunk;
  const long long units = heads * n_slices;
  const long long slots = (long long)std::max(1, num_sms) * occ;
  int best_s = 1;
  double best_cost = 1e300;
  const long long s_max = std::min<long long>(n_chunks, 1024);
  for (long long s = 1; s <= std::max<long long>(1, s_max); ++s) {
    const long long cps = (n_chunks + s - 1) / s;
    const long long s_eff = cps > 0 ? (n_chunks + cps - 1) / cps : 1;
    if (s_eff != s) continue;
    const long long waves = (units * s_eff + slots - 1) / slots;
    // span_state costs about 0.45 of a span_output chunk; the scan and the
    // two extra launches about one chunk.
    if (s_eff > 1 && (double)heads * s_eff * state_floats_per_head(c) * 4.0 > (double)max_scratch) continue;
    const double cost = (double)waves * cps * (s_eff > 1 ? 1.45 : 1.0) + (s_eff > 1 ? 1.0 : 0.0);
    if (cost < best_cost - 1e-9) { best_cost = cost; best_s = (int)s_eff; }
  }
  pl->chunk = chunk;
  pl->slice_width = W;
  pl->n_slices = n_slices;
  pl->n_spans = best_s;
  pl->chunks_per_span = n_chunks > 0 ? (int)((n_chunks + best_s - 1) / best_s) : 0;
  pl->smem_bytes = smem;
  pl->ctas_per_sm = occ;
  pl->scratch_bytes = best_s > 1 ? (size_t)heads * best_s * state_floats_per_head(c) * 4 : 0;
  pl->launches = best_s > 1 ? 3 : 1;
  pl->path = TSA_PATH_SIMT;
  pl->cluster = 1;
  return TSA_OK;
}

// ---------------------------------------------------------------------------
// Dispatch
// ---------------------------------------------------------------------------
template <typename T, int DK, int NT, int W>
static tsa_status launch_prefill_simt(const tsa_plan& pl, PrefillParams p, cudaStream_t s) {
  using L = SimtLayout<DK, NT, W>;
  const unsigned grid = (unsigned)((long long)p.heads * pl.n_slices * pl.n_spans);
  cudaError_t e;
  if (pl.n_spans > 1) {
    e = set_smem_once((const void*)span_state_kernel<T, DK, NT, W>, (int)L::bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(span_state)");
    span_state_kernel<T, DK, NT, W><<<grid, 256, L::bytes, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "launch span_state");
    const int elems4 = (int)(L::DPAD * (p.dv + 1) / 4);
    e = launch_span_scan(p.states, p.scratch, p.heads, pl.n_spans, elems4, p.accumulate, s);
    if (e != cudaSuccess) return cuda_fail(e, "launch span_scan");
  }
  e = set_smem_once((const void*)span_output_kernel<T, DK, NT, W>, (int)L::bytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(span_output)");
  span_output_kernel<T, DK, NT, W><<<grid, 256, L::bytes, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch span_output");
  return TSA_OK;
}

template <typename T, int DK, int NT>
static tsa_status dispatch_prefill_w(const tsa_plan& pl, PrefillParams p, cudaStream_t s) {
  if (pl.slice_width == 64) return launch_prefill_simt<T, DK, NT, 64>(pl, p, s);
  return launch_prefill_simt<T, DK, NT, 32>(pl, p, s);
}

template <typename T>
static tsa_status dispatch_prefill(const tsa_config* c, const tsa_plan& pl, PrefillParams p,
                                   cudaStream_t s) {
#define TSA_PF_CASE(DK, NT) \
  if (c->d_k == DK && c->n_terms == NT) return dispatch_prefill_w<T, DK, NT>(pl, p, s);
  TSA_PF_CASE(16, 1) TSA_PF_CASE(16, 2) TSA_PF_CASE(16, 3) TSA_PF_CASE(16, 4) TSA_PF_CASE(16, 5)
  TSA_PF_CASE(32, 1) TSA_PF_CASE(32, 2) TSA_PF_CASE(32, 3)
#undef TSA_PF_CASE
  return fail(TSA_ERR_UNSUPPORTED, "no prefill kernel for d_k=%d n=%d", c->d_k, c->n_terms);
}

// ---------------------------------------------------------------------------
// The final state only (tsa_prefill_states): the span pass of the prefill
// path and the scan over spans, no outputs.
// ---------------------------------------------------------------------------
template <typename T, int DK, int NT, int W>
static tsa_status launch_states_simt(const tsa_plan& pl, PrefillParams p, cudaStream_t s) {
  using L = SimtLayout<DK, NT, W>;
  const unsigned grid = (unsigned)((long long)p.heads * pl.n_slices * pl.n_spans);
  cudaError_t e = set_smem_once((const void*)span_state_kernel<T, DK, NT, W>, (int)L::bytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(span_state)");
  span_state_kernel<T, DK, NT, W><<<grid, 256, L::bytes, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch span_state");
  const int elems4 = (int)(L::DPAD * (p.dv + 1) / 4);
  e = launch_span_scan(p.states, p.scratch, p.heads, pl.n_spans, elems4, p.accumulate, s);
  if (e != cudaSuccess) return cuda_fail(e, "launch span_scan");
  return TSA_OK;
}

template <typename T>
static tsa_status dispatch_states_simt(const tsa_config* c, const tsa_plan& pl, PrefillParams p, cudaStream_t s) {
#define TSA_ST_CASE(DK, NT)                                                  \
  if (c->d_k == DK && c->n_terms == NT)                                      \
    return pl.slice_width == 64 ? launch_states_simt<T, DK, NT, 64>(pl, p, s) \
                                : launch_states_simt<T, DK, NT, 32>(pl, p, s);
  TSA_ST_CASE(16, 1) TSA_ST_CASE(16, 2) TSA_ST_CASE(16, 3) TSA_ST_CASE(16, 4) TSA_ST_CASE(16, 5)
  TSA_ST_CASE(32, 1) TSA_ST_CASE(32, 2) TSA_ST_CASE(32, 3)
#undef TSA_ST_CASE
  return fail(TSA_ERR_UNSUPPORTED, "no span pass for d_k=%d n=%d", c->d_k, c->n_terms);
}

// The plan of a states-only call: the span pass of the tensor-core path for
// the dtype where it applies (bf16: value-sliced; fp32: split operands), else
// the CUDA-core span pass; spans enough to give every SM a CTA (the pass has
// no output part, so more spans cost only the scan's share).
tsa_status make_states_plan(const tsa_config* c, long long N, int num_sms, tsa_plan* pl) {
  memset(pl, 0, sizeof(*pl));
  if (N > kMaxTokens) return fail(TSA_ERR_INVALID, "N = %lld exceeds 2^31 - 1 tokens a call", N);
  const long long heads = (long long)c->B * c->H;
  int chunk = 64, n_slices = 1, slice_w = c->d_v, path = TSA_PATH_SIMT;
  size_t smem = 0;
  TcSlicing ts;
  if (c->dtype == TSA_BF16 && tc_supported(c->d_k, c->n_terms) && tc_slicing(c->d_k, c->n_terms, c->d_v, &ts)) {
    chunk = 128; n_slices = ts.n_slices; slice_w = ts.nmax - 16; path = TSA_PATH_TC; smem = ts.smem;
  } else if (c->dtype == TSA_F32 && tc32_fits(c->d_k, c->n_terms, c->d_v)) {
    chunk = 128; path = TSA_PATH_TC_F32; smem = tc32_smem(c->d_k, c->n_terms, c->d_v);
  } else {
    const int W = simt_width(c);
    smem = simt_smem_bytes(c->d_k, c->n_terms, W);
    if (smem == 0 || smem > kSmemLimit) return fail(TSA_ERR_UNSUPPORTED, "no kernel fits shared memory");
    slice_w = W;
    n_slices = c->d_v / W;
  }
  const long long n_chunks = (N + chunk - 1) / chunk;
  const long long units = heads * n_slices;
  long long spans = std::max<long long>(1, std::min<long long>(n_chunks, (std::max(1, num_sms) + units - 1) / units));
  while (spans > 1 && (double)heads * spans * state_floats_per_head(c) * 4.0 > (double)(1ull << 30)) --spans;
  const long long cps = n_chunks > 0 ? (n_chunks + spans - 1) / spans : 0;
  spans = cps > 0 ? (n_chunks + cps - 1) / cps : 1;
  pl->chunk = chunk;
  pl->slice_width = slice_w;
  pl->n_slices = n_slices;
  pl->n_spans = (int)spans;
  pl->chunks_per_span = (int)cps;
  pl->ctas_per_sm = 1;
  pl->launches = 2;
  pl->smem_bytes = smem;
  pl->scratch_bytes = (size_t)heads * spans * state_floats_per_head(c) * 4;
  pl->path = path;
  pl->cluster = 1;
  return TSA_OK;
}

tsa_status launch_states(const tsa_config* c, const tsa_plan& pl, PrefillParams p, cudaStream_t s) {
  if (pl.path == TSA_PATH_TC) return launch_span_states_tc(c->d_k, c->n_terms, pl, p, s);
  if (pl.path == TSA_PATH_TC_F32) return launch_states_tc32(c, pl, p, s);
  return (c->dtype == TSA_F32) ? dispatch_states_simt<float>(c, pl, p, s)
                               : dispatch_states_simt<__nv_bfloat16>(c, pl, p, s);
}

// Launch the prefill kernels of `pl` for either dtype (shared with the other
// translation units of the library).
tsa_status launch_prefill(const tsa_config* c, const tsa_plan& pl, PrefillParams p,
                          cudaStream_t s) {
  if (pl.path == TSA_PATH_SHORT) return launch_prefill_short(c, p, s);
  if (pl.path == TSA_PATH_TC)
    return pl.cluster == 2 ? launch_prefill_pair(c, pl, p, s) : launch_prefill_tc(c, pl, p, s);
  if (pl.path == TSA_PATH_TC_F32) return launch_prefill_tc32(c, pl, p, s);
  return (c->dtype == TSA_F32) ? dispatch_prefill<float>(c, pl, p, s)
                               : dispatch_prefill<__nv_bfloat16>(c, pl, p, s);
}

template <typename T, int DK, int NT>
static tsa_status dispatch_decode_dv(int dv, DecodeParams p, cudaStream_t s) {
  const unsigned grid = (unsigned)p.heads;
  switch (dv) {
    case 32: decode_kernel<T, DK, NT, 32><<<grid, 256, 0, s>>>(p); break;
    case 64: decode_kernel<T, DK, NT, 64><<<grid, 256, 0, s>>>(p); break;
    case 128: decode_kernel<T, DK, NT, 128><<<grid, 256, 0, s>>>(p); break;
    default: return fail(TSA_ERR_UNSUPPORTED, "d_v=%d", dv);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch decode");
  return TSA_OK;
}

template <typename T>
static tsa_status dispatch_decode(const tsa_config* c, DecodeParams p, cudaStream_t s) {
#define TSA_DC_CASE(DK, NT) \
  if (c->d_k == DK && c->n_terms == NT) return dispatch_decode_dv<T, DK, NT>(c->d_v, p, s);
  TSA_DC_CASE(16, 1) TSA_DC_CASE(16, 2) TSA_DC_CASE(16, 3) TSA_DC_CASE(16, 4) TSA_DC_CASE(16, 5)
  TSA_DC_CASE(32, 1) TSA_DC_CASE(32, 2) TSA_DC_CASE(32, 3)
#undef TSA_DC_CASE
  return fail(TSA_ERR_UNSUPPORTED, "no decode kernel for d_k=%d n=%d", c->d_k, c->n_terms);
}

// phi(x) of `rows` fp32 input rows: out[r][a] = w_a * x_i * x_j * x_l from the
// feature table (index d_k = the constant 1), one thread per (row, feature).
template <int DK, int NT>
__global__ void feature_map_kernel(const float* __restrict__ x, float* __restrict__ out, long long rows) {
  constexpr int D = feat_dim(DK, NT);
  const long long total = rows * D;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const long long r = e / D;
    const int a = (int)(e - r * D);
    const uint32_t code = g_feat<DK, NT>.code[a];
    float v = g_feat<DK, NT>.w[a];
#pragma unroll
    for (int f = 0; f < (NT > 4 ? 4 : 3); ++f) {
      const int i = (int)((code >> (8 * f)) & 255u);
      if (i != DK) v *= x[r * DK + i];
    }
    out[e] = v;
  }
}

static unsigned grid_for(size_t n, unsigned per_block = 256) {
  const size_t b = (n + per_block - 1) / per_block;
  return (unsigned)std::max<size_t>(1, std::min<size_t>(b, 148u * 16u));
}

}  // namespace tsa

using namespace tsa;

extern "C" {

size_t tsa_feature_dim(int d_k, int n_terms) {
  if (d_k < 1 || n_terms < 1 || d_k > 4096 || n_terms > 16) return 0;
  return (size_t)feat_dim(d_k, n_terms);
}

size_t tsa_state_pad_dim(int d_k, int n_terms) {
  const size_t D = tsa_feature_dim(d_k, n_terms);
  return (D + 3) / 4 * 4;
}

size_t tsa_state_elems(const tsa_config* c) {
  if (!c) return 0;
  return tsa_feature_dim(c->d_k, c->n_terms) * (size_t)(c->d_v + 1);
}

size_t tsa_state_bytes(const tsa_config* c) {
  if (!c || c->B < 1 || c->H < 1 || c->d_v < 1) return 0;
  return (size_t)c->B * c->H * tsa_state_pad_dim(c->d_k, c->n_terms) * (size_t)(c->d_v + 1) * 4;
}

tsa_status tsa_feature_index(int d_k, int n_terms, int* idx, float* weight) {
  if (!idx || !weight) return fail(TSA_ERR_INVALID, "NULL output");
  if (d_k < 1 || n_terms < 1) return fail(TSA_ERR_INVALID, "d_k and n_terms must be >= 1");
#define TSA_FI_CASE(DK, NT)                                                  \
  if (d_k == DK && n_terms == NT) {                                          \
    constexpr FeatTab<DK, NT> t = make_feat_tab<DK, NT>();                   \
    constexpr int F = NT > 4 ? NT - 1 : 3;                                   \
    for (int a = 0; a < FeatTab<DK, NT>::D; ++a) {                           \
      for (int f = 0; f < F; ++f) {                                          \
        const int i = (int)((t.code[a] >> (8 * f)) & 255u);                  \
        idx[F * a + f] = (i == DK) ? -1 : i;                                 \
      }                                                                      \
      weight[a] = t.w[a];                                                    \
    }                                                                        \
    return TSA_OK;                                                           \
  }
  TSA_FI_CASE(16, 1) TSA_FI_CASE(16, 2) TSA_FI_CASE(16, 3) TSA_FI_CASE(16, 4) TSA_FI_CASE(16, 5)
  TSA_FI_CASE(32, 1) TSA_FI_CASE(32, 2) TSA_FI_CASE(32, 3)
#undef TSA_FI_CASE
  return fail(TSA_ERR_UNSUPPORTED, "no feature table for d_k=%d n=%d", d_k, n_terms);
}

tsa_status tsa_feature_map(int d_k, int n_terms, int64_t rows, const float* x, float* out, void* stream) {
  NvtxRange nvtx_range("tsa_feature_map");
  if (d_k < 1 || n_terms < 1) return fail(TSA_ERR_INVALID, "d_k and n_terms must be >= 1");
  if (rows < 0) return fail(TSA_ERR_INVALID, "rows must be >= 0");
  if (rows == 0) return TSA_OK;
  if (!x || !out) return fail(TSA_ERR_INVALID, "x and out must be non-NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t total = (size_t)rows * tsa_feature_dim(d_k, n_terms);
#define TSA_FM_CASE(DK, NT)                                                                    \
  if (d_k == DK && n_terms == NT) {                                                            \
    feature_map_kernel<DK, NT><<<grid_for(total), 256, 0, s>>>(x, out, (long long)rows);      \
    cudaError_t e = cudaGetLastError();                                                        \
    return e == cudaSuccess ? TSA_OK : cuda_fail(e, "launch feature_map");                     \
  }
  TSA_FM_CASE(16, 1) TSA_FM_CASE(16, 2) TSA_FM_CASE(16, 3) TSA_FM_CASE(16, 4) TSA_FM_CASE(16, 5)
  TSA_FM_CASE(32, 1) TSA_FM_CASE(32, 2) TSA_FM_CASE(32, 3)
#undef TSA_FM_CASE
  return fail(TSA_ERR_UNSUPPORTED, "no feature table for d_k=%d n=%d", d_k, n_terms);
}

tsa_status tsa_prefill_plan(const tsa_config* c, int64_t N, int num_sms, tsa_plan* out) {
  if (!out) return fail(TSA_ERR_INVALID, "plan output is NULL");
  tsa_status st = check_config(c);
  if (st != TSA_OK) return st;
  if (N < 0) return fail(TSA_ERR_INVALID, "N must be >= 0");
  if (num_sms <= 0) {
    num_sms = device_sm_count();
    if (num_sms <= 0) return fail(TSA_ERR_CUDA, "no CUDA device to size the plan");
  }
  return make_plan(c, (long long)N, num_sms, out);
}

tsa_status tsa_prefill(const tsa_config* c, int64_t N, const void* q, const void* k, const void* v,
                       void* out, float* states, unsigned flags, void* stream) {
  NvtxRange nvtx_range("tsa_prefill");
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
  tsa_plan pl;
  const int sms = device_sm_count();
  if (sms <= 0) return fail(TSA_ERR_CUDA, "no CUDA device");
  st = make_plan(c, (long long)N, sms, &pl);
  if (st != TSA_OK) return st;

  PrefillParams p;
  p.q = q; p.k = k; p.v = v; p.out = out; p.states = states; p.scratch = nullptr;
  p.N = N; p.heads = c->B * c->H; p.dv = c->d_v; p.n_slices = pl.n_slices;
  p.n_spans = pl.n_spans; p.chunks_per_span = pl.chunks_per_span; p.accumulate = acc ? 1 : 0;
  void* scratch = nullptr;
  if (pl.scratch_bytes) {
    st = scratch_alloc(&scratch, pl.scratch_bytes, s);
    if (st != TSA_OK) return st;
    p.scratch = static_cast<float*>(scratch);
  }
  st = launch_prefill(c, pl, p, s);
  if (scratch) {
    tsa_status st2 = scratch_free(scratch, s);
    if (st == TSA_OK) st = st2;
  }
  return st;
}

tsa_status tsa_prefill_states(const tsa_config* c, int64_t N, const void* k, const void* v, float* states,
                              unsigned flags, void* stream) {
  NvtxRange nvtx_range("tsa_prefill_states");
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
  if (!k || !v) return fail(TSA_ERR_INVALID, "k and v must be non-NULL");
  if (!aligned16(k) || !aligned16(v)) return fail(TSA_ERR_INVALID, "k and v must be 16-byte aligned");
  const int sms = device_sm_count();
  if (sms <= 0) return fail(TSA_ERR_CUDA, "no CUDA device");
  tsa_plan pl;
  st = make_states_plan(c, (long long)N, sms, &pl);
  if (st != TSA_OK) return st;
  PrefillParams p;
  memset(&p, 0, sizeof(p));
  p.k = k; p.v = v; p.states = states;
  p.N = N; p.heads = c->B * c->H; p.dv = c->d_v; p.n_slices = pl.n_slices;
  p.n_spans = pl.n_spans; p.chunks_per_span = pl.chunks_per_span; p.accumulate = acc ? 1 : 0;
  void* scratch = nullptr;
  st = scratch_alloc(&scratch, pl.scratch_bytes, s);
  if (st != TSA_OK) return st;
  p.scratch = static_cast<float*>(scratch);
  st = launch_states(c, pl, p, s);
  tsa_status st2 = scratch_free(scratch, s);
  return st != TSA_OK ? st : st2;
}

tsa_status tsa_decode_step(const tsa_config* c, const void* q, const void* k, const void* v,
                           void* out, float* states, void* stream) {
  NvtxRange nvtx_range("tsa_decode_step");
  tsa_status st = check_config(c);
  if (st != TSA_OK) return st;
  if (!q || !k || !v || !out || !states) return fail(TSA_ERR_INVALID, "NULL pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(states))
    return fail(TSA_ERR_INVALID, "pointers must be 16-byte aligned");
  DecodeParams p;
  p.q = q; p.k = k; p.v = v; p.out = out; p.states = states; p.heads = c->B * c->H;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return (c->dtype == TSA_F32) ? dispatch_decode<float>(c, p, s)
                               : dispatch_decode<__nv_bfloat16>(c, p, s);
}

tsa_status tsa_state_merge(const tsa_config* c, float* a, const float* b, void* stream) {
  NvtxRange nvtx_range("tsa_state_merge");
  tsa_status st = check_config(c);
  if (st != TSA_OK) return st;
  if (!a || !b) return fail(TSA_ERR_INVALID, "NULL state pointer");
  if (!aligned16(a) || !aligned16(b)) return fail(TSA_ERR_INVALID, "states must be 16-byte aligned");
  const size_t n4 = tsa_state_bytes(c) / 16;
  const char* pa = reinterpret_cast<const char*>(a);
  const char* pb = reinterpret_cast<const char*>(b);
  const size_t nb = n4 * 16;
  if (pa != pb && pa < pb + nb && pb < pa + nb)
    return fail(TSA_ERR_INVALID, "a and b overlap partially");
  state_merge_kernel<<<grid_for(n4), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<float4*>(a), reinterpret_cast<const float4*>(b), n4);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch state_merge");
  return TSA_OK;
}

tsa_status tsa_state_to_canonical(const tsa_config* c, const float* states, float* dst, void* stream) {
  NvtxRange nvtx_range("tsa_state_to_canonical");
  tsa_status st = check_config(c);
  if (st != TSA_OK) return st;
  if (!states || !dst) return fail(TSA_ERR_INVALID, "NULL pointer");
  const int D = feat_dim(c->d_k, c->n_terms);
  const int heads = c->B * c->H;
  const size_t total = (size_t)heads * D * (c->d_v + 1);
  state_canonical_kernel<<<grid_for(total), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      states, dst, heads, D, round_up(D, 4), c->d_v);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch state_canonical");
  return TSA_OK;
}

tsa_status tsa_sync_status(void* stream) {
  NvtxRange nvtx_range("tsa_sync_status");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  const tsa_status waits = take_device_error();
  // a failed device check (debug build) is reported before the waits it may
  // have cut short
  const tsa_status checks = take_debug_reports();
  return checks != TSA_OK ? checks : waits;
}

int tsa_debug_build(void) { return dbg::kEnabled ? 1 : 0; }

tsa_status tsa_debug_check_selftest(void* stream) {
  NvtxRange nvtx_range("tsa_debug_check_selftest");
  if (!dbg::kEnabled) return fail(TSA_ERR_UNSUPPORTED, "device checks exist only in the debug build");
  debug_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(510u);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "debug_selftest_kernel");
  return TSA_OK;
}

const char* tsa_status_string(tsa_status s) {
  switch (s) {
    case TSA_OK: return "TSA_OK";
    case TSA_ERR_INVALID: return "TSA_ERR_INVALID";
    case TSA_ERR_UNSUPPORTED: return "TSA_ERR_UNSUPPORTED";
    case TSA_ERR_CUDA: return "TSA_ERR_CUDA";
    case TSA_ERR_TIMEOUT: return "TSA_ERR_TIMEOUT";
    case TSA_ERR_DEVICE_CHECK: return "TSA_ERR_DEVICE_CHECK";
  }
  return "TSA_UNKNOWN_STATUS";
}

const char* tsa_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
