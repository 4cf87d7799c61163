// prefill_pair.cu -- host side of the bf16 tensor-core prefill whose head
// state is shared by a cluster of two CTAs (prefill_pair.cuh): the division
// of the state into tiles, the TMEM and shared-memory layout, the tensor maps
// and the cluster launch.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "tsa_internal.h"
#include "prefill_pair.cuh"
#include "prefill_simt.cuh"

namespace tsa {

// This translation unit's device-check report (debug build; debug_check.cuh).
TSA_DEBUG_REPORT_READER(debug_report_pair)
namespace {

constexpr int kSmemLimit = 227 * 1024;
constexpr int kTmemCols = 512;

int align_up(int x, int a) { return (x + a - 1) / a * a; }

// Shared-memory layout for (ring slots, v buffers, q/k buffers); false if it
// does not fit. The layouts are tried with the deepest ring first: the
// builders hold their inputs in registers, so one q/k buffer costs little.
bool place_smem(PairParams* p, int dk, int s_bytes, int ring, int nvbuf, int nqk) {
  p->qsz = 128 * dk * 2;
  p->vsz = 128 * p->nm * 2;
  int o = 0;
  p->off_q = o; o += nqk * p->qsz;
  p->off_k = o; o += nqk * p->qsz;
  o = align_up(o, 1024);
  p->off_v = o; o += nvbuf * p->vsz;
  o = align_up(o, 1024);
  p->off_p = o; o += 128 * p->kp * 2;
  o = align_up(o, 1024);
  p->off_s = o; o += s_bytes;
  o = align_up(o, 1024);
  p->off_x = o; o += (p->cs == 2) ? (p->dv + 4) * 256 : 0;
  o = align_up(o, 1024);
  p->off_ring = o; o += ring * 16384;
  p->off_bar = o; o += 512;
  if (o > kSmemLimit) return false;
  p->ring = ring; p->nvbuf = nvbuf; p->nqk = nqk;
  return true;
}

}  // namespace

// Division of the state into tiles and the on-chip layout (see
// prefill_pair.cuh). One CTA per (head, span) when all blocks, O and the
// scores fit the 512 TMEM columns; else two: the blocks halved between them,
// an odd block split by columns at the normaliser group.
bool pair_layout(int dk, int nt, int dv, PairParams* p) {
  memset(p, 0, sizeof(*p));
  if (dv % 32 != 0) return false;
  const int D = feat_dim(dk, nt);
  const int nb = (D + 127) / 128;
  const int nm = dv + 16;
  const int ro_last = round_up(D - 128 * (nb - 1), 16);
  auto ro = [&](int f) { return f < nb - 1 ? 128 : ro_last; };
  p->nm = nm;
  p->dv = dv;
  // one CTA
  if (nb <= PR_MAX_TILES && (nb * nm + nm + 128 <= kTmemCols || nb * nm + std::max(nm, 128) <= kTmemCols)) {
    p->cs = 1;
    p->kp = 128;
    p->zc = dv;
    p->ntile[0] = nb;
    int col = 0, so = 0;
    for (int f = 0; f < nb; ++f) {
      p->tile[0][f] = PairTile{f, 0, nm, col, ro(f), so};
      col += nm;
      so += ro(f) * nm * 2;
    }
    p->shared_o = (col + nm + 128 <= kTmemCols) ? 0 : 1;
    p->col_O = col;
    p->col_A = p->shared_o ? col : col + nm;
    const int s_bytes = so;
    const int pref[10][3] = {{4, 2, 2}, {4, 2, 1}, {3, 2, 2}, {3, 2, 1}, {2, 2, 2}, {2, 2, 1},
                           {3, 1, 2}, {3, 1, 1}, {2, 1, 2}, {2, 1, 1}};
    for (auto& c : pref)
      if (place_smem(p, dk, s_bytes, c[0], c[1], c[2])) return true;
    return false;
  }
  // two CTAs
  p->cs = 2;
  p->kp = 64;
  const bool odd = (nb % 2) == 1;
  p->zc = odd ? dv / 2 : dv;
  const int half_blocks = nb / 2;
  int cols[2] = {0, 0}, sb[2] = {0, 0};
  for (int rr = 0; rr < 2; ++rr) {
    int n = 0;
    for (int f = rr * half_blocks; f < (rr + 1) * half_blocks; ++f) {
      if (n >= PR_MAX_TILES) return false;
      p->tile[rr][n++] = PairTile{f, 0, nm, cols[rr], ro(f), sb[rr]};
      cols[rr] += nm;
      sb[rr] += ro(f) * nm * 2;
    }
    if (odd) {
      const int f = nb - 1;
      const int lo = rr == 0 ? 0 : p->zc + 16, w = rr == 0 ? p->zc + 16 : nm - (p->zc + 16);
      if (w > 0) {
        if (n >= PR_MAX_TILES) return false;
        p->tile[rr][n++] = PairTile{f, lo, w, cols[rr], ro(f), sb[rr]};
        cols[rr] += w;
        sb[rr] += ro(f) * w * 2;
      }
    }
    p->ntile[rr] = n;
  }
  const int cmax = std::max(cols[0], cols[1]);
  if (cmax + nm + 64 <= kTmemCols) {
    p->shared_o = 0;
    p->col_O = cmax;
    p->col_A = cmax + nm;
  } else if (cmax + nm <= kTmemCols) {
    p->shared_o = 1;
    p->col_O = p->col_A = cmax;
  } else {
    return false;
  }
  const int s_bytes = std::max(sb[0], sb[1]);
  const int pref[10][3] = {{4, 2, 2}, {4, 2, 1}, {3, 2, 2}, {3, 2, 1}, {2, 2, 2}, {2, 2, 1},
                           {3, 1, 2}, {3, 1, 1}, {2, 1, 2}, {2, 1, 1}};
  for (auto& c : pref)
    if (place_smem(p, dk, s_bytes, c[0], c[1], c[2])) return true;
  return false;
}

bool pair_fits(int dk, int nt, int dv, int* cs, size_t* smem) {
  PairParams p;
  if (!pair_layout(dk, nt, dv, &p)) return false;
  *cs = p.cs;
  *smem = (size_t)p.off_bar + 512;
  return true;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static std::mutex mu;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!fn) {
    void* q = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault, &r) ==
            cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(q);
  }
  return fn;
}

// [heads][N][inner] bf16 as 4-D (8, N, inner/8, heads); a box (8, 128,
// groups, 1) lands as [group][token][8], the core-matrix layout.
tsa_status make_tmap_bf16(CUtensorMap* m, const void* base, int inner, long long N, int heads, int groups) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return fail(TSA_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
  cuuint64_t dims[4] = {8, (cuuint64_t)N, (cuuint64_t)(inner / 8), (cuuint64_t)heads};
  cuuint64_t strides[3] = {(cuuint64_t)inner * 2, 16, (cuuint64_t)N * inner * 2};
  cuuint32_t box[4] = {8, (cuuint32_t)TC_C, (cuuint32_t)groups, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TSA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return TSA_OK;
}

template <int DK, int NT>
tsa_status launch_pair(const tsa_plan& pl, const PrefillParams& pp, cudaStream_t s) {
  PairParams p;
  if (!pair_layout(DK, NT, pp.dv, &p)) return fail(TSA_ERR_UNSUPPORTED, "no two-CTA layout for this shape");
  p.out = pp.out; p.states = pp.states; p.scratch = pp.scratch;
  p.N = pp.N; p.heads = pp.heads; p.n_spans = pl.n_spans;
  p.chunks_per_span = pl.chunks_per_span; p.accumulate = pp.accumulate;
  tc_debug_params(&p.wait_ns, &p.dbg_withhold);
  p.dbg_withhold = (p.dbg_withhold == 2);   // hook 2: rank 0's first partial rows
  tsa_status st = device_error_word(&p.err);
  if (st != TSA_OK) return st;
  // the span pass and scan of a multi-span plan: the value-sliced kernels
  if (pl.n_spans > 1) {
    st = launch_span_states_tc(DK, NT, pl, pp, s);
    if (st != TSA_OK) return st;
  }
  CUtensorMap mq, mk, mv;
  if ((st = make_tmap_bf16(&mq, pp.q, DK, pp.N, pp.heads, DK / 8)) != TSA_OK) return st;
  if ((st = make_tmap_bf16(&mk, pp.k, DK, pp.N, pp.heads, DK / 8)) != TSA_OK) return st;
  if ((st = make_tmap_bf16(&mv, pp.v, pp.dv, pp.N, pp.heads, p.zc / 8)) != TSA_OK) return st;
  const int smem = p.off_bar + 512;
  auto kern = span_output_pair_kernel<DK, NT>;
  cudaError_t e = set_smem_once((const void*)kern, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(span_output_pair)");
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)((long long)pp.heads * pl.n_spans * p.cs));
  cfg.blockDim = dim3(PR_THREADS);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  int na = 0;
  at[na].id = cudaLaunchAttributeClusterDimension;
  at[na].val.clusterDim.x = (unsigned)p.cs;
  at[na].val.clusterDim.y = 1;
  at[na].val.clusterDim.z = 1;
  ++na;
  if (pl.n_spans > 1) {   // overlaps the scan; waits for it before reading the prefixes
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  e = cudaLaunchKernelEx(&cfg, kern, p, mq, mk, mv);
  if (e != cudaSuccess) return cuda_fail(e, "launch span_output_pair");
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch span_output_pair");
  return TSA_OK;
}

}  // namespace

tsa_status launch_prefill_pair(const tsa_config* c, const tsa_plan& pl, const PrefillParams& p, cudaStream_t s) {
#define TSA_PR_CASE(DK, NT) \
  if (c->d_k == DK && c->n_terms == NT) return launch_pair<DK, NT>(pl, p, s);
  TSA_PR_CASE(16, 1) TSA_PR_CASE(16, 2) TSA_PR_CASE(16, 3) TSA_PR_CASE(16, 4)
  TSA_PR_CASE(32, 1) TSA_PR_CASE(32, 2) TSA_PR_CASE(32, 3)
#undef TSA_PR_CASE
  return fail(TSA_ERR_UNSUPPORTED, "no two-CTA prefill for d_k=%d n=%d", c->d_k, c->n_terms);
}

}  // namespace tsa
