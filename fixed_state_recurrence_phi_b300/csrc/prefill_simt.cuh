// prefill_simt.cuh -- chunked causal prefill on the CUDA cores (fp32 FFMA).
//
// The computation (Expanding Attention, arXiv 2610.20637 abstract: n additive
// states, one rank-one update per token, prefill as a parallel scan; Hacker
// News thread on the paper: (Q'K)V = Q'(KV) inside a chunk, and the "+1"
// column carrying the softmax normaliser). For chunk c of C tokens with the
// state S_{<c} of everything before it:
//     num|den  = phi(Q_c) S_{<c}                       (inter-chunk readout)
//              + mask(T_n(Q_c K_c^T)) [V_c, 1]         (intra-chunk, j <= i)
//     out      = num / den
//     S_{<c+1} = S_{<c} + phi(K_c)^T [V_c, 1]          (chunk-state update)
//
// Work split. A head's sequence is cut into spans of whole chunks; d_v is cut
// into slices of W columns (every slice recomputes the cheap features and the
// normaliser column). Three kernels:
//   span_state  : per (head, slice, span) the span's own state sum -> scratch
//   span_scan   : per head, exclusive prefix over spans (+ the caller's initial
//                 state), and the final state -> `states`
//   span_output : per (head, slice, span) the chunk loop above, starting from
//                 the span's prefix state, carried on chip
// With a single span per head only span_output runs; it reads the initial state
// and writes the final one itself.
//
// On chip (shared memory, fp32): the state slice S[DROWS][W] and z[DROWS]; the
// features are built DT at a time: phiQ^T[DT][C] and phiK[C][DT(+4)].
#pragma once
#include <cstring>
#include "common.cuh"
#include "debug_check.cuh"
#include "prefill_params.h"

namespace tsa {

// Shared-memory layout (floats) for feature tiles of DT features.
template <int DK, int NT, int W, int DT_>
struct SimtLayoutDT {
  static constexpr int D = feat_dim(DK, NT);
  static constexpr int DPAD = round_up(D, 4);
  static constexpr int C = 64;
  static constexpr int DT = DT_;
  static constexpr int NTILE = (D + DT - 1) / DT;
  static constexpr int DROWS = NTILE * DT;
  static constexpr int TN = W / 16;      // value columns per thread
  static constexpr int RPT = DT / 16;    // state rows per thread in the update
  static constexpr int XS = DK + 1;      // x row stride; x[DK] = 1.0
  static constexpr int PKS = DT + 4;     // phiK row stride
  static constexpr int NTHR = 256;
  // Order 4 (NT = 5): the state slice (4,845 rows at d_k = 16) does not fit
  // shared memory; each CTA works on its own slice in global memory instead
  // (in place in the caller's state or in its span's scratch slot, one value
  // slice of W = d_v columns), read and written through L1/L2. Order 3 with
  // 64 columns (969 x 64 floats, 248 KB) takes the same layout: one slice
  // instead of two 32-column ones in shared memory builds every feature tile
  // once and gives each thread 4 x 4 outputs per pair of operand loads.
  static constexpr bool SG = NT >= 5 || (NT == 4 && W == 64);
  static constexpr int oS = 0;
  static constexpr int oZ = oS + (SG ? 0 : DROWS * W);
  static constexpr int oCode = oZ + (SG ? 0 : DROWS);
  static constexpr int oW = oCode + round_up(D, 4);
  static constexpr int oXq = oW + round_up(D, 4);
  static constexpr int oXk = oXq + round_up(C * XS, 4);
  static constexpr int oV = oXk + round_up(C * XS, 4);
  static constexpr int oPT = oV + C * W;
  static constexpr int oPhQ = oPT + C * C;
  static constexpr int oPhK = oPhQ + DT * C;
  static constexpr int total = oPhK + C * PKS;
  static constexpr size_t bytes = (size_t)total * 4;
  static_assert(W == 32 || W == 64, "slice width");
  static_assert(DT == 32 || DT == 64, "feature tile");
  static_assert(C == 64 && NTHR == 256, "thread mapping assumes 64 tokens x 256 threads");
};

// Tiles of 64 features where that layout fits and keeps as many CTAs per SM
// as tiles of 32 (each update thread then holds 4 state rows instead of 2,
// so that its shared-memory loads feed twice the FMAs); else 32.
__host__ __device__ constexpr int simt_ctas(size_t bytes) {
  return bytes > 227 * 1024 ? 0 : (2 * (bytes + 1024) <= 228 * 1024 ? 2 : 1);
}
template <int DK, int NT, int W>
struct SimtDT {
  static constexpr size_t b32 = SimtLayoutDT<DK, NT, W, 32>::bytes;
  static constexpr size_t b64 = SimtLayoutDT<DK, NT, W, 64>::bytes;
  static constexpr int value = (simt_ctas(b64) > 0 && simt_ctas(b64) >= simt_ctas(b32)) ? 64 : 32;
};
template <int DK, int NT, int W>
struct SimtLayout : SimtLayoutDT<DK, NT, W, SimtDT<DK, NT, W>::value> {};

// Load the chunk's x rows (q or k) into smem as fp32 with x[DK] = 1.0; rows at
// or beyond `valid` are zero.
template <typename T, int DK, int XS, int C>
__device__ __forceinline__ void load_x_rows(float* xs, const T* g, int valid, int tid) {
  constexpr int V4 = DK / 4;
  for (int e = tid; e < C * V4; e += 256) {
    const int t = e / V4, c4 = (e % V4) * 4;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < valid) x = Elem<T>::load4(g + (size_t)t * DK + c4);
    xs[t * XS + c4 + 0] = x.x; xs[t * XS + c4 + 1] = x.y;
    xs[t * XS + c4 + 2] = x.z; xs[t * XS + c4 + 3] = x.w;
  }
  for (int t = tid; t < C; t += 256) xs[t * XS + DK] = 1.0f;
}

template <typename T, int W, int C>
__device__ __forceinline__ void load_v_rows(float* vs, const T* g, int dv, int valid, int tid) {
  constexpr int V4 = W / 4;
  for (int e = tid; e < C * V4; e += 256) {
    const int t = e / V4, c4 = (e % V4) * 4;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < valid) x = Elem<T>::load4(g + (size_t)t * dv + c4);
    *reinterpret_cast<float4*>(vs + t * W + c4) = x;
  }
}

// Read (or write) the state slice [a < D][cols c0..c0+W) and, if `with_z`, z.
template <int L_DROWS, int W, int D, int DPAD>
__device__ __forceinline__ void state_slice_in(float* S, float* z, const float* g, int dv, int c0,
                                               int tid) {
  for (int e = tid; e < L_DROWS * (W / 4); e += 256) {
    const int a = e / (W / 4), c4 = (e % (W / 4)) * 4;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a < D) x = *reinterpret_cast<const float4*>(g + (size_t)a * dv + c0 + c4);
    *reinterpret_cast<float4*>(S + a * W + c4) = x;
  }
  for (int a = tid; a < L_DROWS; a += 256) z[a] = (a < D) ? g[(size_t)DPAD * dv + a] : 0.0f;
}

template <int L_DROWS, int W, int D, int DPAD>
__device__ __forceinline__ void state_slice_out(float* g, const float* S, const float* z, int dv,
                                                int c0, bool with_z, int tid) {
  for (int e = tid; e < DPAD * (W / 4); e += 256) {
    const int a = e / (W / 4), c4 = (e % (W / 4)) * 4;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a < D) x = *reinterpret_cast<const float4*>(S + a * W + c4);
    *reinterpret_cast<float4*>(g + (size_t)a * dv + c0 + c4) = x;
  }
  if (with_z)
    for (int a = tid; a < DPAD; a += 256) g[(size_t)DPAD * dv + a] = (a < D) ? z[a] : 0.0f;
}

// Build one feature tile: phiQ^T[a][t] (if WITH_Q) and phiK[t][a] for the DT
// features a0..a0+DT. Key rows at or beyond `valid` get zero features so that
// padding tokens add nothing to the state.
template <int DK, int NT, int W, bool WITH_Q>
__device__ __forceinline__ void build_phi_tile(float* sm, int a0, int valid, int tid) {
  using L = SimtLayout<DK, NT, W>;
  const uint32_t* code = reinterpret_cast<const uint32_t*>(sm + L::oCode);
  const float* wt = sm + L::oW;
  const float* xq = sm + L::oXq;
  const float* xk = sm + L::oXk;
  float* phq = sm + L::oPhQ;
  float* phk = sm + L::oPhK;
  constexpr int FPG = L::DT / 4;                      // features per thread
  const int tok = tid & (L::C - 1), fg = tid >> 6;  // 4 groups of DT/4 features
  float fk[FPG];
#pragma unroll
  for (int u = 0; u < FPG; ++u) {
    const int a = a0 + fg * FPG + u;
    float vq = 0.f, vk = 0.f;
    if (a < L::D) {
      const uint32_t cd = code[a];
      const int i = cd & 255, j = (cd >> 8) & 255, l = (cd >> 16) & 255;
      const float w = wt[a];
      if (WITH_Q) vq = w * xq[tok * L::XS + i] * xq[tok * L::XS + j] * xq[tok * L::XS + l];
      vk = w * xk[tok * L::XS + i] * xk[tok * L::XS + j] * xk[tok * L::XS + l];
      if constexpr (NT > 4) {
        const int m = cd >> 24;
        if (WITH_Q) vq *= xq[tok * L::XS + m];
        vk *= xk[tok * L::XS + m];
      }
    }
    if (tok >= valid) vk = 0.f;
    if (WITH_Q) phq[(fg * FPG + u) * L::C + tok] = vq;
    fk[u] = vk;
  }
#pragma unroll
  for (int u = 0; u < FPG; u += 4)
    *reinterpret_cast<float4*>(phk + tok * L::PKS + fg * FPG + u) = make_float4(fk[u], fk[u + 1], fk[u + 2], fk[u + 3]);
}

// S[a0 + RPT*ta + r][tc*TN + c] += sum_t phiK[t][RPT*ta + r] * V[t][tc*TN + c]
// z[a0 + RPT*ta + r]             += sum_t phiK[t][RPT*ta + r]
// S and z are the CTA's state slice (shared memory, or global memory in the
// SG layout, whose rows stop at D: rows past it are neither read nor written).
template <int DK, int NT, int W>
__device__ __forceinline__ void update_tile(float* sm, float* S, float* z, int a0, int tid) {
  using L = SimtLayout<DK, NT, W>;
  constexpr int TN = L::TN, RPT = L::RPT;
  const float* phk = sm + L::oPhK;
  const float* vs = sm + L::oV;
  const int ta = tid >> 4, tc = tid & 15;
  auto live = [&](int r) { return !L::SG || a0 + RPT * ta + r < L::D; };
  float s[RPT][TN];
#pragma unroll
  for (int r = 0; r < RPT; ++r)
#pragma unroll
    for (int c = 0; c < TN; ++c) s[r][c] = live(r) ? S[(a0 + RPT * ta + r) * W + tc * TN + c] : 0.f;
  float zp[RPT];
#pragma unroll
  for (int r = 0; r < RPT; ++r) zp[r] = 0.f;
#pragma unroll 8
  for (int t = 0; t < L::C; ++t) {
    float kk[RPT];
    if constexpr (RPT == 4) {
      const float4 x = *reinterpret_cast<const float4*>(phk + t * L::PKS + 4 * ta);
      kk[0] = x.x; kk[1] = x.y; kk[2] = x.z; kk[3] = x.w;
    } else {
      const float2 x = *reinterpret_cast<const float2*>(phk + t * L::PKS + 2 * ta);
      kk[0] = x.x; kk[1] = x.y;
    }
    float vv[TN];
    if constexpr (TN == 4) {
      const float4 x = *reinterpret_cast<const float4*>(vs + t * W + tc * 4);
      vv[0] = x.x; vv[1] = x.y; vv[2] = x.z; vv[3] = x.w;
    } else {
      const float2 x = *reinterpret_cast<const float2*>(vs + t * W + tc * 2);
      vv[0] = x.x; vv[1] = x.y;
    }
#pragma unroll
    for (int r = 0; r < RPT; ++r)
#pragma unroll
      for (int c = 0; c < TN; ++c) s[r][c] = fmaf(kk[r], vv[c], s[r][c]);
    if ((t & 15) == tc) {
#pragma unroll
      for (int r = 0; r < RPT; ++r) zp[r] += kk[r];
    }
  }
#pragma unroll
  for (int r = 0; r < RPT; ++r)
#pragma unroll
    for (int c = 0; c < TN; ++c)
      if (live(r)) S[(a0 + RPT * ta + r) * W + tc * TN + c] = s[r][c];
#pragma unroll
  for (int r = 0; r < RPT; ++r)
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) zp[r] += __shfl_xor_sync(0xffffffffu, zp[r], off);
  if (tc == 0) {
#pragma unroll
    for (int r = 0; r < RPT; ++r)
      if (live(r)) z[a0 + RPT * ta + r] += zp[r];
  }
}

// The span pass in the global-state layout: the same update, with this
// thread's state rows of the tile in registers (s) on entry and the rows of
// the tile at pf_a0 (this thread's again: a thread owns the same rows in
// every tile pass) loaded into s before it returns, their loads issued before
// this tile's token loop so that their latency overlaps it; pf_a0 < 0: none.
template <int DK, int NT, int W>
__device__ __forceinline__ void update_tile_sg(float* sm, float* S, float* z, int a0, int pf_a0,
                                               float (&s)[SimtLayout<DK, NT, W>::RPT][SimtLayout<DK, NT, W>::TN],
                                               int tid) {
  using L = SimtLayout<DK, NT, W>;
  constexpr int TN = L::TN, RPT = L::RPT;
  static_assert(L::SG, "global-state layout only");
  const float* phk = sm + L::oPhK;
  const float* vs = sm + L::oV;
  const int ta = tid >> 4, tc = tid & 15;
  float nx[RPT][TN];
#pragma unroll
  for (int r = 0; r < RPT; ++r)
#pragma unroll
    for (int c = 0; c < TN; ++c)
      nx[r][c] = (pf_a0 >= 0 && pf_a0 + RPT * ta + r < L::D) ? S[(pf_a0 + RPT * ta + r) * W + tc * TN + c] : 0.f;
  float zp[RPT];
#pragma unroll
  for (int r = 0; r < RPT; ++r) zp[r] = 0.f;
#pragma unroll 8
  for (int t = 0; t < L::C; ++t) {
    float kk[RPT];
    if constexpr (RPT == 4) {
      const float4 x = *reinterpret_cast<const float4*>(phk + t * L::PKS + 4 * ta);
      kk[0] = x.x; kk[1] = x.y; kk[2] = x.z; kk[3] = x.w;
    } else {
      const float2 x = *reinterpret_cast<const float2*>(phk + t * L::PKS + 2 * ta);
      kk[0] = x.x; kk[1] = x.y;
    }
    float vv[TN];
    if constexpr (TN == 4) {
      const float4 x = *reinterpret_cast<const float4*>(vs + t * W + tc * 4);
      vv[0] = x.x; vv[1] = x.y; vv[2] = x.z; vv[3] = x.w;
    } else {
      const float2 x = *reinterpret_cast<const float2*>(vs + t * W + tc * 2);
      vv[0] = x.x; vv[1] = x.y;
    }
#pragma unroll
    for (int r = 0; r < RPT; ++r)
#pragma unroll
      for (int c = 0; c < TN; ++c) s[r][c] = fmaf(kk[r], vv[c], s[r][c]);
    if ((t & 15) == tc) {
#pragma unroll
      for (int r = 0; r < RPT; ++r) zp[r] += kk[r];
    }
  }
#pragma unroll
  for (int r = 0; r < RPT; ++r)
#pragma unroll
    for (int c = 0; c < TN; ++c)
      if (a0 + RPT * ta + r < L::D) S[(a0 + RPT * ta + r) * W + tc * TN + c] = s[r][c];
#pragma unroll
  for (int r = 0; r < RPT; ++r)
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) zp[r] += __shfl_xor_sync(0xffffffffu, zp[r], off);
  if (tc == 0) {
#pragma unroll
    for (int r = 0; r < RPT; ++r)
      if (a0 + RPT * ta + r < L::D) z[a0 + RPT * ta + r] += zp[r];
  }
#pragma unroll
  for (int r = 0; r < RPT; ++r)
#pragma unroll
    for (int c = 0; c < TN; ++c) s[r][c] = nx[r][c];
}

template <int DK, int NT>
__device__ __forceinline__ void load_feat_table(uint32_t* code, float* w, int tid) {
  constexpr int D = feat_dim(DK, NT);
  for (int a = tid; a < D; a += 256) {
    if constexpr (NT > 4) {   // 38 KB: from global memory, not the constant bank
      code[a] = __ldg(&g_feat<DK, NT>.code[a]);
      w[a] = __ldg(&g_feat<DK, NT>.w[a]);
    } else {
      code[a] = c_feat<DK, NT>.code[a];
      w[a] = c_feat<DK, NT>.w[a];
    }
  }
}

// Zero one head's state block of `elems` floats (a multiple of 4), by one CTA.
__device__ __forceinline__ void zero_block(float* g, size_t elems, int tid) {
  float4* g4 = reinterpret_cast<float4*>(g);
  for (size_t e = tid; e < elems / 4; e += 256) g4[e] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ---------------------------------------------------------------------------
// span_state: the state contribution of one span (one dv slice) -> scratch.
// ---------------------------------------------------------------------------
template <typename T, int DK, int NT, int W>
__global__ void __launch_bounds__(256)
span_state_kernel(PrefillParams p) {
  using L = SimtLayout<DK, NT, W>;
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  const int tid = threadIdx.x;
  const int span = blockIdx.x % p.n_spans;
  const int slice = (blockIdx.x / p.n_spans) % p.n_slices;
  const int head = blockIdx.x / (p.n_spans * p.n_slices);
  TSA_DCHECK(head < p.heads, dbg::kWorkUnit, head, p.heads);
  const int c0 = slice * W;
  const long long t_begin = (long long)span * p.chunks_per_span * L::C;
  const long long t_end = min(p.N, t_begin + (long long)p.chunks_per_span * L::C);

  load_feat_table<DK, NT>(reinterpret_cast<uint32_t*>(sm + L::oCode), sm + L::oW, tid);
  float *S, *z;
  if constexpr (L::SG) {   // the span's sum is built in its scratch slot (one slice, W = d_v)
    float* g = p.scratch + ((size_t)head * p.n_spans + span) * (size_t)L::DPAD * (p.dv + 1);
    zero_block(g, (size_t)L::DPAD * (p.dv + 1), tid);
    S = g;
    z = g + (size_t)L::DPAD * p.dv;
  } else {
    S = sm + L::oS;
    z = sm + L::oZ;
    for (int e = tid; e < L::DROWS * W; e += 256) sm[L::oS + e] = 0.f;
    for (int e = tid; e < L::DROWS; e += 256) sm[L::oZ + e] = 0.f;
  }

  const T* kg = static_cast<const T*>(p.k) + (size_t)head * p.N * DK;
  const T* vg = static_cast<const T*>(p.v) + (size_t)head * p.N * p.dv + c0;
  // global-state layout: this thread's rows of the next tile, prefetched
  float srow[L::RPT][L::TN];
#pragma unroll
  for (int r = 0; r < L::RPT; ++r)
#pragma unroll
    for (int c = 0; c < L::TN; ++c) srow[r][c] = 0.f;   // the slot starts at zero
  for (long long t0 = t_begin; t0 < t_end; t0 += L::C) {
    const int valid = (int)min((long long)L::C, t_end - t0);
    __syncthreads();
    load_x_rows<T, DK, L::XS, L::C>(sm + L::oXk, kg + (size_t)t0 * DK, valid, tid);
    load_v_rows<T, W, L::C>(sm + L::oV, vg + (size_t)t0 * p.dv, p.dv, valid, tid);
    __syncthreads();
    for (int tile = 0; tile < L::NTILE; ++tile) {
      build_phi_tile<DK, NT, W, false>(sm, tile * L::DT, valid, tid);
      __syncthreads();
      if constexpr (L::SG) {
        // the next tile's rows: this chunk's next tile, else the first tile
        // of the next chunk (this thread wrote them itself)
        const int pf = tile + 1 < L::NTILE ? (tile + 1) * L::DT : (t0 + L::C < t_end ? 0 : -1);
        update_tile_sg<DK, NT, W>(sm, S, z, tile * L::DT, pf, srow, tid);
      } else {
        update_tile<DK, NT, W>(sm, sm + L::oS, sm + L::oZ, tile * L::DT, tid);
      }
      __syncthreads();
    }
  }
  if constexpr (!L::SG) {
    __syncthreads();
    float* dst = p.scratch + ((size_t)head * p.n_spans + span) * (size_t)L::DPAD * (p.dv + 1);
    state_slice_out<L::DROWS, W, L::D, L::DPAD>(dst, sm + L::oS, sm + L::oZ, p.dv, c0, slice == 0, tid);
  }
}

// ---------------------------------------------------------------------------
// span_scan: exclusive prefix of span states, per head and element; the
// running total after the last span is the final state.
// ---------------------------------------------------------------------------
static __global__ void __launch_bounds__(128)
span_scan_kernel(float* __restrict__ states, float* __restrict__ scratch, int heads, int n_spans,
                 int elems4, int accumulate) {
  // the output pass may be launched now; it waits for this grid before it
  // reads the prefixes. This grid waits for the span pass likewise.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // heads along x (up to 2^31 - 1 of them), element blocks along y (a few
  // hundred at most)
  const int head = blockIdx.x;
  const int e = blockIdx.y * blockDim.x + threadIdx.x;
  if (e >= elems4 || head >= heads) return;
  float4* st = reinterpret_cast<float4*>(states) + (size_t)head * elems4;
  float4* sc = reinterpret_cast<float4*>(scratch) + (size_t)head * n_spans * elems4;
  float4 run = accumulate ? st[e] : make_float4(0.f, 0.f, 0.f, 0.f);
  // spans in groups of 16: all loads of a group are issued before its stores,
  // so the memory latency is paid once per group rather than once per span
  constexpr int G = 16;
  for (int s0 = 0; s0 < n_spans; s0 += G) {
    float4 x[G];
#pragma unroll
    for (int u = 0; u < G; ++u)
      if (s0 + u < n_spans) x[u] = sc[(size_t)(s0 + u) * elems4 + e];
#pragma unroll
    for (int u = 0; u < G; ++u)
      if (s0 + u < n_spans) {
        sc[(size_t)(s0 + u) * elems4 + e] = run;
        run.x += x[u].x; run.y += x[u].y; run.z += x[u].z; run.w += x[u].w;
      }
  }
  st[e] = run;
}

// Launch the span scan. Its carveout is pinned to the shared-memory maximum,
// like the prefill kernels around it, so that the SMs do not repartition
// L1/shared memory between the three launches of a multi-span prefill.
cudaError_t set_carveout_once(const void* kernel, int carveout);   // tsa_abi.cu: once per device
static inline cudaError_t launch_span_scan(float* states, float* scratch, int heads, int n_spans, int elems4,
                                           int accumulate, cudaStream_t s) {
  cudaError_t ce = set_carveout_once((const void*)span_scan_kernel, (int)cudaSharedmemCarveoutMaxShared);
  if (ce != cudaSuccess) return ce;
  // launched with a programmatic dependency on the span pass before it
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)heads, (elems4 + 127) / 128);
  cfg.blockDim = dim3(128);
  cfg.stream = s;
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, span_scan_kernel, states, scratch, heads, n_spans, elems4, accumulate);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// span_output: outputs of one span (one dv slice), state carried on chip.
// ---------------------------------------------------------------------------
template <typename T, int DK, int NT, int W>
__global__ void __launch_bounds__(256)
span_output_kernel(PrefillParams p) {
  using L = SimtLayout<DK, NT, W>;
  constexpr int C = L::C, TN = L::TN, XS = L::XS;
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  float *S, *z;
  const float* xq = sm + L::oXq;
  const float* xk = sm + L::oXk;
  const float* vs = sm + L::oV;
  float* pt = sm + L::oPT;
  const float* phq = sm + L::oPhQ;

  const int tid = threadIdx.x;
  const int tr = tid >> 4, tc = tid & 15;   // tokens 4tr..4tr+3, columns tc*TN..
  const int span = blockIdx.x % p.n_spans;
  const int slice = (blockIdx.x / p.n_spans) % p.n_slices;
  const int head = blockIdx.x / (p.n_spans * p.n_slices);
  TSA_DCHECK(head < p.heads, dbg::kWorkUnit, head, p.heads);
  const int c0 = slice * W;
  const long long t_begin = (long long)span * p.chunks_per_span * C;
  const long long t_end = min(p.N, t_begin + (long long)p.chunks_per_span * C);
  const size_t st_elems = (size_t)L::DPAD * (p.dv + 1);
  const bool single = (p.n_spans == 1);

  load_feat_table<DK, NT>(reinterpret_cast<uint32_t*>(sm + L::oCode), sm + L::oW, tid);
  if constexpr (L::SG) {
    // in place: the caller's state (one span) or the span's prefix slot
    float* g = single ? p.states + head * st_elems
                      : p.scratch + ((size_t)head * p.n_spans + span) * st_elems;
    if (single && !p.accumulate) zero_block(g, st_elems, tid);
    S = g;
    z = g + (size_t)L::DPAD * p.dv;
  } else if (single) {
    S = sm + L::oS;
    z = sm + L::oZ;
    if (p.accumulate) {
      state_slice_in<L::DROWS, W, L::D, L::DPAD>(S, z, p.states + head * st_elems, p.dv, c0, tid);
    } else {
      for (int e = tid; e < L::DROWS * W; e += 256) S[e] = 0.f;
      for (int e = tid; e < L::DROWS; e += 256) z[e] = 0.f;
    }
  } else {
    S = sm + L::oS;
    z = sm + L::oZ;
    state_slice_in<L::DROWS, W, L::D, L::DPAD>(
        S, z, p.scratch + ((size_t)head * p.n_spans + span) * st_elems, p.dv, c0, tid);
  }

  const T* qg = static_cast<const T*>(p.q) + (size_t)head * p.N * DK;
  const T* kg = static_cast<const T*>(p.k) + (size_t)head * p.N * DK;
  const T* vg = static_cast<const T*>(p.v) + (size_t)head * p.N * p.dv + c0;
  T* og = static_cast<T*>(p.out) + (size_t)head * p.N * p.dv + c0;

  for (long long t0 = t_begin; t0 < t_end; t0 += C) {
    const int valid = (int)min((long long)C, t_end - t0);
    const bool need_update = single || (t0 + C < t_end);
    __syncthreads();
    load_x_rows<T, DK, XS, C>(sm + L::oXq, qg + (size_t)t0 * DK, valid, tid);
    load_x_rows<T, DK, XS, C>(sm + L::oXk, kg + (size_t)t0 * DK, valid, tid);
    load_v_rows<T, W, C>(sm + L::oV, vg + (size_t)t0 * p.dv, p.dv, valid, tid);
    __syncthreads();

    // intra-chunk kernel weights P[i][j] = T_n(q_i.k_j) for j <= i, stored P^T
    {
      float a[4][4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) a[r][c] = 0.f;
#pragma unroll
      for (int e = 0; e < DK; ++e) {
        float qv[4], kv[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) qv[r] = xq[(4 * tr + r) * XS + e];
#pragma unroll
        for (int c = 0; c < 4; ++c) kv[c] = xk[(4 * tc + c) * XS + e];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) a[r][c] = fmaf(qv[r], kv[c], a[r][c]);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float col[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int i = 4 * tr + r, j = 4 * tc + c;
          col[r] = (j <= i) ? taylor_T<NT>(a[r][c]) : 0.f;
        }
        *reinterpret_cast<float4*>(pt + (4 * tc + c) * C + 4 * tr) =
            make_float4(col[0], col[1], col[2], col[3]);
      }
    }
    __syncthreads();

    float acc[4][TN];
    float den[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      den[r] = 0.f;
#pragma unroll
      for (int c = 0; c < TN; ++c) acc[r][c] = 0.f;
    }
    // intra: acc += P [V, 1] over j <= 4tr+3 (P is zero above the diagonal)
    {
      const int jmax = 4 * tr + 4;
      for (int j = 0; j < jmax; ++j) {
        const float4 pp = *reinterpret_cast<const float4*>(pt + j * C + 4 * tr);
        float vv[TN];
        if constexpr (TN == 4) {
          const float4 x = *reinterpret_cast<const float4*>(vs + j * W + tc * 4);
          vv[0] = x.x; vv[1] = x.y; vv[2] = x.z; vv[3] = x.w;
        } else {
          const float2 x = *reinterpret_cast<const float2*>(vs + j * W + tc * 2);
          vv[0] = x.x; vv[1] = x.y;
        }
        const float pr[4] = {pp.x, pp.y, pp.z, pp.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < TN; ++c) acc[r][c] = fmaf(pr[r], vv[c], acc[r][c]);
        if ((j & 15) == tc) {
#pragma unroll
          for (int r = 0; r < 4; ++r) den[r] += pr[r];
        }
      }
    }

    // inter: acc += phi(Q) S_{<c}, tile by tile; then S += phi(K)^T [V, 1]
    for (int tile = 0; tile < L::NTILE; ++tile) {
      const int a0 = tile * L::DT;
      build_phi_tile<DK, NT, W, true>(sm, a0, valid, tid);
      __syncthreads();
      auto readout_row = [&](int a) {
        const float4 qq = *reinterpret_cast<const float4*>(phq + a * C + 4 * tr);
        float ss[TN];
        if constexpr (TN == 4) {
          const float4 x = *reinterpret_cast<const float4*>(S + (a0 + a) * W + tc * 4);
          ss[0] = x.x; ss[1] = x.y; ss[2] = x.z; ss[3] = x.w;
        } else {
          const float2 x = *reinterpret_cast<const float2*>(S + (a0 + a) * W + tc * 2);
          ss[0] = x.x; ss[1] = x.y;
        }
        const float qr[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < TN; ++c) acc[r][c] = fmaf(qr[r], ss[c], acc[r][c]);
      };
      if constexpr (L::SG) {
        // rows from global memory: 16 loads in flight per thread on full
        // tiles; the last tile stops at D, where the global state ends
        const int amax = min(L::DT, L::D - a0);
        if (amax == L::DT && TN == 4) {
          // 16 rows' loads issued before their FMAs
          for (int b = 0; b < L::DT; b += 16) {
            float4 sv[16];
#pragma unroll
            for (int u = 0; u < 16; ++u)
              sv[u] = *reinterpret_cast<const float4*>(S + (a0 + b + u) * W + tc * 4);
#pragma unroll
            for (int u = 0; u < 16; ++u) {
              const float4 qq = *reinterpret_cast<const float4*>(phq + (b + u) * C + 4 * tr);
              const float qr[4] = {qq.x, qq.y, qq.z, qq.w};
              const float ss[4] = {sv[u].x, sv[u].y, sv[u].z, sv[u].w};
#pragma unroll
              for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(qr[r], ss[c], acc[r][c]);
            }
          }
        } else {
          for (int a = 0; a < amax; ++a) readout_row(a);
        }
      } else {
#pragma unroll 8
        for (int a = 0; a < L::DT; ++a) readout_row(a);
      }
#pragma unroll
      for (int h = 0; h < L::DT / 16; ++h) {
        const int a = tc + 16 * h;
        const float4 qq = *reinterpret_cast<const float4*>(phq + a * C + 4 * tr);
        const float zz = (!L::SG || a0 + a < L::D) ? z[a0 + a] : 0.f;
        den[0] = fmaf(qq.x, zz, den[0]); den[1] = fmaf(qq.y, zz, den[1]);
        den[2] = fmaf(qq.z, zz, den[2]); den[3] = fmaf(qq.w, zz, den[3]);
      }
      __syncthreads();
      if (need_update) {
        update_tile<DK, NT, W>(sm, S, z, a0, tid);
        __syncthreads();
      }
    }

    // normaliser: reduce the den partials over the 16 column threads
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) den[r] += __shfl_xor_sync(0xffffffffu, den[r], off);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = 4 * tr + r;
      if (i < valid) {
        const float inv = 1.0f / den[r];
        T* dst = og + (size_t)(t0 + i) * p.dv + tc * TN;
        if constexpr (TN == 4) {
          Elem<T>::store4(dst, make_float4(acc[r][0] * inv, acc[r][1] * inv, acc[r][2] * inv,
                                           acc[r][3] * inv));
        } else {
          Elem<T>::store2(dst, make_float2(acc[r][0] * inv, acc[r][1] * inv));
        }
      }
    }
  }

  if (!L::SG && single) {
    __syncthreads();
    state_slice_out<L::DROWS, W, L::D, L::DPAD>(p.states + head * st_elems, S, z, p.dv, c0,
                                                slice == 0, tid);
  }
}

}  // namespace tsa
