// prefill_tc.cuh -- chunked causal prefill on the 5th-generation tensor cores
// (tcgen05.mma kind::f16: bf16 operands, fp32 accumulators in TMEM, operand
// tiles fed by TMA), for bf16 q, k, v.
//
// The computation is the one of prefill_simt.cuh (Expanding Attention, arXiv
// 2610.20637 abstract: additive states, one rank-one update per token, prefill
// as a scan over chunks; Hacker News thread on the paper: (Q'K)V = Q'(KV) and the
// "+1" normaliser column). For chunk c of C = 128 tokens and the state S_{<c}:
//     A        = Q_c K_c^T                                   (MMA, M=N=128, K=d)
//     P        = mask_{j<=i}(T_n(A))             -> bf16     (CUDA cores)
//     O        = P [V_c, 1] + phi(Q_c) [S_{<c}, z_{<c}]      (MMA)
//     S_{<c+1} = S_{<c} + phi(K_c)^T [V_c, 1]                (MMA)
//     out      = O[:, :W] / O[:, W]
// The normaliser rides in the MMAs as one extra 16-column group: the value
// tile carries a column of ones after its W value columns, and the state the
// matching column z = sum phi(k). So O[:, W] is the softmax-style denominator.
//
// On chip, per CTA (one head, one span of chunks, one slice of W value
// columns): the fp32 state lives in TMEM as NB blocks of 128 feature rows x
// (W + 16) columns; its bf16 copy (the B operand of the readout) in shared
// memory. The accumulator of A and O shares a further max(128, W + 16)
// columns. The feature tiles phi(Q_c), phi(K_c) are built 128 features at a
// time by the CUDA cores; one tile layout serves phi(Q) as a K-major A operand
// (readout, M = tokens) and phi(K) as an MN-major A operand (update,
// M = features).
//
// Shared-memory tiles (no swizzle; byte offsets of element (row, col)):
//   sQ, sK : [e/8][t][8]              (TMA box; K-major, LBO 2048, SBO 128)
//   sV     : [c/8][t][8]              (TMA box; MN-major B, LBO 128, SBO 2048)
//   sP     : (i/8)*2048 + (j/8)*128 + (i%8)*16 + (j%8)*2   (K-major A)
//   sPQ/sPK: (t/8)*2048 + (a/8)*128 + (t%8)*16 + (a%8)*2   (K-major A / MN-major A)
//   sS_f   : (c/8)*2048 + a*16 + (c%8)*2                   (MN-major B)
// Every wait on an mbarrier is bounded; on time-out the CTA records an error
// word, stops issuing work, and releases its TMEM.
#pragma once
#include <cuda.h>
#include "common.cuh"
#include "tc_ptx.cuh"
#include "feature_build.cuh"

namespace tsa {

constexpr int TC_C = 128;
constexpr int TC_THREADS = 256;
constexpr int TC_MAX_SLICES = 4;
constexpr uint64_t TC_WAIT_NS = 1000000000ull;   // 1 s per wait

struct TcParams {
  void* out;
  float* states;     // [heads][DPAD*(dv+1)]
  float* scratch;    // [heads][n_spans][DPAD*(dv+1)] (n_spans > 1)
  int* err;          // device error word (set on a timed-out wait)
  long long N;
  int heads, dv, n_spans, chunks_per_span, accumulate, n_slices, nmax;
  int slice_c0[TC_MAX_SLICES];
  int slice_w[TC_MAX_SLICES];
};

// Byte offsets of the shared-memory tiles (identical on host and device).
struct TcSmem {
  size_t q, k, v, p, pq, pk, s, sblk, bar, total;
  __host__ __device__ TcSmem(int dk, int nmax, int nb) {
    q = 0;
    k = q + (size_t)128 * dk * 2;
    v = k + (size_t)128 * dk * 2;
    p = v + (size_t)128 * nmax * 2;
    pq = p + 32768;
    pk = pq + 32768;
    s = pk + 32768;
    sblk = (size_t)128 * nmax * 2;
    bar = s + (size_t)nb * sblk;
    total = bar + 64;
  }
};

__device__ __forceinline__ bool tc_any_fail(bool ok) { return __syncthreads_or(ok ? 0 : 1) != 0; }

// The d inputs of token t from a [e/8][t][8] bf16 tile, as fp32.
template <int DK>
__device__ __forceinline__ void tc_load_x(const uint8_t* tile, int t, float (&x)[DK + 1]) {
#pragma unroll
  for (int g = 0; g < DK / 8; ++g) {
    const uint4 u = *reinterpret_cast<const uint4*>(tile + g * 2048 + t * 16);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[8 * g + 2 * e] = __uint_as_float(w[e] << 16);
      x[8 * g + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
  }
}

__device__ __forceinline__ uint4 tc_pack8(const float* v) {
  return make_uint4(tc::pack_bf16x2(v[0], v[1]), tc::pack_bf16x2(v[2], v[3]),
                    tc::pack_bf16x2(v[4], v[5]), tc::pack_bf16x2(v[6], v[7]));
}

// Column ones of the value tile: column W is 1.0 (bf16 0x3F80), W+1..W+15 zero.
__device__ __forceinline__ void tc_write_ones(uint8_t* sV, int W, int tid) {
  for (int e = tid; e < 128 * 2; e += TC_THREADS) {
    const int t = e >> 1, g = e & 1;
    *reinterpret_cast<uint4*>(sV + (W / 8 + g) * 2048 + t * 16) =
        make_uint4(g == 0 ? 0x3F80u : 0u, 0u, 0u, 0u);
  }
}

// Store the TMEM state (NB blocks x nm columns) of this slice to a global state
// block: value columns c0..c0+W, z (if with_z), zero padding rows D..DPAD-1.
template <int D, int DPAD, int NB>
__device__ __forceinline__ void tc_store_state(float* dst, uint32_t tm, uint32_t lane_off, int nm, int W,
                                               int c0, int dv, bool with_z, int wq, int lane, int half) {
  for (int f = 0; f < NB; ++f) {
    const int a = f * 128 + wq * 32 + lane;
    for (int g = half; g < nm / 16; g += 2) {
      uint32_t r[16];
      tc::tmem_ld16(tm + lane_off + f * nm + g * 16, r);
      tc::tmem_wait_ld();
      if (a < DPAD) {
        if (g * 16 < W) {
          float4* o = reinterpret_cast<float4*>(dst + (size_t)a * dv + c0 + g * 16);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o[e] = (a < D) ? make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                                         __uint_as_float(r[4 * e + 2]), __uint_as_float(r[4 * e + 3]))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        } else if (with_z && g * 16 == W) {
          dst[(size_t)DPAD * dv + a] = (a < D) ? __uint_as_float(r[0]) : 0.0f;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// span_state_tc: the state sum of one span (one slice) -> scratch.
// ---------------------------------------------------------------------------
template <int DK, int NT>
__global__ void __launch_bounds__(TC_THREADS, 1)
span_state_tc_kernel(const TcParams p, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v) {
  using FC = FeatConst<DK, NT>;
  constexpr int D = FC::D, NB = FC::NB, DPAD = round_up(D, 4);
  extern __shared__ __align__(1024) uint8_t smem[];
  const TcSmem L(DK, p.nmax, NB);
  uint8_t* sK = smem + L.k;
  uint8_t* sV = smem + L.v;
  uint8_t* sPh[2] = {smem + L.pq, smem + L.pk};
  uint64_t* bar_tma = reinterpret_cast<uint64_t*>(smem + L.bar);
  uint64_t* bar_b = bar_tma + 1;   // [2], one per feature buffer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_tma + 3);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wq = warp & 3, half = warp >> 2;
  const int span = blockIdx.x % p.n_spans;
  const int slice = (blockIdx.x / p.n_spans) % p.n_slices;
  const int head = blockIdx.x / (p.n_spans * p.n_slices);
  const int W = p.slice_w[slice], c0 = p.slice_c0[slice], nm = W + 16;
  const long long t_begin = (long long)span * p.chunks_per_span * TC_C;
  const long long t_end = min(p.N, t_begin + (long long)p.chunks_per_span * TC_C);

  if (warp == 0) tc::tmem_alloc(tmem_slot, 512);
  if (tid == 0) {
    tc::mbar_init(bar_tma, 1); tc::mbar_init(bar_b, 1); tc::mbar_init(bar_b + 1, 1);
    tc::mbar_fence_init();
  }
  tc_write_ones(sV, W, tid);
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = *tmem_slot;
  const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
  const uint32_t id_up = tc::idesc_bf16(128, nm, true, true);
  const uint32_t aV = tc::smem_u32(sV);
  const uint32_t aPh[2] = {tc::smem_u32(sPh[0]), tc::smem_u32(sPh[1])};
  const uint32_t tx_bytes = (uint32_t)(128 * DK * 2 + 128 * W * 2);
  const int t = tid & 127;
  const int prow = (t / 8) * 2048 + (t % 8) * 16;

  uint32_t ph_tma = 0, ph_b[2] = {0, 0};
  bool pend[2] = {false, false};
  bool aborted = false, first = true;
  for (long long t0 = t_begin; t0 < t_end && !aborted; t0 += TC_C) {
    const int valid = (int)min((long long)TC_C, t_end - t0);
    // both feature buffers' MMAs (which read sV) must be done before the next tiles land
    for (int b = 0; b < 2 && !aborted; ++b)
      if (pend[b]) {
        const bool ok = tc::mbar_wait(bar_b + b, ph_b[b], TC_WAIT_NS);
        ph_b[b] ^= 1; pend[b] = false;
        if (tc_any_fail(ok)) aborted = true;
      }
    if (aborted) break;
    if (tid == 0) {
      tc::mbar_arrive_expect_tx(bar_tma, tx_bytes);
      tc::tma_load_4d(sK, &tm_k, bar_tma, 0, (int)t0, 0, head);
      for (int u = 0; u < W / 16; ++u)
        tc::tma_load_4d(sV + u * 4096, &tm_v, bar_tma, 0, (int)t0, (c0 + 16 * u) / 8, head);
    }
    {
      const bool ok = tc::mbar_wait(bar_tma, ph_tma, TC_WAIT_NS);
      ph_tma ^= 1;
      if (tc_any_fail(ok)) { aborted = true; break; }
    }
    float xk[DK + 1];
    tc_load_x<DK>(sK, t, xk);
    xk[DK] = (t < valid) ? 1.0f : 0.0f;
    for (int f = 0; f < NB; ++f) {
      const int b = f & 1;
      if (pend[b]) {
        const bool ok = tc::mbar_wait(bar_b + b, ph_b[b], TC_WAIT_NS);
        ph_b[b] ^= 1; pend[b] = false;
        if (tc_any_fail(ok)) { aborted = true; break; }
      }
      build_phi_half<DK, NT, false>(f, half, xk, xk, nullptr, sPh[b] + prow);
      tc::fence_proxy_async();
      tc::fence_before_sync();
      __syncthreads();
      if (tid == 0) {
        tc::fence_after_sync();
#pragma unroll
        for (int s = 0; s < 8; ++s)
          tc::mma_bf16(tm + f * nm, tc::sdesc(aPh[b] + s * 4096, 2048, 128),
                       tc::sdesc(aV + s * 256, 128, 2048), id_up, (s > 0 || !first) ? 1u : 0u);
        tc::mma_commit(bar_b + b);
      }
      pend[b] = true;
    }
    first = false;
  }
  for (int b = 0; b < 2; ++b)
    if (pend[b]) {
      const bool ok = tc::mbar_wait(bar_b + b, ph_b[b], TC_WAIT_NS);
      ph_b[b] ^= 1; pend[b] = false;
      if (tc_any_fail(ok)) aborted = true;
    }
  tc::fence_after_sync();
  if (!aborted) {
    float* dst = p.scratch + ((size_t)head * p.n_spans + span) * (size_t)DPAD * (p.dv + 1);
    tc_store_state<D, DPAD, NB>(dst, tm, lane_off, nm, W, c0, p.dv, slice == 0, wq, lane, half);
  } else if (tid == 0) {
    atomicExch(p.err, 1);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tm, 512);
  }
}

// ---------------------------------------------------------------------------
// span_output_tc: outputs of one span (one slice), state carried in TMEM.
// ---------------------------------------------------------------------------
template <typename T, int DK, int NT>
__global__ void __launch_bounds__(TC_THREADS, 1)
span_output_tc_kernel(const TcParams p, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using FC = FeatConst<DK, NT>;
  constexpr int D = FC::D, NB = FC::NB, DPAD = round_up(D, 4);
  extern __shared__ __align__(1024) uint8_t smem[];
  const TcSmem L(DK, p.nmax, NB);
  uint8_t* sQ = smem + L.q;
  uint8_t* sK = smem + L.k;
  uint8_t* sV = smem + L.v;
  uint8_t* sP = smem + L.p;
  uint8_t* sPQ = smem + L.pq;
  uint8_t* sPK = smem + L.pk;
  uint8_t* sS = smem + L.s;
  uint64_t* bar_tma = reinterpret_cast<uint64_t*>(smem + L.bar);
  uint64_t* bar_mma = bar_tma + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_tma + 3);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wq = warp & 3, half = warp >> 2;
  const int span = blockIdx.x % p.n_spans;
  const int slice = (blockIdx.x / p.n_spans) % p.n_slices;
  const int head = blockIdx.x / (p.n_spans * p.n_slices);
  const int W = p.slice_w[slice], c0 = p.slice_c0[slice], nm = W + 16;
  const long long t_begin = (long long)span * p.chunks_per_span * TC_C;
  const long long t_end = min(p.N, t_begin + (long long)p.chunks_per_span * TC_C);
  const bool single = (p.n_spans == 1);
  const size_t st_elems = (size_t)DPAD * (p.dv + 1);

  if (warp == 0) tc::tmem_alloc(tmem_slot, 512);
  if (tid == 0) {
    tc::mbar_init(bar_tma, 1); tc::mbar_init(bar_mma, 1);
    tc::mbar_fence_init();
  }
  tc_write_ones(sV, W, tid);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = *tmem_slot;
  const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
  const uint32_t col_O = (uint32_t)(NB * nm);

  // initial state: span prefix (several spans), caller's state (ACCUMULATE) or 0
  {
    const float* src = nullptr;
    if (!single) src = p.scratch + ((size_t)head * p.n_spans + span) * st_elems;
    else if (p.accumulate) src = p.states + (size_t)head * st_elems;
    for (int f = 0; f < NB; ++f) {
      const int ar = wq * 32 + lane, a = f * 128 + ar;
      for (int g = half; g < nm / 16; g += 2) {
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c = g * 16 + e;
          float x = 0.0f;
          if (src != nullptr && a < D) {
            if (c < W) x = src[(size_t)a * p.dv + c0 + c];
            else if (c == W) x = src[(size_t)DPAD * p.dv + a];
          }
          v[e] = x;
        }
        uint32_t r[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(v[e]);
        tc::tmem_st16(tm + lane_off + f * nm + g * 16, r);
        uint8_t* d = sS + f * L.sblk + ar * 16;
        *reinterpret_cast<uint4*>(d + (2 * g) * 2048) = tc_pack8(v);
        *reinterpret_cast<uint4*>(d + (2 * g + 1) * 2048) = tc_pack8(v + 8);
      }
    }
    tc::tmem_wait_st();
  }
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  const uint32_t id_qk = tc::idesc_bf16(128, 128, false, false);
  const uint32_t id_pv = tc::idesc_bf16(128, nm, false, true);
  const uint32_t id_up = tc::idesc_bf16(128, nm, true, true);
  const uint32_t aQ = tc::smem_u32(sQ), aK = tc::smem_u32(sK), aV = tc::smem_u32(sV);
  const uint32_t aP = tc::smem_u32(sP), aPQ = tc::smem_u32(sPQ), aPK = tc::smem_u32(sPK);
  const uint32_t aS = tc::smem_u32(sS);
  const uint32_t tx_bytes = (uint32_t)(2 * 128 * DK * 2 + 128 * W * 2);
  T* og = static_cast<T*>(p.out) + (size_t)head * p.N * p.dv + c0;
  const int t = tid & 127;
  const int prow = (t / 8) * 2048 + (t % 8) * 16;
  const int i = wq * 32 + lane;   // TMEM lane = query row / feature row

  uint32_t ph_tma = 0, ph_mma = 0;
  bool aborted = false;
  for (long long t0 = t_begin; t0 < t_end && !aborted; t0 += TC_C) {
    const int valid = (int)min((long long)TC_C, t_end - t0);
    const bool need_update = single || (t0 + TC_C < t_end);
    if (tid == 0) {
      tc::mbar_arrive_expect_tx(bar_tma, tx_bytes);
      tc::tma_load_4d(sQ, &tm_q, bar_tma, 0, (int)t0, 0, head);
      tc::tma_load_4d(sK, &tm_k, bar_tma, 0, (int)t0, 0, head);
      for (int u = 0; u < W / 16; ++u)
        tc::tma_load_4d(sV + u * 4096, &tm_v, bar_tma, 0, (int)t0, (c0 + 16 * u) / 8, head);
    }
    {
      const bool ok = tc::mbar_wait(bar_tma, ph_tma, TC_WAIT_NS);
      ph_tma ^= 1;
      if (tc_any_fail(ok)) { aborted = true; break; }
    }
    // A = Q K^T
    if (tid == 0) {
      tc::fence_after_sync();
#pragma unroll
      for (int s = 0; s < DK / 16; ++s)
        tc::mma_bf16(tm + col_O, tc::sdesc(aQ + s * 4096, 2048, 128), tc::sdesc(aK + s * 4096, 2048, 128),
                     id_qk, s > 0 ? 1u : 0u);
      tc::mma_commit(bar_mma);
    }
    {
      const bool ok = tc::mbar_wait(bar_mma, ph_mma, TC_WAIT_NS);
      ph_mma ^= 1;
      if (tc_any_fail(ok)) { aborted = true; break; }
    }
    tc::fence_after_sync();
    // P = mask(T_n(A)) -> bf16 tile
    {
      uint8_t* prow_p = sP + (i / 8) * 2048 + (i % 8) * 16;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int j0 = half * 64 + cc * 16;
        uint32_t r[16];
        tc::tmem_ld16(tm + lane_off + col_O + j0, r);
        tc::tmem_wait_ld();
        float pv[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pv[e] = (j0 + e <= i && i < valid) ? taylor_T<NT>(__uint_as_float(r[e])) : 0.0f;
        *reinterpret_cast<uint4*>(prow_p + (j0 / 8) * 128) = tc_pack8(pv);
        *reinterpret_cast<uint4*>(prow_p + (j0 / 8 + 1) * 128) = tc_pack8(pv + 8);
      }
    }
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    // O = P [V, 1]
    if (tid == 0) {
      tc::fence_after_sync();
#pragma unroll
      for (int s = 0; s < 8; ++s)
        tc::mma_bf16(tm + col_O, tc::sdesc(aP + s * 256, 128, 2048), tc::sdesc(aV + s * 256, 128, 2048), id_pv,
                     s > 0 ? 1u : 0u);
    }
    float xq[DK + 1], xk[DK + 1];
    tc_load_x<DK>(sQ, t, xq);
    tc_load_x<DK>(sK, t, xk);
    xq[DK] = 1.0f;
    xk[DK] = (t < valid) ? 1.0f : 0.0f;
    for (int f = 0; f < NB; ++f) {
      build_phi_half<DK, NT, true>(f, half, xq, xk, sPQ + prow, sPK + prow);
      tc::fence_proxy_async();
      tc::fence_before_sync();
      __syncthreads();
      if (tid == 0) {
        tc::fence_after_sync();
        const uint32_t aSf = aS + (uint32_t)(f * L.sblk);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          tc::mma_bf16(tm + col_O, tc::sdesc(aPQ + s * 256, 128, 2048), tc::sdesc(aSf + s * 256, 128, 2048),
                       id_pv, 1u);
        if (need_update) {
#pragma unroll
          for (int s = 0; s < 8; ++s)
            tc::mma_bf16(tm + f * nm, tc::sdesc(aPK + s * 4096, 2048, 128), tc::sdesc(aV + s * 256, 128, 2048),
                         id_up, 1u);
        }
        tc::mma_commit(bar_mma);
      }
      {
        const bool ok = tc::mbar_wait(bar_mma, ph_mma, TC_WAIT_NS);
        ph_mma ^= 1;
        if (tc_any_fail(ok)) { aborted = true; break; }
      }
      tc::fence_after_sync();
      if (need_update) {
        // S_{<c+1} block f -> bf16 copy for the next chunk's readout
        uint8_t* d = sS + f * L.sblk + i * 16;
        for (int g = half; g < nm / 16; g += 2) {
          uint32_t r[16];
          tc::tmem_ld16(tm + lane_off + f * nm + g * 16, r);
          tc::tmem_wait_ld();
          float v[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]);
          *reinterpret_cast<uint4*>(d + (2 * g) * 2048) = tc_pack8(v);
          *reinterpret_cast<uint4*>(d + (2 * g + 1) * 2048) = tc_pack8(v + 8);
        }
      }
    }
    if (aborted) break;
    // out = O[:, :W] / O[:, W]
    {
      uint32_t r[16];
      tc::tmem_ld16(tm + lane_off + col_O + W, r);
      tc::tmem_wait_ld();
      const float inv = 1.0f / __uint_as_float(r[0]);
      for (int g = half; g < W / 16; g += 2) {
        tc::tmem_ld16(tm + lane_off + col_O + g * 16, r);
        tc::tmem_wait_ld();
        if (i < valid) {
          T* dst = og + (size_t)(t0 + i) * p.dv + g * 16;
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            Elem<T>::store4(dst + e, make_float4(__uint_as_float(r[e]) * inv, __uint_as_float(r[e + 1]) * inv,
                                                 __uint_as_float(r[e + 2]) * inv,
                                                 __uint_as_float(r[e + 3]) * inv));
        }
      }
    }
    tc::fence_before_sync();
    __syncthreads();
  }
  tc::fence_after_sync();
  if (!aborted) {
    if (single)
      tc_store_state<D, DPAD, NB>(p.states + (size_t)head * st_elems, tm, lane_off, nm, W, c0, p.dv,
                                  slice == 0, wq, lane, half);
  } else if (tid == 0) {
    atomicExch(p.err, 1);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tm, 512);
  }
}

}  // namespace tsa
