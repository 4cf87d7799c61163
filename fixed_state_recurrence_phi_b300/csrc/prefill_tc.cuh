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
constexpr int TC_THREADS = 288;   // 8 worker warps + 1 issuer warp
constexpr int TC_WORKERS = 256;
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
// q, k, v tiles are double-buffered (the next chunk's tiles land by TMA while
// the current chunk runs); two 32 KB ring slots hold the feature tiles (and P).
struct TcSmem {
  size_t xt, vt, s, sblk, bar, total;
  __host__ __device__ TcSmem(int dk, int nmax, int nb) {
    xt = (size_t)128 * dk * 2;
    vt = (size_t)128 * nmax * 2;
    s = 4 * xt + 2 * vt + 2 * 32768;
    sblk = vt;
    bar = s + (size_t)nb * sblk;
    total = bar + 128;
  }
  __host__ __device__ size_t q(int b) const { return b * xt; }
  __host__ __device__ size_t k(int b) const { return (2 + b) * xt; }
  __host__ __device__ size_t v(int b) const { return 4 * xt + b * vt; }
  __host__ __device__ size_t ring(int r) const { return 4 * xt + 2 * vt + r * 32768; }
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
  for (int e = tid; e < 128 * 2; e += TC_WORKERS) {
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

// Work unit of a CTA: (head, span, value slice).
struct TcUnit {
  int span, slice, head, W, c0, nm, n_chunks;
  long long t_begin, t_end;
};

__device__ __forceinline__ TcUnit tc_unit(const TcParams& p) {
  TcUnit u;
  u.slice = blockIdx.x % p.n_slices;
  u.span = (blockIdx.x / p.n_slices) % p.n_spans;
  u.head = blockIdx.x / (p.n_spans * p.n_slices);
  u.W = p.slice_w[0];
  u.c0 = 0;
#pragma unroll
  for (int k = 0; k < TC_MAX_SLICES; ++k)
    if (k == u.slice) { u.W = p.slice_w[k]; u.c0 = p.slice_c0[k]; }
  u.nm = u.W + 16;
  u.t_begin = (long long)u.span * p.chunks_per_span * TC_C;
  u.t_end = min(p.N, u.t_begin + (long long)p.chunks_per_span * TC_C);
  u.n_chunks = (int)((u.t_end - u.t_begin + TC_C - 1) / TC_C);
  return u;
}

// mbarriers of a CTA (shared memory, in this order) and their arrival counts:
//   tfull[2]  TMA tiles of buffer b landed      (1 + tx bytes, issuer)
//   tempty[2] workers are done reading buffer b  (8, one per worker warp)
//   sfull[2]  workers wrote ring slot s          (8 per CTA of the cluster)
//   sempty[2] the MMAs reading ring slot s done  (1 per CTA, multicast commit)
//   qk        A = Q K^T is in TMEM               (1, commit)
//   odone     O of the chunk is complete         (1, commit)
//   ofree     workers have read O                (8)
//   conv      workers converted the state blocks (8)
//   chunk     every MMA of the chunk is done     (1, commit)
//   drain     every MMA issued is done           (1, commit)
struct TcBars {
  uint64_t* b;
  __device__ uint64_t* tfull(int i) const { return b + i; }
  __device__ uint64_t* tempty(int i) const { return b + 2 + i; }
  __device__ uint64_t* sfull(int i) const { return b + 4 + i; }
  __device__ uint64_t* sempty(int i) const { return b + 6 + i; }
  __device__ uint64_t* qk() const { return b + 8; }
  __device__ uint64_t* odone() const { return b + 9; }
  __device__ uint64_t* ofree() const { return b + 10; }
  __device__ uint64_t* conv() const { return b + 11; }
  __device__ uint64_t* chunk() const { return b + 12; }
  __device__ uint64_t* drain() const { return b + 13; }
  __device__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(b + 14); }
  __device__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(b + 14) + 1; }
  // sfull collects one arrival per worker warp of every CTA of the cluster,
  // sempty one (multicast) commit per CTA.
  __device__ void init(int ns) const {
    const uint32_t cnt[14] = {1, 1, 8, 8, 8u * ns, 8u * ns, (uint32_t)ns, (uint32_t)ns, 1, 1, 8, 8, 1, 1};
    for (int k = 0; k < 14; ++k) tc::mbar_init(b + k, cnt[k]);
    *abort_flag() = 0;
    tc::mbar_fence_init();
  }
};

// Issue the TMA loads of one chunk (k and v; q too if `tq`) into buffer b.
__device__ __forceinline__ void tc_issue_tiles(const TcSmem& L, uint8_t* smem, uint64_t* bar, int b,
                                               const CUtensorMap* tq, const CUtensorMap* tk,
                                               const CUtensorMap* tv, long long t0, int head, int c0, int W,
                                               int dk) {
  const uint32_t bytes = (uint32_t)((tq ? 2 : 1) * 128 * dk * 2 + 128 * W * 2);
  tc::mbar_arrive_expect_tx(bar, bytes);
  if (tq) tc::tma_load_4d(smem + L.q(b), tq, bar, 0, (int)t0, 0, head);
  tc::tma_load_4d(smem + L.k(b), tk, bar, 0, (int)t0, 0, head);
  for (int u = 0; u < W / 16; ++u)
    tc::tma_load_4d(smem + L.v(b) + u * 4096, tv, bar, 0, (int)t0, (c0 + 16 * u) / 8, head);
}

// A worker warp's side of the two-slot ring. A slot exists in every CTA of
// the cluster and each CTA's workers write their share of it into all of them:
// before writing slot s the warp waits until the MMAs of every CTA that read
// the slot's previous contents are done (sempty counts one multicast commit
// per CTA); after writing it arrives on sfull[s] of every CTA.
template <int NS>
struct TcWorkerRing {
  uint32_t eph = 0, pend = 0;
  uint32_t sfull_c[2][NS];   // shared::cluster addresses of sfull[s] in each CTA
  __device__ __forceinline__ void setup(const TcBars& B) {
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
      for (int r = 0; r < NS; ++r) sfull_c[s][r] = tc::mapa(tc::smem_u32(B.sfull(s)), (uint32_t)r);
  }
  __device__ __forceinline__ bool acquire(const TcBars& B, int s) {
    if (!((pend >> s) & 1u)) return true;
    const bool ok = (NS == 1)
        ? tc::mbar_wait_or_abort(B.sempty(s), (eph >> s) & 1u, TC_WAIT_NS, B.abort_flag())
        : tc::mbar_wait_cluster_or_abort(B.sempty(s), (eph >> s) & 1u, TC_WAIT_NS, B.abort_flag());
    eph ^= 1u << s;
    pend &= ~(1u << s);
    return __all_sync(0xffffffffu, ok);   // the whole warp gives up together
  }
  __device__ __forceinline__ void release(const TcBars& B, int s, int lane) {
    if constexpr (NS == 1) tc::fence_proxy_async();
    else tc::fence_proxy_async_cluster();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) {
      if constexpr (NS == 1) {
        tc::mbar_arrive(B.sfull(s));
      } else {
#pragma unroll
        for (int r = 0; r < NS; ++r) tc::mbar_arrive_cluster(s ? sfull_c[1][r] : sfull_c[0][r]);
      }
    }
    pend |= 1u << s;
  }
};

__device__ __forceinline__ void tc_warp_arrive(uint64_t* bar, int lane) {
  tc::fence_before_sync();
  __syncwarp();
  if (lane == 0) tc::mbar_arrive(bar);
}

// The issuer frees ring slot s in every CTA of the cluster once its MMAs are done.
template <int NS>
__device__ __forceinline__ void tc_commit_slot(const TcBars& B, int s) {
  if constexpr (NS == 1) tc::mma_commit(B.sempty(s));
  else tc::mma_commit_multicast(B.sempty(s), (uint16_t)((1u << NS) - 1u));
}

// The issuer's last act: wait (bounded) until every MMA it issued and every
// TMA load it requested has completed, so that the tensor memory can be freed.
__device__ __forceinline__ void tc_issuer_drain(const TcBars& B, int filled, int consumed) {
  tc::mma_commit(B.drain());
  tc::mbar_wait(B.drain(), 0, TC_WAIT_NS);
  for (; consumed < filled; ++consumed) tc::mbar_wait(B.tfull(consumed & 1), (consumed >> 1) & 1u, TC_WAIT_NS);
}

// ---------------------------------------------------------------------------
// span_state_tc: the state sum of one span (one slice) -> scratch.
// Workers build phi(K) blocks into the ring; the issuer runs the update MMAs.
// ---------------------------------------------------------------------------
template <int DK, int NT, int NS>
__global__ void __launch_bounds__(TC_THREADS, 1)
span_state_tc_kernel(const TcParams p, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v) {
  using FC = FeatConst<DK, NT>;
  constexpr int D = FC::D, NB = FC::NB, DPAD = round_up(D, 4);
  extern __shared__ __align__(1024) uint8_t smem[];
  const TcSmem L(DK, p.nmax, NB);
  const TcBars B{reinterpret_cast<uint64_t*>(smem + L.bar)};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wq = warp & 3, half = (warp >> 2) & 1;
  const TcUnit u = tc_unit(p);
  const int nm = u.nm;

  if (warp == 0) tc::tmem_alloc(B.tmem_slot(), 512);
  if (tid == 0) B.init(NS);
  if (tid < TC_WORKERS) {
    tc_write_ones(smem + L.v(0), u.W, tid);
    tc_write_ones(smem + L.v(1), u.W, tid);
  }
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncthreads();
  if constexpr (NS > 1) tc::cluster_sync();   // every peer's barriers exist before any remote arrival
  tc::fence_after_sync();
  const uint32_t tm = *B.tmem_slot();
  const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
  volatile int* abort_flag = B.abort_flag();
  const int rank = (NS > 1) ? (int)tc::cluster_rank() : 0;

  if (warp == 8) {
    if (lane == 0) {
      const uint32_t id_up = tc::idesc_bf16(128, nm, true, true);
      const uint32_t aRing0 = tc::smem_u32(smem + L.ring(0));
      uint32_t fph = 0;
      int r = 0, filled = 0, consumed = 0;
      if (u.n_chunks > 0) {
        tc_issue_tiles(L, smem, B.tfull(0), 0, nullptr, &tm_k, &tm_v, u.t_begin, u.head, u.c0, u.W, DK);
        filled = 1;
      }
      for (int c = 0; c < u.n_chunks; ++c) {
        const int buf = c & 1;
        if (!tc::mbar_wait_or_abort(B.tfull(buf), (c >> 1) & 1u, TC_WAIT_NS, abort_flag)) break;
        ++consumed;
        if (c > 0 && !tc::mbar_wait_or_abort(B.chunk(), (c - 1) & 1u, TC_WAIT_NS, abort_flag)) break;
        if (c + 1 < u.n_chunks) {
          if (c + 1 >= 2 &&
              !tc::mbar_wait_or_abort(B.tempty(buf ^ 1), ((c - 1) >> 1) & 1u, TC_WAIT_NS, abort_flag))
            break;
          tc_issue_tiles(L, smem, B.tfull(buf ^ 1), buf ^ 1, nullptr, &tm_k, &tm_v, u.t_begin + (c + 1) * TC_C,
                         u.head, u.c0, u.W, DK);
          ++filled;
        }
        const uint32_t aV = tc::smem_u32(smem + L.v(buf));
        bool ok = true;
        for (int f = 0; f < NB; ++f, ++r) {
          const int s = r & 1;
          ok = (NS == 1) ? tc::mbar_wait_or_abort(B.sfull(s), (fph >> s) & 1u, TC_WAIT_NS, abort_flag)
                         : tc::mbar_wait_cluster_or_abort(B.sfull(s), (fph >> s) & 1u, TC_WAIT_NS, abort_flag);
          fph ^= 1u << s;
          if (!ok) break;
          tc::fence_after_sync();
          const uint32_t aA = aRing0 + (uint32_t)s * 32768u;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            tc::mma_bf16(tm + f * nm, (tc::sdesc(aA, 2048, 128) + (uint64_t)(k * 256)), (tc::sdesc(aV, 128, 2048) + (uint64_t)(k * 16)),
                         id_up, (k > 0 || c > 0) ? 1u : 0u);
          tc_commit_slot<NS>(B, s);
        }
        if (!ok) break;
        tc::mma_commit(B.chunk());
      }
      tc_issuer_drain(B, filled, consumed);
    }
  } else {
    const int t = tid & 127;
    const int prow = (t / 8) * 2048 + (t % 8) * 16;
    TcWorkerRing<NS> ring;
    ring.setup(B);
    uint32_t rc0[NS];   // ring slot 0 of every CTA, shared::cluster addresses
#pragma unroll
    for (int q = 0; q < NS; ++q) rc0[q] = tc::mapa(tc::smem_u32(smem + L.ring(0)), (uint32_t)q);
    int r = 0;
    for (int c = 0; c < u.n_chunks; ++c) {
      const long long t0 = u.t_begin + (long long)c * TC_C;
      const int buf = c & 1;
      const int valid = (int)min((long long)TC_C, u.t_end - t0);
      if (!__all_sync(0xffffffffu, tc::mbar_wait_or_abort(B.tfull(buf), (c >> 1) & 1u, TC_WAIT_NS, abort_flag)))
        break;
      float xk[DK + 1];
      tc_load_x<DK>(smem + L.k(buf), t, xk);
      xk[DK] = (t < valid) ? 1.0f : 0.0f;
      tc_warp_arrive(B.tempty(buf), lane);
      bool ok = true;
      for (int f = 0; f < NB; ++f, ++r) {
        const int s = r & 1;
        if (!(ok = ring.acquire(B, s))) break;
        uint32_t rem[NS];
#pragma unroll
        for (int q = 0; q < NS; ++q) rem[q] = rc0[q] + (uint32_t)s * 32768u + (uint32_t)prow;
        build_phi_rank<DK, NT, NS>(rank, f, half, xk, smem + L.ring(s) + prow, rem);
        ring.release(B, s, lane);
      }
      if (!ok) break;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const bool aborted = *abort_flag != 0;
  if (!aborted && tid < TC_WORKERS) {
    float* dst = p.scratch + ((size_t)u.head * p.n_spans + u.span) * (size_t)DPAD * (p.dv + 1);
    tc_store_state<D, DPAD, NB>(dst, tm, lane_off, nm, u.W, u.c0, p.dv, u.slice == 0, wq, lane, half);
  }
  if (aborted && tid == 0) atomicExch(p.err, 1);
  tc::fence_before_sync();
  __syncthreads();
  if constexpr (NS > 1) tc::cluster_sync();   // no peer still writes into this CTA
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tm, 512);
  }
}

// ---------------------------------------------------------------------------
// span_output_tc: outputs of one span (one slice), state carried in TMEM.
// Per chunk the issuer runs Q K^T, then P [V,1] (P from ring slot), the NB
// readout MMAs phi(Q_f) [S_f, z_f] (O complete -> odone), and the NB update
// MMAs phi(K_f)^T [V,1] into the TMEM state; the workers turn A into P, build
// phi(Q_f) then phi(K_f) into the ring one block ahead of the MMAs, write the
// output once O is complete, and convert each updated state block to its bf16
// copy for the next chunk's readout. The next chunk's tiles land meanwhile.
// ---------------------------------------------------------------------------
template <typename T, int DK, int NT, int NS>
__global__ void __launch_bounds__(TC_THREADS, 1)
span_output_tc_kernel(const TcParams p, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using FC = FeatConst<DK, NT>;
  constexpr int D = FC::D, NB = FC::NB, DPAD = round_up(D, 4);
  extern __shared__ __align__(1024) uint8_t smem[];
  const TcSmem L(DK, p.nmax, NB);
  const TcBars B{reinterpret_cast<uint64_t*>(smem + L.bar)};
  uint8_t* sS = smem + L.s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wq = warp & 3, half = (warp >> 2) & 1;
  const TcUnit u = tc_unit(p);
  const int W = u.W, nm = u.nm;
  const bool single = (p.n_spans == 1);
  const size_t st_elems = (size_t)DPAD * (p.dv + 1);

  if (warp == 0) tc::tmem_alloc(B.tmem_slot(), 512);
  if (tid == 0) B.init(NS);
  if (tid < TC_WORKERS) {
    tc_write_ones(smem + L.v(0), W, tid);
    tc_write_ones(smem + L.v(1), W, tid);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = *B.tmem_slot();
  const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
  const uint32_t col_O = (uint32_t)(NB * nm);
  const int i = wq * 32 + lane;   // TMEM lane = query row / feature row of a block
  volatile int* abort_flag = B.abort_flag();

  // initial state: span prefix (several spans), caller's state (ACCUMULATE) or 0
  if (tid < TC_WORKERS) {
    const float* src = nullptr;
    if (!single) src = p.scratch + ((size_t)u.head * p.n_spans + u.span) * st_elems;
    else if (p.accumulate) src = p.states + (size_t)u.head * st_elems;
    for (int f = 0; f < NB; ++f) {
      const int a = f * 128 + i;
      for (int g = half; g < nm / 16; g += 2) {
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c = g * 16 + e;
          float x = 0.0f;
          if (src != nullptr && a < D) {
            if (c < W) x = src[(size_t)a * p.dv + u.c0 + c];
            else if (c == W) x = src[(size_t)DPAD * p.dv + a];
          }
          v[e] = x;
        }
        uint32_t r[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(v[e]);
        tc::tmem_st16(tm + lane_off + f * nm + g * 16, r);
        uint8_t* d = sS + f * L.sblk + i * 16;
        *reinterpret_cast<uint4*>(d + (2 * g) * 2048) = tc_pack8(v);
        *reinterpret_cast<uint4*>(d + (2 * g + 1) * 2048) = tc_pack8(v + 8);
      }
    }
    tc::tmem_wait_st();
  }
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncthreads();
  if constexpr (NS > 1) tc::cluster_sync();   // every peer's barriers exist before any remote arrival
  tc::fence_after_sync();
  const int rank = (NS > 1) ? (int)tc::cluster_rank() : 0;

  if (warp == 8) {
    // ------------------------------ issuer ---------------------------------
    if (lane == 0) {
      const uint32_t id_qk = tc::idesc_bf16(128, 128, false, false);
      const uint32_t id_pv = tc::idesc_bf16(128, nm, false, true);
      const uint32_t id_up = tc::idesc_bf16(128, nm, true, true);
      const uint32_t aRing0 = tc::smem_u32(smem + L.ring(0));
      const uint32_t aS = tc::smem_u32(sS);
      uint32_t fph = 0;
      int r = 0, filled = 0, consumed = 0;
      auto wait = [&](uint64_t* bar, uint32_t par) {
        return tc::mbar_wait_or_abort(bar, par, TC_WAIT_NS, abort_flag);
      };
      auto take_slot = [&](int s) {
        const bool ok = (NS == 1)
            ? tc::mbar_wait_or_abort(B.sfull(s), (fph >> s) & 1u, TC_WAIT_NS, abort_flag)
            : tc::mbar_wait_cluster_or_abort(B.sfull(s), (fph >> s) & 1u, TC_WAIT_NS, abort_flag);
        fph ^= 1u << s;
        tc::fence_after_sync();
        return ok;
      };
      if (u.n_chunks > 0) {
        tc_issue_tiles(L, smem, B.tfull(0), 0, &tm_q, &tm_k, &tm_v, u.t_begin, u.head, u.c0, W, DK);
        filled = 1;
      }
      for (int c = 0; c < u.n_chunks; ++c) {
        const int buf = c & 1;
        const bool need_update = single || (c + 1 < u.n_chunks);
        if (!wait(B.tfull(buf), (c >> 1) & 1u)) break;
        ++consumed;
        if (c > 0 && !wait(B.ofree(), (c - 1) & 1u)) break;
        tc::fence_after_sync();
        const uint32_t aQ = tc::smem_u32(smem + L.q(buf)), aK = tc::smem_u32(smem + L.k(buf));
        const uint32_t aV = tc::smem_u32(smem + L.v(buf));
#pragma unroll
        for (int k = 0; k < DK / 16; ++k)
          tc::mma_bf16(tm + col_O, (tc::sdesc(aQ, 2048, 128) + (uint64_t)(k * 256)), (tc::sdesc(aK, 2048, 128) + (uint64_t)(k * 256)),
                       id_qk, k > 0 ? 1u : 0u);
        tc::mma_commit(B.qk());
        // the previous chunk's MMAs (readers of buffer buf^1) must be done
        if (c > 0 && !wait(B.chunk(), (c - 1) & 1u)) break;
        if (c + 1 < u.n_chunks) {
          if (c + 1 >= 2 && !wait(B.tempty(buf ^ 1), ((c - 1) >> 1) & 1u)) break;
          tc_issue_tiles(L, smem, B.tfull(buf ^ 1), buf ^ 1, &tm_q, &tm_k, &tm_v, u.t_begin + (c + 1) * TC_C,
                         u.head, u.c0, W, DK);
          ++filled;
        }
        // O = P [V, 1]
        {
          const int s = r & 1;
          if (!take_slot(s)) break;
          const uint32_t aA = aRing0 + (uint32_t)s * 32768u;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            tc::mma_bf16(tm + col_O, (tc::sdesc(aA, 128, 2048) + (uint64_t)(k * 16)), (tc::sdesc(aV, 128, 2048) + (uint64_t)(k * 16)),
                         id_pv, k > 0 ? 1u : 0u);
          tc_commit_slot<NS>(B, s);
          ++r;
        }
        if (c > 0 && !wait(B.conv(), (c - 1) & 1u)) break;
        bool ok = true;
        // O += phi(Q_f) [S_f, z_f]
        for (int f = 0; f < NB; ++f, ++r) {
          const int s = r & 1;
          if (!(ok = take_slot(s))) break;
          const uint32_t aA = aRing0 + (uint32_t)s * 32768u;
          const uint32_t aSf = aS + (uint32_t)(f * L.sblk);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            tc::mma_bf16(tm + col_O, (tc::sdesc(aA, 128, 2048) + (uint64_t)(k * 16)), (tc::sdesc(aSf, 128, 2048) + (uint64_t)(k * 16)),
                         id_pv, 1u);
          tc_commit_slot<NS>(B, s);
        }
        if (!ok) break;
        tc::mma_commit(B.odone());
        // S_f += phi(K_f)^T [V, 1]
        if (need_update) {
          for (int f = 0; f < NB; ++f, ++r) {
            const int s = r & 1;
            if (!(ok = take_slot(s))) break;
            const uint32_t aA = aRing0 + (uint32_t)s * 32768u;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              tc::mma_bf16(tm + f * nm, (tc::sdesc(aA, 2048, 128) + (uint64_t)(k * 256)), (tc::sdesc(aV, 128, 2048) + (uint64_t)(k * 16)),
                           id_up, 1u);
            tc_commit_slot<NS>(B, s);
          }
          if (!ok) break;
        }
        tc::mma_commit(B.chunk());
      }
      tc_issuer_drain(B, filled, consumed);
    }
  } else {
    // ------------------------------ workers --------------------------------
    const int t = tid & 127;
    const int prow = (t / 8) * 2048 + (t % 8) * 16;
    const int row_hi = wq * 32 + 31;
    T* og = static_cast<T*>(p.out) + (size_t)u.head * p.N * p.dv + u.c0;
    TcWorkerRing<NS> ring;
    ring.setup(B);
    uint32_t rc0[NS];   // ring slot 0 of every CTA, shared::cluster addresses
#pragma unroll
    for (int q = 0; q < NS; ++q) rc0[q] = tc::mapa(tc::smem_u32(smem + L.ring(0)), (uint32_t)q);
    // key groups of P that this CTA computes (and stores to every CTA)
    const int pg0 = tc_group0(NS, rank), pgm = tc_group_mid(NS, rank), pg1 = tc_group0(NS, rank + 1);
    const int pga = half ? pgm : pg0, pgb = half ? pg1 : pgm;
    int r = 0;
    auto wait = [&](uint64_t* bar, uint32_t par) {
      return __all_sync(0xffffffffu, tc::mbar_wait_or_abort(bar, par, TC_WAIT_NS, abort_flag));
    };
    // S block f (TMEM) -> its bf16 copy, the next chunk's readout operand
    auto convert_block = [&](int f) {
      uint8_t* d = sS + f * L.sblk + i * 16;
      for (int g = half; g < nm / 16; g += 2) {
        uint32_t rr[16];
        tc::tmem_ld16(tm + lane_off + f * nm + g * 16, rr);
        tc::tmem_wait_ld();
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(rr[e]);
        *reinterpret_cast<uint4*>(d + (2 * g) * 2048) = tc_pack8(v);
        *reinterpret_cast<uint4*>(d + (2 * g + 1) * 2048) = tc_pack8(v + 8);
      }
    };
    for (int c = 0; c < u.n_chunks; ++c) {
      const long long t0 = u.t_begin + (long long)c * TC_C;
      const int buf = c & 1;
      const int valid = (int)min((long long)TC_C, u.t_end - t0);
      const bool need_update = single || (c + 1 < u.n_chunks);
      if (!wait(B.tfull(buf), (c >> 1) & 1u)) break;
      float xq[DK + 1], xk[DK + 1];
      tc_load_x<DK>(smem + L.q(buf), t, xq);
      tc_load_x<DK>(smem + L.k(buf), t, xk);
      xq[DK] = 1.0f;
      xk[DK] = (t < valid) ? 1.0f : 0.0f;
      tc_warp_arrive(B.tempty(buf), lane);
      if (!wait(B.qk(), c & 1u)) break;
      tc::fence_after_sync();
      // P = mask(T_n(A)) -> bf16 ring slot: (i/8)*2048 + (j/8)*128 + (i%8)*16
      {
        const int s = r & 1;
        if (!ring.acquire(B, s)) break;
        const uint32_t prow_off = (uint32_t)((i / 8) * 2048 + (i % 8) * 16);
        uint8_t* prow_p = smem + L.ring(s) + prow_off;
        for (int g = pga; g < pgb; ++g) {
          const int j0 = 8 * g;
          uint4 w = make_uint4(0u, 0u, 0u, 0u);
          if (j0 <= row_hi) {   // warp-uniform: groups above the diagonal are zero
            uint32_t rr[8];
            tc::tmem_ld8(tm + lane_off + col_O + j0, rr);
            tc::tmem_wait_ld();
            float pv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              pv[e] = (j0 + e <= i && i < valid) ? taylor_T<NT>(__uint_as_float(rr[e])) : 0.0f;
            w = tc_pack8(pv);
          }
          *reinterpret_cast<uint4*>(prow_p + g * 128) = w;
#pragma unroll
          for (int q = 0; q < NS; ++q)
            if (q != rank) tc::st_cluster_v4(rc0[q] + (uint32_t)s * 32768u + prow_off + g * 128, w);
        }
        ring.release(B, s, lane);
        ++r;
      }
      // feature blocks: phi(Q_0..NB-1) for the readout, then phi(K_0..NB-1)
      bool ok = true;
      const int r_upd = r + NB;
      for (int k = 0; k < 2 * NB; ++k, ++r) {
        const bool upd = (k >= NB);
        const int f = upd ? k - NB : k;
        if (k == NB) {
          // O complete: out = O[:, :W] / O[:, W]
          if (!(ok = wait(B.odone(), c & 1u))) break;
          tc::fence_after_sync();
          uint32_t rr[16];
          tc::tmem_ld16(tm + lane_off + col_O + W, rr);
          tc::tmem_wait_ld();
          const float inv = 1.0f / __uint_as_float(rr[0]);
          for (int g = half; g < W / 16; g += 2) {
            tc::tmem_ld16(tm + lane_off + col_O + g * 16, rr);
            tc::tmem_wait_ld();
            if (i < valid) {
              T* dst = og + (size_t)(t0 + i) * p.dv + g * 16;
#pragma unroll
              for (int e = 0; e < 16; e += 4)
                Elem<T>::store4(dst + e,
                                make_float4(__uint_as_float(rr[e]) * inv, __uint_as_float(rr[e + 1]) * inv,
                                            __uint_as_float(rr[e + 2]) * inv, __uint_as_float(rr[e + 3]) * inv));
            }
          }
          tc_warp_arrive(B.ofree(), lane);
          if (!need_update) break;
        }
        const int s = r & 1;
        if (!(ok = ring.acquire(B, s))) break;
        if (upd && f >= 2) {   // the slot's previous reader was the update of block f-2
          tc::fence_after_sync();
          convert_block(f - 2);
        }
        float x[DK + 1];
#pragma unroll
        for (int e = 0; e <= DK; ++e) x[e] = upd ? xk[e] : xq[e];
        uint32_t rem[NS];
#pragma unroll
        for (int q = 0; q < NS; ++q) rem[q] = rc0[q] + (uint32_t)s * 32768u + (uint32_t)prow;
        build_phi_rank<DK, NT, NS>(rank, f, half, x, smem + L.ring(s) + prow, rem);
        ring.release(B, s, lane);
      }
      if (!ok) break;
      if (need_update) {
        for (int f = (NB >= 2 ? NB - 2 : 0); f < NB; ++f) {
          if (!(ok = ring.acquire(B, (r_upd + f) & 1))) break;
          tc::fence_after_sync();
          convert_block(f);
        }
        if (!ok) break;
      }
      tc::fence_proxy_async();
      tc_warp_arrive(B.conv(), lane);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const bool aborted = *abort_flag != 0;
  if (!aborted && single && tid < TC_WORKERS)
    tc_store_state<D, DPAD, NB>(p.states + (size_t)u.head * st_elems, tm, lane_off, nm, W, u.c0, p.dv,
                                u.slice == 0, wq, lane, half);
  if (aborted && tid == 0) atomicExch(p.err, 1);
  tc::fence_before_sync();
  __syncthreads();
  if constexpr (NS > 1) tc::cluster_sync();   // no peer still writes into this CTA
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tm, 512);
  }
}

}  // namespace tsa
