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
// (W + 16) columns, its bf16 copy (the B operand of the readout) in shared
// memory. A and O share a further max(128, W + 16) TMEM columns. The feature
// tiles phi(Q_c), phi(K_c) are built 128 features at a time by the CUDA cores
// into a ring of 32 KB slots; one tile layout serves phi(Q) as a K-major A
// operand (readout, M = tokens) and phi(K) as an MN-major A operand (update,
// M = features).
//
// Warp roles: 8 worker warps (TMEM lane quarter = warp % 4, column half =
// warp / 4) build P and the feature tiles, write the outputs and convert the
// updated state to bf16; one issuer warp (one lane) issues the TMA loads and
// the MMAs. They hand off through mbarriers only. Per chunk c the issuer runs
//     P [V,1] -> readouts phi(Q_f) [S_f,z_f] -> (O complete) -> update 0 ->
//     Q_{c+1} K_{c+1}^T (as soon as the workers have read O) -> updates 1..
// so that A of the next chunk is ready when the workers finish the chunk.
//
// Shared-memory tiles (no swizzle; byte offsets of element (row, col)):
//   sQ, sK : [e/8][t][8]              (TMA box; K-major, LBO 2048, SBO 128)
//   sV     : [c/8][t][8]              (TMA box; MN-major B, LBO 128, SBO 2048)
//   P      : (i/8)*2048 + (j/8)*128 + (i%8)*16 + (j%8)*2   (K-major A)
//   phi    : (t/8)*2048 + (a/8)*128 + (t%8)*16 + (a%8)*2   (K-major A / MN-major A)
//   sS_f   : (c/8)*2048 + a*16 + (c%8)*2                   (MN-major B)
// Every wait on an mbarrier is bounded; on time-out the CTA records an error
// word, stops issuing work, waits (bounded) for what it has in flight, and
// releases its TMEM.
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
constexpr int TC_MAX_RING = 3;
constexpr uint64_t TC_WAIT_NS = 1000000000ull;   // 1 s: the default bound of every wait

struct TcParams {
  void* out;
  float* states;     // [heads][DPAD*(dv+1)]
  float* scratch;    // [heads][n_spans][DPAD*(dv+1)] (n_spans > 1)
  int* err;          // device error word (set on a timed-out wait)
  long long N;
  int heads, dv, n_spans, chunks_per_span, accumulate, n_slices, nmax, ring;
  int span_layout;   // fp32 span pass: its own shared-memory layout (Tc32Smem)
  unsigned long long wait_ns;   // bound of each wait between the warp roles
  int dbg_withhold;  // testing only: 1 = the issuer never publishes the first chunk's O
  int slice_c0[TC_MAX_SLICES];
  int slice_w[TC_MAX_SLICES];
};

// Byte offsets of the shared-memory tiles (identical on host and device):
// q and k tiles (single), v tiles (double-buffered: the next chunk's lands by
// TMA while the current one is still read by the update MMAs), `ring` slots of
// 32 KB, the bf16 state copy (NB blocks), then the barriers.
struct TcSmem {
  static constexpr size_t tile = 32768;   // a ring slot: 128 rows of 128 features
  size_t xt, vt, s, sblk, bar, total;
  int ring;
  __host__ __device__ TcSmem(int dk, int nmax, int nb, int ring_slots) {
    ring = ring_slots;
    xt = (size_t)128 * dk * 2;
    vt = (size_t)128 * nmax * 2;
    s = 2 * xt + 2 * vt + (size_t)ring * tile;
    sblk = vt;
    bar = s + (size_t)nb * sblk;
    total = bar + 256;
  }
  __host__ __device__ size_t q() const { return 0; }
  __host__ __device__ size_t k() const { return xt; }
  __host__ __device__ size_t v(int b) const { return 2 * xt + b * vt; }
  __host__ __device__ size_t slot(int r) const { return 2 * xt + 2 * vt + (size_t)r * tile; }
};

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
          if (!TSA_DCHECK_STATE((size_t)a * dv + c0 + g * 16, 16, (size_t)DPAD * dv)) continue;
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
  TSA_DCHECK(u.head < p.heads, dbg::kWorkUnit, u.head, p.heads);
  u.t_begin = (long long)u.span * p.chunks_per_span * TC_C;
  u.t_end = min(p.N, u.t_begin + (long long)p.chunks_per_span * TC_C);
  u.n_chunks = (int)((u.t_end - u.t_begin + TC_C - 1) / TC_C);
  return u;
}

// mbarriers of a CTA (shared memory, in this order) and their arrival counts:
//   qkfull     q, k tiles of the chunk landed          (1 + tx bytes)
//   qkempty    workers have read q, k into registers   (8, one per worker warp)
//   vfull[2]   v tile of buffer b landed               (1 + tx bytes)
//   sfull[3]   workers wrote ring slot s               (8)
//   sempty[3]  the MMAs reading ring slot s are done   (1, tcgen05.commit)
//   qk         A = Q K^T is in TMEM                    (1, commit)
//   odone      O of the chunk is complete              (1, commit)
//   ofree      workers have read O                     (8)
//   conv       workers converted the state blocks      (8)
//   chunk      every MMA of the chunk is done          (1, commit)
//   drain      every MMA issued is done                (1, commit)
struct TcBars {
  uint64_t* b;
  __device__ uint64_t* qkfull() const { return b + 0; }
  __device__ uint64_t* qkempty() const { return b + 1; }
  __device__ uint64_t* vfull(int i) const { return b + 2 + i; }
  __device__ uint64_t* sfull(int i) const { return b + 4 + i; }
  __device__ uint64_t* sempty(int i) const { return b + 7 + i; }
  __device__ uint64_t* qk() const { return b + 10; }
  __device__ uint64_t* odone() const { return b + 11; }
  __device__ uint64_t* ofree() const { return b + 12; }
  __device__ uint64_t* conv() const { return b + 13; }
  __device__ uint64_t* chunk() const { return b + 14; }
  __device__ uint64_t* drain() const { return b + 15; }
  __device__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(b + 16); }
  __device__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(b + 16) + 1; }
  // the bound of each wait (the kernel's wait_ns), set by init
  __device__ uint64_t* wait_limit() const { return b + 24; }
  __device__ void init(uint64_t wait_ns) const {
    const uint32_t cnt[16] = {1, 8, 1, 1, 8, 8, 8, 1, 1, 1, 1, 1, 8, 8, 1, 1};
    for (int k = 0; k < 16; ++k) tc::mbar_init(b + k, cnt[k]);
    *abort_flag() = 0;
    *wait_limit() = wait_ns;
    tc::mbar_fence_init();
  }
};

__device__ __forceinline__ bool tc_wait(const TcBars& B, uint64_t* bar, uint32_t parity) {
  return tc::mbar_wait_or_abort(bar, parity, *B.wait_limit(), B.abort_flag());
}
// A worker warp waits as one: if any lane gives up, the whole warp does.
__device__ __forceinline__ bool tc_wait_warp(const TcBars& B, uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, tc_wait(B, bar, parity));
}
__device__ __forceinline__ void tc_warp_arrive(uint64_t* bar, int lane) {
  tc::fence_before_sync();
  __syncwarp();
  if (lane == 0) tc::mbar_arrive(bar);
}

// TMA loads of the q, k tiles of the chunk at t0 (q too if `tq`).
__device__ __forceinline__ void tc_issue_qk(const TcSmem& L, uint8_t* smem, uint64_t* bar,
                                            const CUtensorMap* tq, const CUtensorMap* tk, long long t0, int head,
                                            int dk) {
  if (!tc::elect_one()) return;
  tc::mbar_arrive_expect_tx(bar, (uint32_t)((tq ? 2 : 1) * 128 * dk * 2));
  if (tq) tc::tma_load_4d(smem + L.q(), tq, bar, 0, (int)t0, 0, head);
  tc::tma_load_4d(smem + L.k(), tk, bar, 0, (int)t0, 0, head);
}
// TMA loads of the W value columns c0.. of the chunk at t0 into buffer b.
__device__ __forceinline__ void tc_issue_v(const TcSmem& L, uint8_t* smem, uint64_t* bar, int b,
                                           const CUtensorMap* tv, long long t0, int head, int c0, int W) {
  if (!tc::elect_one()) return;
  tc::mbar_arrive_expect_tx(bar, (uint32_t)(128 * W * 2));
  for (int u = 0; u < W / 16; ++u)
    tc::tma_load_4d(smem + L.v(b) + u * 4096, tv, bar, 0, (int)t0, (c0 + 16 * u) / 8, head);
}

// Ring position shared (in lock step) by the issuer and the workers: uses go
// to slots 0, 1, .., R-1, 0, ..
struct TcRingPos {
  int s = 0, R = 2;
  __device__ __forceinline__ void next() { s = (s + 1 == R) ? 0 : s + 1; }
};

// A worker warp's side of the ring: before writing slot s it waits for the
// commit of the MMAs that read the slot's previous contents; after writing it
// publishes the slot (one arrival per warp).
struct TcWorkerRing {
  uint32_t eph = 0, pend = 0;
  __device__ __forceinline__ bool acquire(const TcBars& B, int s) {
    if (!((pend >> s) & 1u)) return true;
    const bool ok = tc_wait_warp(B, B.sempty(s), (eph >> s) & 1u);
    eph ^= 1u << s;
    pend &= ~(1u << s);
    return ok;
  }
  __device__ __forceinline__ void release(const TcBars& B, int s, int lane) {
    tc::fence_proxy_async();
    tc_warp_arrive(B.sfull(s), lane);
    pend |= 1u << s;
  }
};

// The issuer's side: wait until every worker warp has written slot s.
struct TcIssuerRing {
  uint32_t fph = 0;
  __device__ __forceinline__ bool take(const TcBars& B, int s) {
    const bool ok = tc_wait_warp(B, B.sfull(s), (fph >> s) & 1u);
    fph ^= 1u << s;
    tc::fence_after_sync();
    return ok;
  }
};

// The issuer's last act: wait (bounded) until every MMA it issued and every
// TMA load it requested has completed, so that the tensor memory can be freed.
__device__ __forceinline__ void tc_issuer_drain(const TcBars& B, int qk_req, int qk_got, int v_req, int v_got) {
  tc::mma_commit_elect(B.drain());
  tc::mbar_wait(B.drain(), 0, TC_WAIT_NS);
  for (; qk_got < qk_req; ++qk_got) tc::mbar_wait(B.qkfull(), qk_got & 1u, TC_WAIT_NS);
  for (; v_got < v_req; ++v_got) tc::mbar_wait(B.vfull(v_got & 1), (v_got >> 1) & 1u, TC_WAIT_NS);
}

// ---------------------------------------------------------------------------
// span_state_tc: the state sum of one span (one slice) -> scratch.
// Workers build phi(K) blocks into the ring; the issuer runs the update MMAs
// and keeps the k and v tiles one chunk ahead.
// ---------------------------------------------------------------------------
template <int DK, int NT>
__global__ void __launch_bounds__(TC_THREADS, 1)
span_state_tc_kernel(const TcParams p, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v) {
  using FC = FeatConst<DK, NT>;
  constexpr int D = FC::D, NB = FC::NB, DPAD = round_up(D, 4);
  extern __shared__ __align__(1024) uint8_t smem[];
  const TcSmem L(DK, p.nmax, NB, p.ring);
  const TcBars B{reinterpret_cast<uint64_t*>(smem + L.bar)};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wq = warp & 3, half = (warp >> 2) & 1;
  const TcUnit u = tc_unit(p);
  const int nm = u.nm;

  if (warp == 0) tc::tmem_alloc(B.tmem_slot(), 512);
  if (tid == 0) B.init(p.wait_ns);
  if (tid < TC_WORKERS) {
    tc_write_ones(smem + L.v(0), u.W, tid);
    tc_write_ones(smem + L.v(1), u.W, tid);
  }
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = *B.tmem_slot();
  const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
  TcRingPos pos;
  pos.R = p.ring;

  if (warp == 8) {
    {   // the whole issuer warp runs the loop; one elected lane issues
      const uint32_t id_up = tc::idesc_bf16(128, nm, true, true);
      TcIssuerRing ring;
      int qk_req = 0, qk_got = 0, v_req = 0, v_got = 0;
      if (u.n_chunks > 0) {
        tc_issue_qk(L, smem, B.qkfull(), nullptr, &tm_k, u.t_begin, u.head, DK);
        tc_issue_v(L, smem, B.vfull(0), 0, &tm_v, u.t_begin, u.head, u.c0, u.W);
        qk_req = v_req = 1;
      }
      for (int c = 0; c < u.n_chunks; ++c) {
        const int buf = c & 1;
        const long long t0 = u.t_begin + (long long)c * TC_C;
        if (!tc_wait_warp(B, B.qkfull(), c & 1u)) break;
        ++qk_got;
        if (c + 1 < u.n_chunks) {
          if (!tc_wait_warp(B, B.qkempty(), c & 1u)) break;   // workers have the k inputs in registers
          tc_issue_qk(L, smem, B.qkfull(), nullptr, &tm_k, t0 + TC_C, u.head, DK);
          ++qk_req;
        }
        if (c > 0 && !tc_wait_warp(B, B.chunk(), (c - 1) & 1u)) break;   // v buffer buf^1 is free again
        if (c + 1 < u.n_chunks) {
          tc_issue_v(L, smem, B.vfull(buf ^ 1), buf ^ 1, &tm_v, t0 + TC_C, u.head, u.c0, u.W);
          ++v_req;
        }
        if (!tc_wait_warp(B, B.vfull(buf), (c >> 1) & 1u)) break;
        ++v_got;
        const uint64_t dV = tc::sdesc(tc::smem_u32(smem + L.v(buf)), 128, 2048);
        bool ok = true;
        for (int f = 0; f < NB; ++f, pos.next()) {
          if (!(ok = ring.take(B, pos.s))) break;
          const uint64_t dA = tc::sdesc(tc::smem_u32(smem + L.slot(pos.s)), 2048, 128);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            tc::mma_bf16_elect(tm + f * nm, dA + (uint64_t)(k * 256), dV + (uint64_t)(k * 16), id_up,
                         (k > 0 || c > 0) ? 1u : 0u);
          tc::mma_commit_elect(B.sempty(pos.s));
        }
        if (!ok) break;
        tc::mma_commit_elect(B.chunk());
      }
      tc_issuer_drain(B, qk_req, qk_got, v_req, v_got);
    }
  } else {
    const int t = tid & 127;
    const int prow = (t / 8) * 2048 + (t % 8) * 16;
    TcWorkerRing ring;
    for (int c = 0; c < u.n_chunks; ++c) {
      const long long t0 = u.t_begin + (long long)c * TC_C;
      const int valid = (int)min((long long)TC_C, u.t_end - t0);
      if (!tc_wait_warp(B, B.qkfull(), c & 1u)) break;
      float xk[DK + 1];
      tc_load_x<DK>(smem + L.k(), t, xk);
      xk[DK] = (t < valid) ? 1.0f : 0.0f;
      tc_warp_arrive(B.qkempty(), lane);
      bool ok = true;
      for (int f = 0; f < NB; ++f, pos.next()) {
        if (!(ok = ring.acquire(B, pos.s))) break;
        build_phi_half<DK, NT>(f, half, xk, smem + L.slot(pos.s) + prow);
        ring.release(B, pos.s, lane);
      }
      if (!ok) break;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const bool aborted = *B.abort_flag() != 0;
  if (!aborted && tid < TC_WORKERS) {
    float* dst = p.scratch + ((size_t)u.head * p.n_spans + u.span) * (size_t)DPAD * (p.dv + 1);
    tc_store_state<D, DPAD, NB>(dst, tm, lane_off, nm, u.W, u.c0, p.dv, u.slice == 0, wq, lane, half);
  }
  if (aborted && tid == 0) atomicExch(p.err, 1);
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
  const TcSmem L(DK, p.nmax, NB, p.ring);
  const TcBars B{reinterpret_cast<uint64_t*>(smem + L.bar)};
  uint8_t* sS = smem + L.s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wq = warp & 3, half = (warp >> 2) & 1;
  const TcUnit u = tc_unit(p);
  const int W = u.W, nm = u.nm;
  const bool single = (p.n_spans == 1);
  const size_t st_elems = (size_t)DPAD * (p.dv + 1);

  if (warp == 0) tc::tmem_alloc(B.tmem_slot(), 512);
  if (tid == 0) B.init(p.wait_ns);
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

  // the first chunk's q, k, v at once: they land while the state is read
  if (warp == 8 && u.n_chunks > 0) {
    tc_issue_qk(L, smem, B.qkfull(), &tm_q, &tm_k, u.t_begin, u.head, DK);
    tc_issue_v(L, smem, B.vfull(0), 0, &tm_v, u.t_begin, u.head, u.c0, W);
    __syncwarp();
  }
  // initial state: span prefix (several spans), caller's state (ACCUMULATE) or 0;
  // thread = feature row, its half of the column groups, up to three groups'
  // 16-byte loads in flight at once
  if (tid < TC_WORKERS) {
    const float* src = nullptr;
    if (!single) src = p.scratch + ((size_t)u.head * p.n_spans + u.span) * st_elems;
    else if (p.accumulate) src = p.states + (size_t)u.head * st_elems;
    constexpr int GB = 3;
    for (int f = 0; f < NB; ++f) {
      const int a = f * 128 + i;
      const bool have = src != nullptr && a < D;
      for (int g0 = half; g0 < nm / 16; g0 += 2 * GB) {
        float4 x[GB][4];
#pragma unroll
        for (int j = 0; j < GB; ++j) {
          const int g = g0 + 2 * j;
#pragma unroll
          for (int e = 0; e < 4; ++e) x[j][e] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (have && g < nm / 16) {
            if (g * 16 < W) {
              if (TSA_DCHECK_STATE((size_t)a * p.dv + u.c0 + g * 16, 16, (size_t)DPAD * p.dv)) {
                const float4* s4 = reinterpret_cast<const float4*>(src + (size_t)a * p.dv + u.c0 + g * 16);
#pragma unroll
                for (int e = 0; e < 4; ++e) x[j][e] = s4[e];
              }
            } else if (g * 16 == W) {
              x[j][0].x = src[(size_t)DPAD * p.dv + a];
            }
          }
        }
#pragma unroll
        for (int j = 0; j < GB; ++j) {
          const int g = g0 + 2 * j;
          if (g >= nm / 16) break;
          float v[16];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            v[4 * e] = x[j][e].x; v[4 * e + 1] = x[j][e].y; v[4 * e + 2] = x[j][e].z; v[4 * e + 3] = x[j][e].w;
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
    }
    tc::tmem_wait_st();
  }
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  TcRingPos pos;
  pos.R = p.ring;

  if (warp == 8) {
    // ------------------------------ issuer ---------------------------------
    {   // the whole issuer warp runs the loop; one elected lane issues
      const uint32_t id_qk = tc::idesc_bf16(128, 128, false, false);
      const uint32_t id_pv = tc::idesc_bf16(128, nm, false, true);
      const uint32_t id_up = tc::idesc_bf16(128, nm, true, true);
      const uint64_t dQ = tc::sdesc(tc::smem_u32(smem + L.q()), 2048, 128);
      const uint64_t dK = tc::sdesc(tc::smem_u32(smem + L.k()), 2048, 128);
      const uint32_t aS = tc::smem_u32(sS);
      TcIssuerRing ring;
      int qk_req = 0, qk_got = 0, v_req = 0, v_got = 0;
      auto issue_qk_mma = [&]() {
#pragma unroll
        for (int k = 0; k < DK / 16; ++k)
          tc::mma_bf16_elect(tm + col_O, dQ + (uint64_t)(k * 256), dK + (uint64_t)(k * 256), id_qk, k > 0 ? 1u : 0u);
        tc::mma_commit_elect(B.qk());
      };
      bool ok = true;
      if (u.n_chunks > 0) {
        qk_req = v_req = 1;   // issued before the initial state was read
        ok = tc_wait_warp(B, B.qkfull(), 0u);
        if (ok) {
          ++qk_got;
          tc::fence_after_sync();
          issue_qk_mma();   // A of chunk 0
        }
      }
      for (int c = 0; c < u.n_chunks && ok; ++c) {
        const int buf = c & 1;
        const long long t0 = u.t_begin + (long long)c * TC_C;
        const bool need_update = single || (c + 1 < u.n_chunks);
        const bool has_next = (c + 1 < u.n_chunks);
        // q, k tiles of the next chunk: once the workers hold this chunk's in
        // registers and Q K^T of this chunk (the other reader) has completed
        if (has_next) {
          if (!(ok = tc_wait_warp(B, B.qkempty(), c & 1u))) break;
          if (!(ok = tc_wait_warp(B, B.qk(), c & 1u))) break;
          tc_issue_qk(L, smem, B.qkfull(), &tm_q, &tm_k, t0 + TC_C, u.head, DK);
          ++qk_req;
        }
        // v tile of the next chunk into the buffer the previous chunk used
        if (c > 0 && !(ok = tc_wait_warp(B, B.chunk(), (c - 1) & 1u))) break;
        if (has_next) {
          tc_issue_v(L, smem, B.vfull(buf ^ 1), buf ^ 1, &tm_v, t0 + TC_C, u.head, u.c0, W);
          ++v_req;
        }
        if (!(ok = tc_wait_warp(B, B.vfull(buf), (c >> 1) & 1u))) break;
        ++v_got;
        const uint64_t dV = tc::sdesc(tc::smem_u32(smem + L.v(buf)), 128, 2048);
        // O = P [V, 1]
        if (!(ok = ring.take(B, pos.s))) break;
        {
          const uint64_t dP = tc::sdesc(tc::smem_u32(smem + L.slot(pos.s)), 128, 2048);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            tc::mma_bf16_elect(tm + col_O, dP + (uint64_t)(k * 16), dV + (uint64_t)(k * 16), id_pv, k > 0 ? 1u : 0u);
          tc::mma_commit_elect(B.sempty(pos.s));
          pos.next();
        }
        // the bf16 state copy must hold S_{<c} (converted by the workers)
        if (c > 0 && !(ok = tc_wait_warp(B, B.conv(), (c - 1) & 1u))) break;
        // O += phi(Q_f) [S_f, z_f]
        for (int f = 0; f < NB; ++f, pos.next()) {
          if (!(ok = ring.take(B, pos.s))) break;
          const uint64_t dA = tc::sdesc(tc::smem_u32(smem + L.slot(pos.s)), 128, 2048);
          const uint64_t dS = tc::sdesc(aS + (uint32_t)(f * L.sblk), 128, 2048);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            tc::mma_bf16_elect(tm + col_O, dA + (uint64_t)(k * 16), dS + (uint64_t)(k * 16), id_pv, 1u);
          tc::mma_commit_elect(B.sempty(pos.s));
        }
        if (!ok) break;
        tc::mma_commit_elect(B.odone());
        // S_f += phi(K_f)^T [V, 1]; after block 0, the next chunk's Q K^T as
        // soon as the workers have read O (A and O share their TMEM columns)
        for (int f = 0; f < (need_update ? NB : 0); ++f, pos.next()) {
          if (!(ok = ring.take(B, pos.s))) break;
          const uint64_t dA = tc::sdesc(tc::smem_u32(smem + L.slot(pos.s)), 2048, 128);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            tc::mma_bf16_elect(tm + f * nm, dA + (uint64_t)(k * 256), dV + (uint64_t)(k * 16), id_up, 1u);
          tc::mma_commit_elect(B.sempty(pos.s));
          if (f == 0 && has_next) {
            if (!(ok = tc_wait_warp(B, B.ofree(), c & 1u))) break;
            if (!(ok = tc_wait_warp(B, B.qkfull(), (c + 1) & 1u))) break;
            ++qk_got;
            tc::fence_after_sync();
            issue_qk_mma();
          }
        }
        if (!ok) break;
        tc::mma_commit_elect(B.chunk());
      }
      tc_issuer_drain(B, qk_req, qk_got, v_req, v_got);
    }
  } else {
    // ------------------------------ workers --------------------------------
    // feature tiles: token t, half of a block
    const int t = tid & 127;
    const int prow = (t / 8) * 2048 + (t % 8) * 16;
    const int row_hi = wq * 32 + 31;
    T* og = static_cast<T*>(p.out) + (size_t)u.head * p.N * p.dv + u.c0;
    TcWorkerRing ring;
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
      const int valid = (int)min((long long)TC_C, u.t_end - t0);
      const bool need_update = single || (c + 1 < u.n_chunks);
      // the bf16 copy of the updated state is the next chunk's readout operand;
      // after the last chunk nothing reads it (the issuer's drain orders the
      // final state store after the updates)
      const bool need_copy = need_update && (c + 1 < u.n_chunks);
      if (!tc_wait_warp(B, B.qkfull(), c & 1u)) break;
      float xq[DK + 1], xk[DK + 1];
      tc_load_x<DK>(smem + L.q(), t, xq);
      tc_load_x<DK>(smem + L.k(), t, xk);
      xq[DK] = 1.0f;
      xk[DK] = (t < valid) ? 1.0f : 0.0f;
      tc_warp_arrive(B.qkempty(), lane);
      if (!tc_wait_warp(B, B.qk(), c & 1u)) break;
      tc::fence_after_sync();
      // P = mask(T_n(A)) -> bf16 ring slot: (i/8)*2048 + (j/8)*128 + (i%8)*16
      if (!ring.acquire(B, pos.s)) break;
      {
        uint8_t* prow_p = smem + L.slot(pos.s) + (i / 8) * 2048 + (i % 8) * 16;
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          const int jb = half * 64 + 32 * q2;
          if (jb <= row_hi) {   // warp-uniform: 32 keys above the diagonal are zero
            uint32_t rr[32];
            tc::tmem_ld32(tm + lane_off + col_O + jb, rr);
            tc::tmem_wait_ld();
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              float pv[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const int j = jb + 8 * g + e;
                pv[e] = (j <= i && i < valid) ? taylor_T<NT>(__uint_as_float(rr[8 * g + e])) : 0.0f;
              }
              *reinterpret_cast<uint4*>(prow_p + ((jb + 8 * g) / 8) * 128) = tc_pack8(pv);
            }
          } else {
#pragma unroll
            for (int g = 0; g < 4; ++g)
              *reinterpret_cast<uint4*>(prow_p + ((jb + 8 * g) / 8) * 128) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      ring.release(B, pos.s, lane);
      pos.next();
      // Feature uses: phi(Q_0..NB-1) for the readout, then phi(K_0..NB-1) for
      // the update. The output is written once O is complete: after the first
      // update tile (which goes in before O is done), or after the readouts
      // when there is no update. One build call site keeps the code compact.
      const int nuse = NB + (need_update ? NB : 0);
      const int k_out = (NB + 1 < nuse) ? NB + 1 : nuse;
      const int s_upd0 = (pos.s + NB) % pos.R;   // ring slot of update block 0
      bool ok = true;
      for (int k = 0; k <= nuse; ++k) {
        if (k == k_out) {
          // out = O[:, :W] / O[:, W]
          if (!(ok = tc_wait_warp(B, B.odone(), c & 1u))) break;
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
        }
        if (k == nuse) break;
        const bool upd = (k >= NB);
        const int f = upd ? k - NB : k;
        if (!(ok = ring.acquire(B, pos.s))) break;
        if (need_copy && upd && f >= pos.R) {   // the slot last held update f - R: convert that block
          tc::fence_after_sync();
          convert_block(f - pos.R);
        }
        float x[DK + 1];
#pragma unroll
        for (int e = 0; e <= DK; ++e) x[e] = upd ? xk[e] : xq[e];
        build_phi_half<DK, NT>(f, half, x, smem + L.slot(pos.s) + prow);
        ring.release(B, pos.s, lane);
        pos.next();
      }
      if (!ok) break;
      if (need_copy) {
        for (int f = (NB > pos.R ? NB - pos.R : 0); f < NB; ++f) {
          const int s = (s_upd0 + f) % pos.R;
          if (!(ok = ring.acquire(B, s))) break;
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
  const bool aborted = *B.abort_flag() != 0;
  if (!aborted && single && tid < TC_WORKERS)
    tc_store_state<D, DPAD, NB>(p.states + (size_t)u.head * st_elems, tm, lane_off, nm, W, u.c0, p.dv,
                                u.slice == 0, wq, lane, half);
  if (aborted && tid == 0) atomicExch(p.err, 1);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tm, 512);
  }
}

}  // namespace tsa
