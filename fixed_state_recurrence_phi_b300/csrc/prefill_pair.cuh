// prefill_pair.cuh -- chunked causal prefill of bf16 q, k, v on the tcgen05
// tensor cores, for heads whose fp32 state is too large for one SM's tensor
// memory: a cluster of two CTAs shares each (head, span).
//
// The computation is that of prefill_tc.cuh (Expanding Attention, arXiv
// 2610.20637 abstract: additive states, one rank-one update per token, prefill
// as a scan over chunks; Hacker News thread on the paper: (Q'K)V = Q'(KV) and
// the "+1" normaliser column). For chunk c of C = 128 tokens:
//     O        = P [V_c, 1] + sum_f phi(Q_c)_f [S_f, z_f]        (MMA)
//     S_f     += phi(K_c)_f^T [V_c, 1]                           (MMA)
//     out      = O[:, values] / O[:, den]
// with P = mask_{j<=i}(T_n(Q_c K_c^T)).
//
// Work split of the two CTAs (rank r of the cluster):
//  - the state: the feature blocks (128 rows each) are divided between the
//    CTAs as "tiles"; a tile is a block with a range of the state's columns.
//    Both CTAs' tiles stay in their own TMEM for the whole span, so each MMA
//    runs at the full width N = d_v + 16 (no value-column slicing). With an
//    odd number of blocks the last block is split by columns.
//  - the intra-chunk part: CTA r takes keys [64r, 64r + 64) of the chunk
//    (Q K^T with N = 64, its P tile, P V with K = 64).
//  - each CTA's O is then a partial sum over its tiles and its keys; CTA r
//    finalises rows [64r, 64r + 64): the other CTA sends its partial O rows
//    for them through distributed shared memory (plain remote stores and a
//    remote mbarrier arrive).
// The same kernel runs a single CTA per (head, span) when the state fits
// (cs = 1: all tiles, all keys, no exchange).
//
// Column order of the state tiles, of O and of the value tile: the d_v value
// columns with the 16-column normaliser group inserted at column zc
// ([v_0 .. v_zc) | 1, 0 x 15 | v_zc .. v_dv)), so that a block split at zc
// gives each CTA a contiguous column range. The value tile's column zc is 1.0:
// the normaliser z = sum phi(k) and the denominator come out of the same MMAs.
//
// Warp roles (544 threads):
//   TMEM warps (0-7)    thread = TMEM lane (query row / feature row), half of
//                       the columns by warp / 4: P from the scores, the output
//                       (and the exchange), the bf16 state copies
//   builder warps (8-15) feature tiles phi(Q) (readout: 128 tokens x 64
//                       features) and phi(K) (update: 64 tokens x 128
//                       features) into a ring of 16 KB shared-memory slots
//   issuer warp (16)    TMA loads and MMAs
// Every wait is bounded; a wait that runs out sets the CTA's (and the peer
// CTA's) abort flag, the CTA stops, drains what it has in flight, releases its
// TMEM and records the failure in the library's device error word.
#pragma once
#include <cuda.h>
#include "common.cuh"
#include "tc_ptx.cuh"
#include "feature_build.cuh"
#include "prefill_tc.cuh"

namespace tsa {

constexpr int PR_MAX_TILES = 6;
constexpr int PR_THREADS = 544;
constexpr int PR_BUILDER0 = 256;
constexpr int PR_ISSUER_WARP = 16;
constexpr int PR_MAX_RING = 4;

struct PairTile {
  int blk;      // feature block (rows 128*blk ..)
  int lo;       // first column (in the column order above)
  int w;        // width, a multiple of 16
  int col;      // TMEM column of the tile
  int ro_rows;  // rows the readout reads (the block's valid rows, rounded up to 16)
  int s_off;    // byte offset of its bf16 copy in the copy area
};

struct PairParams {
  void* out;
  float* states;        // [heads][DPAD*(dv+1)]
  const float* scratch; // span prefixes [heads][n_spans][DPAD*(dv+1)] (n_spans > 1)
  int* err;
  long long N;
  int heads, dv, n_spans, chunks_per_span, accumulate;
  int cs;        // CTAs per (head, span): 1 or 2
  int zc;        // column of the normaliser group
  int nm;        // d_v + 16
  int kp;        // keys of the intra-chunk part per CTA (128 / cs)
  int shared_o;  // the scores use O's TMEM columns (no room for both)
  int col_O, col_A;
  int ring, nvbuf, nqk;
  int ntile[2];
  PairTile tile[2][PR_MAX_TILES];
  // shared-memory byte offsets
  int off_q, off_k, off_v, off_p, off_s, off_ring, off_x, off_bar;
  int qsz, vsz;
  unsigned long long wait_ns;
  int dbg_withhold;   // testing only: 1 = rank 0 withholds its first exchange publication
};

// mbarriers (shared memory, 8 bytes each) and their arrival counts.
struct PairBars {
  uint64_t* b;
  __device__ uint64_t* qkfull(int i) const { return b + 0 + i; }   // q, k tiles landed (1 + tx)
  __device__ uint64_t* qkempty(int i) const { return b + 2 + i; }  // builders read them (8)
  __device__ uint64_t* vfull(int i) const { return b + 4 + i; }    // v tile landed (1 + tx)
  __device__ uint64_t* qk() const { return b + 6; }                // scores in TMEM (commit)
  __device__ uint64_t* pready() const { return b + 7; }            // P tile written (8)
  __device__ uint64_t* pvdone() const { return b + 8; }            // P V MMAs done (commit)
  __device__ uint64_t* odone() const { return b + 9; }             // O complete (commit)
  __device__ uint64_t* ofree() const { return b + 10; }            // O read out (8)
  __device__ uint64_t* chunk() const { return b + 11; }            // all MMAs of the chunk (commit)
  __device__ uint64_t* drain() const { return b + 12; }            // all MMAs issued (commit)
  __device__ uint64_t* xfull() const { return b + 13; }            // peer's partial rows arrived (128, remote)
  __device__ uint64_t* xfree() const { return b + 14; }            // peer consumed our partial rows (128, remote)
  __device__ uint64_t* updt(int t) const { return b + 15 + t; }    // tile t's updates done (commit)
  __device__ uint64_t* conv(int t) const { return b + 21 + t; }    // tile t's bf16 copy written (8)
  __device__ uint64_t* rfull(int s) const { return b + 27 + s; }   // ring slot written (8)
  __device__ uint64_t* rempty(int s) const { return b + 31 + s; }  // ring slot's MMAs done (commit)
  __device__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(b + 35); }
  __device__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(b + 35) + 1; }
  __device__ uint64_t* wait_limit() const { return b + 36; }
  __device__ uint32_t* peer_abort() const { return reinterpret_cast<uint32_t*>(b + 37); }   // cluster address
  __device__ void init(const PairParams& p) const {
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(qkfull(i), 1);
      tc::mbar_init(qkempty(i), 8);
      tc::mbar_init(vfull(i), 1);
    }
    tc::mbar_init(qk(), 1);
    tc::mbar_init(pready(), 8);
    tc::mbar_init(pvdone(), 1);
    tc::mbar_init(odone(), 1);
    tc::mbar_init(ofree(), 8);
    tc::mbar_init(chunk(), 1);
    tc::mbar_init(drain(), 1);
    tc::mbar_init(xfull(), 128);
    tc::mbar_init(xfree(), 128);
    for (int t = 0; t < PR_MAX_TILES; ++t) {
      tc::mbar_init(updt(t), 1);
      tc::mbar_init(conv(t), 8);
    }
    for (int s = 0; s < PR_MAX_RING; ++s) {
      tc::mbar_init(rfull(s), 8);
      tc::mbar_init(rempty(s), 1);
    }
    *abort_flag() = 0;
    *wait_limit() = p.wait_ns;
    *peer_abort() = 0;
    tc::mbar_fence_init();
  }
};
constexpr int PR_BAR_BYTES = 38 * 8;

// A bounded wait; on time-out this CTA and its peer give up (abort flags).
__device__ __forceinline__ bool pr_wait(const PairBars& B, uint64_t* bar, uint32_t parity, bool cluster_acq = false) {
  if (cluster_acq ? tc::mbar_try_wait_cluster(bar, parity) : tc::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = tc::global_ns();
  const uint64_t lim = *B.wait_limit();
  while (true) {
    if (cluster_acq ? tc::mbar_try_wait_cluster(bar, parity) : tc::mbar_try_wait(bar, parity)) return true;
    if (*B.abort_flag()) return false;
    if (tc::global_ns() - t0 > lim) {
      *B.abort_flag() = 1;
      const uint32_t pa = *B.peer_abort();
      if (pa) tc::st_cluster_flag(pa, 1u);
      return false;
    }
  }
}
// A warp waits as one.
__device__ __forceinline__ bool pr_wait_warp(const PairBars& B, uint64_t* bar, uint32_t parity,
                                             bool cluster_acq = false) {
  return __all_sync(0xffffffffu, pr_wait(B, bar, parity, cluster_acq));
}

// ---- feature tiles ----------------------------------------------------------
// 32 features (block F, features 32G .. 32G + 31) of one token as 4 groups of
// 8 bf16, stored 128 bytes apart from `dst`.
template <int DK, int NT, int F, int G>
__device__ __forceinline__ void pr_phi32(const uint32_t* xp, float x0, uint8_t* dst) {
  constexpr int A = F * 128 + 32 * G;
  *reinterpret_cast<uint4*>(dst + 0) = feat8p<DK, NT, A + 0>(xp, x0);
  *reinterpret_cast<uint4*>(dst + 128) = feat8p<DK, NT, A + 8>(xp, x0);
  *reinterpret_cast<uint4*>(dst + 256) = feat8p<DK, NT, A + 16>(xp, x0);
  *reinterpret_cast<uint4*>(dst + 384) = feat8p<DK, NT, A + 24>(xp, x0);
}
// Runtime (block f, quarter g) -> instantiation; one call site per kernel.
template <int DK, int NT, int F = 0>
__device__ __forceinline__ void pr_build32(int f, int g, const uint32_t* xp, float x0, uint8_t* dst) {
  if constexpr (F < FeatConst<DK, NT>::NB) {
    if (f == F) {
      switch (g) {
        case 0: pr_phi32<DK, NT, F, 0>(xp, x0, dst); break;
        case 1: pr_phi32<DK, NT, F, 1>(xp, x0, dst); break;
        case 2: pr_phi32<DK, NT, F, 2>(xp, x0, dst); break;
        default: pr_phi32<DK, NT, F, 3>(xp, x0, dst); break;
      }
      return;
    }
    pr_build32<DK, NT, F + 1>(f, g, xp, x0, dst);
  }
}

// A token's d inputs from a [e/8][t][8] bf16 tile, as packed bf16 pairs.
template <int DK>
__device__ __forceinline__ void pr_load_xp(const uint8_t* tile, int t, uint32_t (&xp)[DK / 2]) {
#pragma unroll
  for (int g = 0; g < DK / 8; ++g) {
    const uint4 u = *reinterpret_cast<const uint4*>(tile + g * 2048 + t * 16);
    xp[4 * g] = u.x; xp[4 * g + 1] = u.y; xp[4 * g + 2] = u.z; xp[4 * g + 3] = u.w;
  }
}

// Position in the ring (lock step between issuer and builders).
struct PrRing {
  int s = 0, n = 2;
  uint32_t ph = 0;     // per-slot phase bits of the barrier this side waits on
  uint32_t used = 0;   // builder side: slot holds a tile whose MMAs may still run
};

// Readout uses of a tile: 64-feature halves that hold rows the readout reads.
__host__ __device__ constexpr int pr_ro_halves(int ro_rows) { return (ro_rows + 63) / 64; }

// The column of O that value column vv lands in.
__device__ __forceinline__ int pr_ocol(int vv, int zc) { return vv < zc ? vv : vv + 16; }

// ---------------------------------------------------------------------------
template <int DK, int NT>
__global__ void __launch_bounds__(PR_THREADS, 1)
span_output_pair_kernel(const __grid_constant__ PairParams p, const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using FC = FeatConst<DK, NT>;
  constexpr int D = FC::D, DPAD = round_up(D, 4);
  extern __shared__ __align__(1024) uint8_t smem[];
  const PairBars B{reinterpret_cast<uint64_t*>(smem + p.off_bar)};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = (p.cs == 2) ? (int)tc::cluster_rank() : 0;
  const int unit = blockIdx.x / p.cs;
  const int span = unit % p.n_spans, head = unit / p.n_spans;
  const long long t_begin = (long long)span * p.chunks_per_span * TC_C;
  const long long t_end = min(p.N, t_begin + (long long)p.chunks_per_span * TC_C);
  const int n_chunks = (int)((t_end - t_begin + TC_C - 1) / TC_C);
  const bool single = (p.n_spans == 1);
  TSA_DCHECK(head < p.heads, dbg::kWorkUnit, head, p.heads);
  const int ntile = p.ntile[r];
  const int zc = p.zc, nm = p.nm, dv = p.dv;
  const size_t st_elems = (size_t)DPAD * (dv + 1);
  TSA_TRACE_DECL

  if (warp == 0) tc::tmem_alloc(B.tmem_slot(), 512);
  if (tid == 0) {
    B.init(p);
    if (p.cs == 2) *B.peer_abort() = tc::map_rank(tc::smem_u32((const void*)B.abort_flag()), (uint32_t)(r ^ 1));
  }
  // the normaliser group of every v buffer: column zc = 1.0, the rest 0
  if (tid < 256) {
    for (int vb = 0; vb < p.nvbuf; ++vb)
      for (int e = tid; e < 256; e += 256) {
        const int t = e >> 1, g = e & 1;
        *reinterpret_cast<uint4*>(smem + p.off_v + vb * p.vsz + (zc / 8 + g) * 2048 + t * 16) =
            make_uint4(g == 0 ? 0x3F80u : 0u, 0u, 0u, 0u);
      }
  }
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncthreads();
  if (p.cs == 2) tc::cluster_sync();   // the peer's barriers exist before any remote arrive
  tc::fence_after_sync();
  const uint32_t tm = *B.tmem_slot();

  if (warp == PR_ISSUER_WARP) {
    // ------------------------------ issuer ---------------------------------
    const uint32_t id_qk = tc::idesc_bf16(128, p.kp, false, false);
    const uint32_t id_pv = tc::idesc_bf16(128, nm, false, true);
    const uint32_t aQ = tc::smem_u32(smem + p.off_q), aK = tc::smem_u32(smem + p.off_k);
    const uint32_t aV = tc::smem_u32(smem + p.off_v), aP = tc::smem_u32(smem + p.off_p);
    const uint32_t aS = tc::smem_u32(smem + p.off_s), aR = tc::smem_u32(smem + p.off_ring);
    int qk_req = 0, qk_got = 0, v_req = 0, v_got = 0;
    PrRing ring;
    ring.n = p.ring;
    auto load_qk = [&](int c) {
      const int b = c % p.nqk;
      if (tc::elect_one()) {
        tc::mbar_arrive_expect_tx(B.qkfull(b), (uint32_t)(2 * p.qsz));
        const int t0 = (int)(t_begin + (long long)c * TC_C);
        tc::tma_load_4d(smem + p.off_q + b * p.qsz, &tm_q, B.qkfull(b), 0, t0, 0, head);
        tc::tma_load_4d(smem + p.off_k + b * p.qsz, &tm_k, B.qkfull(b), 0, t0, 0, head);
      }
      __syncwarp();
      ++qk_req;
    };
    auto load_v = [&](int c) {
      const int b = c % p.nvbuf;
      if (tc::elect_one()) {
        tc::mbar_arrive_expect_tx(B.vfull(b), (uint32_t)(TC_C * dv * 2));
        const int t0 = (int)(t_begin + (long long)c * TC_C);
        uint8_t* dst = smem + p.off_v + b * p.vsz;
        tc::tma_load_4d(dst, &tm_v, B.vfull(b), 0, t0, 0, head);
        if (zc < dv) tc::tma_load_4d(dst + (zc / 8 + 2) * 2048, &tm_v, B.vfull(b), 0, t0, zc / 8, head);
      }
      __syncwarp();
      ++v_req;
    };
    auto issue_qk_mma = [&](int c) {
      const int b = c % p.nqk;
      const uint64_t dQ = tc::sdesc(aQ + b * p.qsz, 2048, 128);
      const uint64_t dK = tc::sdesc(aK + b * p.qsz + r * 1024, 2048, 128);   // keys 64r ..
#pragma unroll
      for (int k = 0; k < DK / 16; ++k)
        tc::mma_bf16_elect(tm + p.col_A, dQ + (uint64_t)(k * 256), dK + (uint64_t)(k * 256), id_qk, k > 0 ? 1u : 0u);
      tc::mma_commit_elect(B.qk());
    };
    bool ok = true;
    if (n_chunks > 0) {
      load_qk(0);
      load_v(0);
      ok = pr_wait_warp(B, B.qkfull(0), 0u);
      if (ok) {
        ++qk_got;
        tc::fence_after_sync();
        issue_qk_mma(0);
      }
    }
    for (int c = 0; c < n_chunks && ok; ++c) {
      const bool has_next = c + 1 < n_chunks;
      const bool need_update = single || has_next;
      const int vb = c % p.nvbuf;
      // P of this chunk is written (so Q K^T of this chunk is done)
      TSA_TRACE_EVENT(100, c);
      if (!(ok = pr_wait_warp(B, B.pready(), c & 1u))) break;
      TSA_TRACE_EVENT(101, c);
      tc::fence_after_sync();
      // the next chunk's q, k: its buffer's readers hold their inputs in
      // registers (one buffer: this chunk's builders; two: the previous
      // chunk's), and this chunk's Q K^T is done (P is written)
      if (has_next) {
        if (p.nqk == 1) {
          if (!(ok = pr_wait_warp(B, B.qkempty(0), c & 1u))) break;
        } else if (c >= 1) {
          if (!(ok = pr_wait_warp(B, B.qkempty((c + 1) & 1), ((c - 1) >> 1) & 1u))) break;
        }
        load_qk(c + 1);
      }
      // the next chunk's v into the other buffer (two buffers): chunk c-1 is done
      if (has_next && p.nvbuf == 2) {
        if (c >= 1 && !(ok = pr_wait_warp(B, B.chunk(), (c - 1) & 1u))) break;
        load_v(c + 1);
      }
      // O may be overwritten: the previous chunk's O has been read out
      if (c >= 1 && !p.shared_o && !(ok = pr_wait_warp(B, B.ofree(), (c - 1) & 1u))) break;
      // O = sum over this CTA's tiles of phi(Q_f) [S_f, z_f] (its columns of O)
      bool first = true;
      for (int t = 0; t < ntile && ok; ++t) {
        const PairTile& T = p.tile[r][t];
        if (!(ok = pr_wait_warp(B, B.conv(t), c & 1u))) break;
        TSA_TRACE_EVENT(103, t);
        tc::fence_after_sync();
        const uint32_t id_ro = tc::idesc_bf16(128, T.w, false, true);
        const uint64_t dS = tc::sdesc(aS + (uint32_t)T.s_off, 128, (uint32_t)T.ro_rows * 16);
        for (int h = 0; h < pr_ro_halves(T.ro_rows); ++h) {
          if (!(ok = pr_wait_warp(B, B.rfull(ring.s), (ring.ph >> ring.s) & 1u))) break;
          ring.ph ^= 1u << ring.s;
          tc::fence_after_sync();
          const uint64_t dA = tc::sdesc(aR + (uint32_t)ring.s * 16384u, 128, 1024);
          const int ks = min(64, T.ro_rows - 64 * h) / 16;
          for (int k = 0; k < ks; ++k) {
            tc::mma_bf16_elect(tm + p.col_O + (uint32_t)T.lo, dA + (uint64_t)(k * 16),
                               dS + (uint64_t)(64 * h + 16 * k), id_ro, first ? 0u : 1u);
            first = false;
          }
          tc::mma_commit_elect(B.rempty(ring.s));
          ring.s = (ring.s + 1 == ring.n) ? 0 : ring.s + 1;
        }
      }
      if (!ok) break;
      // O += P [V, 1] over this CTA's keys
      if (!(ok = pr_wait_warp(B, B.vfull(vb), (c / p.nvbuf) & 1u))) break;
      ++v_got;
      tc::fence_after_sync();
      const uint32_t vbase = aV + (uint32_t)(vb * p.vsz);
      {
        const uint64_t dP = tc::sdesc(aP, 128, (uint32_t)p.kp * 16);
        const uint64_t dV = tc::sdesc(vbase + (uint32_t)(r * 64 * 16), 128, 2048);
        for (int k = 0; k < p.kp / 16; ++k)
          tc::mma_bf16_elect(tm + p.col_O, dP + (uint64_t)(k * 16), dV + (uint64_t)(k * 16), id_pv, 1u);
        tc::mma_commit_elect(B.pvdone());
      }
      tc::mma_commit_elect(B.odone());
      TSA_TRACE_EVENT(106, c);
      // separate score columns: the next chunk's Q K^T now
      if (has_next && !p.shared_o) {
        if (!(ok = pr_wait_warp(B, B.qkfull((c + 1) % p.nqk), ((c + 1) / p.nqk) & 1u))) break;
        ++qk_got;
        tc::fence_after_sync();
        issue_qk_mma(c + 1);
      }
      // S_f += phi(K_f)^T [V, 1] (the tile's columns), 64 tokens per ring slot
      if (need_update) {
        for (int t = 0; t < ntile && ok; ++t) {
          const PairTile& T = p.tile[r][t];
          const uint32_t id_up = tc::idesc_bf16(128, T.w, true, true);
          const uint64_t dV = tc::sdesc(vbase + (uint32_t)((T.lo / 8) * 2048), 128, 2048);
          for (int h = 0; h < 2; ++h) {
            if (!(ok = pr_wait_warp(B, B.rfull(ring.s), (ring.ph >> ring.s) & 1u))) break;
            ring.ph ^= 1u << ring.s;
            tc::fence_after_sync();
            const uint64_t dA = tc::sdesc(aR + (uint32_t)ring.s * 16384u, 2048, 128);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc::mma_bf16_elect(tm + (uint32_t)T.col, dA + (uint64_t)(k * 256), dV + (uint64_t)(64 * h + 16 * k),
                                 id_up, 1u);
            tc::mma_commit_elect(B.rempty(ring.s));
            ring.s = (ring.s + 1 == ring.n) ? 0 : ring.s + 1;
          }
          if (!ok) break;
          tc::mma_commit_elect(B.updt(t));
        }
        if (!ok) break;
      }
      tc::mma_commit_elect(B.chunk());
      TSA_TRACE_EVENT(109, c);
      if (has_next && p.shared_o) {
        // shared columns: the scores go where O is, after O has been read out
        if (p.shared_o && !(ok = pr_wait_warp(B, B.ofree(), c & 1u))) break;
        if (!(ok = pr_wait_warp(B, B.qkfull((c + 1) % p.nqk), ((c + 1) / p.nqk) & 1u))) break;
        ++qk_got;
        tc::fence_after_sync();
        issue_qk_mma(c + 1);
      }
      if (has_next && p.nvbuf == 1) {
        // one v buffer: the next chunk's v once this chunk's MMAs are done
        if (!(ok = pr_wait_warp(B, B.chunk(), c & 1u))) break;
        load_v(c + 1);
      }
    }
    // drain: every MMA issued, every load requested
    tc::mma_commit_elect(B.drain());
    tc::mbar_wait(B.drain(), 0, TC_WAIT_NS);
    for (; qk_got < qk_req; ++qk_got)
      tc::mbar_wait(B.qkfull(qk_got % p.nqk), (qk_got / p.nqk) & 1u, TC_WAIT_NS);
    for (; v_got < v_req; ++v_got)
      tc::mbar_wait(B.vfull(v_got % p.nvbuf), (v_got / p.nvbuf) & 1u, TC_WAIT_NS);
  } else if (tid < PR_BUILDER0) {
    // ---------------------------- TMEM warps -------------------------------
    const int wq = warp & 3, half = warp >> 2;
    const int i = wq * 32 + lane;                 // TMEM lane: query row / feature row
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int row_hi = wq * 32 + 31;
    const bool own_rows = (p.cs == 1) || ((i >> 6) == r);   // warp-uniform
    __nv_bfloat16* og = static_cast<__nv_bfloat16*>(p.out) + (size_t)head * p.N * dv;
    const float* st_src = nullptr;
    if (!single) st_src = p.scratch + ((size_t)head * p.n_spans + span) * st_elems;
    else if (p.accumulate) st_src = p.states + (size_t)head * st_elems;
    // TMEM tile t -> its bf16 copy: element (a, col) at (col/8)*ro_rows*16 + a*16 + (col%8)*2
    auto convert = [&](int t) {
      const PairTile& T = p.tile[r][t];
      uint8_t* d = smem + p.off_s + T.s_off + i * 16;
      const int rs = T.ro_rows * 16;
      for (int g = half; g < T.w / 16; g += 2) {
        uint32_t rr[16];
        tc::tmem_ld16(tm + lane_off + (uint32_t)(T.col + g * 16), rr);
        tc::tmem_wait_ld();
        if (i < T.ro_rows) {
          float v[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(rr[e]);
          *reinterpret_cast<uint4*>(d + (2 * g) * rs) = tc_pack8(v);
          *reinterpret_cast<uint4*>(d + (2 * g + 1) * rs) = tc_pack8(v + 8);
        }
      }
    };
    // P = mask(T_n(A)) for this CTA's keys -> the P tile (K-major A):
    // (i/8)*(kp*16) + (j/8)*128 + (i%8)*16 + (j%8)*2
    auto compute_p = [&](int c, int valid) -> bool {
      if (!pr_wait_warp(B, B.qk(), c & 1u)) return false;
      if (c >= 1 && !pr_wait_warp(B, B.pvdone(), (c - 1) & 1u)) return false;   // the P tile is free
      tc::fence_after_sync();
      uint8_t* prow = smem + p.off_p + (i / 8) * (p.kp * 16) + (i % 8) * 16;
      for (int jb = 32 * half; jb < p.kp; jb += 64) {
        const int jg = r * 64 + jb;   // the chunk's key index of this 32-key piece
        if (jg <= row_hi) {           // warp-uniform: 32 keys above the diagonal are zero
          uint32_t rr[32];
          tc::tmem_ld32(tm + lane_off + (uint32_t)(p.col_A + jb), rr);
          tc::tmem_wait_ld();
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            float pv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int j = jg + 8 * g + e;
              pv[e] = (j <= i && i < valid) ? taylor_T<NT>(__uint_as_float(rr[8 * g + e])) : 0.0f;
            }
            *reinterpret_cast<uint4*>(prow + ((jb + 8 * g) / 8) * 128) = tc_pack8(pv);
          }
        } else {
#pragma unroll
          for (int g = 0; g < 4; ++g)
            *reinterpret_cast<uint4*>(prow + ((jb + 8 * g) / 8) * 128) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      tc::fence_proxy_async();
      tc_warp_arrive(B.pready(), lane);
      return true;
    };
    // the exchange area: [col/4][64 rows][4] fp32 (the d_v values, then the
    // denominator in group dv/4)
    const uint32_t x_local = tc::smem_u32(smem + p.off_x);
    const uint32_t x_peer = (p.cs == 2) ? tc::map_rank(x_local, (uint32_t)(r ^ 1)) : 0u;
    const uint32_t xfull_peer = (p.cs == 2) ? tc::map_rank(tc::smem_u32(B.xfull()), (uint32_t)(r ^ 1)) : 0u;
    const uint32_t xfree_peer = (p.cs == 2) ? tc::map_rank(tc::smem_u32(B.xfree()), (uint32_t)(r ^ 1)) : 0u;
    const int vh = dv / 2;                       // value columns of this thread's half
    const int oc0 = pr_ocol(half * vh, zc);      // first O column of them (contiguous)
    const int xrow = i & 63;
    bool ok = true;
    for (int c = 0; c < n_chunks && ok; ++c) {
      const long long t0 = t_begin + (long long)c * TC_C;
      const int valid = (int)min((long long)TC_C, t_end - t0);
      const bool has_next = c + 1 < n_chunks;
      const bool need_update = single || has_next;
      if (c == 0) {
        // the span's initial state (prefix / caller's state / 0) -> TMEM tiles
        tc::grid_dep_wait();
        for (int t = 0; t < ntile; ++t) {
          const PairTile& T = p.tile[r][t];
          const int a = T.blk * 128 + i;
          for (int g = half; g < T.w / 16; g += 2) {
            uint32_t rr[16];
            const int cc0 = T.lo + g * 16;   // first column of this group
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
              float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
              const int cc = cc0 + 4 * e4;
              if (st_src != nullptr && a < D) {
                if (cc < zc || cc >= zc + 16) {
                  const int vcol = cc < zc ? cc : cc - 16;   // the value column
                  if (TSA_DCHECK_STATE((size_t)a * dv + vcol, 4, (size_t)DPAD * dv))
                    x = *reinterpret_cast<const float4*>(st_src + (size_t)a * dv + vcol);
                } else if (cc == zc) {
                  x.x = st_src[(size_t)DPAD * dv + a];
                }
              }
              rr[4 * e4] = __float_as_uint(x.x);
              rr[4 * e4 + 1] = __float_as_uint(x.y);
              rr[4 * e4 + 2] = __float_as_uint(x.z);
              rr[4 * e4 + 3] = __float_as_uint(x.w);
            }
            tc::tmem_st16(tm + lane_off + (uint32_t)(T.col + g * 16), rr);
          }
        }
        tc::tmem_wait_st();
        tc::fence_after_sync();
        for (int t = 0; t < ntile; ++t) convert(t);
        tc::fence_proxy_async();
        for (int t = 0; t < ntile; ++t) tc_warp_arrive(B.conv(t), lane);
        if (!(ok = compute_p(0, valid))) break;
      } else if (p.shared_o) {
        if (!(ok = compute_p(c, valid))) break;
      }
      // ---- the output of chunk c
      TSA_TRACE_EVENT(201, c);
      if (!(ok = pr_wait_warp(B, B.odone(), c & 1u))) break;
      TSA_TRACE_EVENT(202, c);
      tc::fence_after_sync();
      if (p.cs == 1 || own_rows) {
        float inv;
        {
          uint32_t rd[16];
          tc::tmem_ld16(tm + lane_off + (uint32_t)(p.col_O + zc), rd);
          tc::tmem_wait_ld();
          float den = __uint_as_float(rd[0]);
          if (p.cs == 2) {
            if (!(ok = pr_wait_warp(B, B.xfull(), c & 1u, true))) break;
            den += reinterpret_cast<const float4*>(smem + p.off_x)[(dv / 4) * 64 + xrow].x;
          }
          inv = 1.0f / den;
        }
        for (int e0 = 0; e0 < vh; e0 += 16) {
          uint32_t rr[16];
          tc::tmem_ld16(tm + lane_off + (uint32_t)(p.col_O + oc0 + e0), rr);
          tc::tmem_wait_ld();
          float v[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(rr[e]);
          if (p.cs == 2) {
            const float4* xs = reinterpret_cast<const float4*>(smem + p.off_x);
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
              const float4 y = xs[((half * vh + e0) / 4 + e4) * 64 + xrow];
              v[4 * e4] += y.x; v[4 * e4 + 1] += y.y; v[4 * e4 + 2] += y.z; v[4 * e4 + 3] += y.w;
            }
          }
          if (i < valid) {
            __nv_bfloat16* dst = og + (size_t)(t0 + i) * dv + half * vh + e0;
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] *= inv;
            *reinterpret_cast<uint4*>(dst) = tc_pack8(v);
            *reinterpret_cast<uint4*>(dst + 8) = tc_pack8(v + 8);
          }
        }
        if (p.cs == 2) tc::mbar_arrive_cluster(xfree_peer);   // our exchange area may be refilled
      } else {
        // the peer's rows: our partial sums go to its exchange area
        if (c >= 1 && !(ok = pr_wait_warp(B, B.xfree(), (c - 1) & 1u, true))) break;
        for (int e0 = 0; e0 < vh; e0 += 16) {
          uint32_t rr[16];
          tc::tmem_ld16(tm + lane_off + (uint32_t)(p.col_O + oc0 + e0), rr);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4)
            tc::st_cluster_f4(x_peer + (uint32_t)(((half * vh + e0) / 4 + e4) * 64 + xrow) * 16u,
                              make_float4(__uint_as_float(rr[4 * e4]), __uint_as_float(rr[4 * e4 + 1]),
                                          __uint_as_float(rr[4 * e4 + 2]), __uint_as_float(rr[4 * e4 + 3])));
        }
        if (half == 0) {
          uint32_t rd[16];
          tc::tmem_ld16(tm + lane_off + (uint32_t)(p.col_O + zc), rd);
          tc::tmem_wait_ld();
          tc::st_cluster_f4(x_peer + (uint32_t)((dv / 4) * 64 + xrow) * 16u,
                            make_float4(__uint_as_float(rd[0]), 0.f, 0.f, 0.f));
        }
        // (testing only: with dbg_withhold, rank 0 never publishes its first
        // chunk's partial rows, so its peer's wait for them runs out)
        if (!(p.dbg_withhold && c == 0 && r == 0)) tc::mbar_arrive_cluster(xfull_peer);
      }
      tc::fence_before_sync();
      tc_warp_arrive(B.ofree(), lane);
      TSA_TRACE_EVENT(204, c);
      // ---- separate score columns, Q K^T issued early: the next chunk's P now
      if (has_next && !p.shared_o) {
        const int valid1 = (int)min((long long)TC_C, t_end - (t0 + TC_C));
        if (!(ok = compute_p(c + 1, valid1))) break;
      }
      // ---- the state copies for the next chunk's readouts
      if (need_update && has_next) {
        for (int t = 0; t < ntile && ok; ++t) {
          if (!(ok = pr_wait_warp(B, B.updt(t), c & 1u))) break;
          tc::fence_after_sync();
          convert(t);
          tc::fence_proxy_async();
          tc_warp_arrive(B.conv(t), lane);
        }
      }
    }
  } else if (warp < PR_ISSUER_WARP) {
    // --------------------------- builder warps ------------------------------
    // One pass over the chunk's ring uses: the readout tiles of each tile's
    // block (64-feature halves; token t, quarter 2h + qr), then its two update
    // tiles (64 tokens each; token 64h + tq, quarter qq). The three tokens'
    // inputs (packed bf16 pairs) are read once per chunk into registers and the
    // q, k buffer is released at once.
    const int bt = tid - PR_BUILDER0;
    const int t = bt & 127, qr = bt >> 7;
    const int tq = bt & 63, qq = bt >> 6;
    const int ro_row = (t / 8) * 1024 + (t % 8) * 16 + (4 * qr) * 128;
    const int up_row = (tq / 8) * 2048 + (tq % 8) * 16 + (4 * qq) * 128;
    int n_ro = 0;
    for (int tt = 0; tt < ntile; ++tt) n_ro += pr_ro_halves(p.tile[r][tt].ro_rows);
    PrRing ring;
    ring.n = p.ring;
    for (int c = 0; c < n_chunks; ++c) {
      const long long t0 = t_begin + (long long)c * TC_C;
      const int valid = (int)min((long long)TC_C, t_end - t0);
      const bool need_update = single || (c + 1 < n_chunks);
      const int qb = c % p.nqk;
      TSA_TRACE_EVENT(300, c);
      if (!pr_wait_warp(B, B.qkfull(qb), (c / p.nqk) & 1u)) break;
      TSA_TRACE_EVENT(301, c);
      uint32_t xq[DK / 2], xk0[DK / 2], xk1[DK / 2];
      pr_load_xp<DK>(smem + p.off_q + qb * p.qsz, t, xq);
      pr_load_xp<DK>(smem + p.off_k + qb * p.qsz, tq, xk0);
      pr_load_xp<DK>(smem + p.off_k + qb * p.qsz, 64 + tq, xk1);
      tc_warp_arrive(B.qkempty(qb), lane);
      const int nuse = n_ro + (need_update ? 2 * ntile : 0);
      bool ok = true;
      int tt = 0, h = 0;
      for (int u = 0; u < nuse; ++u) {
        const bool upd = u >= n_ro;
        if (u == n_ro) { tt = 0; h = 0; }
        const PairTile& T = p.tile[r][tt];
        if ((ring.used >> ring.s) & 1u) {
          if (!(ok = pr_wait_warp(B, B.rempty(ring.s), (ring.ph >> ring.s) & 1u))) break;
          ring.ph ^= 1u << ring.s;
        }
        TSA_TRACE_EVENT(302, ring.s);
        const int tok = upd ? 64 * h + tq : t;
        if (upd || 64 * h + 32 * qr < T.ro_rows) {
          uint32_t xp[DK / 2];
#pragma unroll
          for (int e = 0; e < DK / 2; ++e) xp[e] = upd ? (h ? xk1[e] : xk0[e]) : xq[e];
          TSA_TRACE_EVENT(304, 0);
          const float x0 = (!upd || tok < valid) ? 1.0f : 0.0f;
          pr_build32<DK, NT>(T.blk, upd ? qq : 2 * h + qr, xp, x0,
                             smem + p.off_ring + ring.s * 16384 + (upd ? up_row : ro_row));
          TSA_TRACE_EVENT(305, 0);
        }
        tc::fence_proxy_async();
        TSA_TRACE_EVENT(306, 0);
        tc_warp_arrive(B.rfull(ring.s), lane);
        TSA_TRACE_EVENT(303, ring.s);
        ring.used |= 1u << ring.s;
        ring.s = (ring.s + 1 == ring.n) ? 0 : ring.s + 1;
        if (++h == (upd ? 2 : pr_ro_halves(T.ro_rows))) { h = 0; ++tt; }
      }
      if (!ok) break;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const bool aborted = *B.abort_flag() != 0;
  // the final state (single span): each CTA stores its tiles
  if (!aborted && single && tid < PR_BUILDER0) {
    const int wq = warp & 3, half = warp >> 2;
    const int i = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    float* dst = p.states + (size_t)head * st_elems;
    for (int t = 0; t < ntile; ++t) {
      const PairTile& T = p.tile[r][t];
      const int a = T.blk * 128 + i;
      for (int g = half; g < T.w / 16; g += 2) {
        uint32_t rr[16];
        tc::tmem_ld16(tm + lane_off + (uint32_t)(T.col + g * 16), rr);
        tc::tmem_wait_ld();
        if (a >= DPAD) continue;
        const int cc0 = T.lo + g * 16;
        if (cc0 == zc) {
          dst[(size_t)DPAD * dv + a] = (a < D) ? __uint_as_float(rr[0]) : 0.0f;
        } else {
          const int v0 = cc0 < zc ? cc0 : cc0 - 16;
          if (!TSA_DCHECK_STATE((size_t)a * dv + v0, 16, (size_t)DPAD * dv)) continue;
          float4* o = reinterpret_cast<float4*>(dst + (size_t)a * dv + v0);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o[e] = (a < D) ? make_float4(__uint_as_float(rr[4 * e]), __uint_as_float(rr[4 * e + 1]),
                                         __uint_as_float(rr[4 * e + 2]), __uint_as_float(rr[4 * e + 3]))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  }
  if (aborted && tid == 0) atomicExch(p.err, 1);
  tc::fence_before_sync();
  __syncthreads();
  // neither CTA of a pair leaves while the other may still write to its
  // shared memory or arrive on its barriers
  if (p.cs == 2) tc::cluster_sync();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tm, 512);
  }
}

}  // namespace tsa
