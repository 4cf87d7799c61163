// prefill_tc32.cuh -- chunked causal prefill of fp32 q, k, v on the tensor
// cores with split-bf16 operands.
//
// Same computation and chunk recurrence as prefill_tc.cuh (Expanding
// Attention, arXiv 2610.20637 abstract; Hacker News thread on the paper:
// (Q'K)V = Q'(KV) and the "+1" normaliser column), for inputs whose results
// must match to 1e-4. Every operand x is split as x = hi + lo with
// hi = bf16(x) and lo = bf16(x - hi) (16 significant bits together), and every
// product as
//     A B  ~  A_hi B_hi + A_hi B_lo + A_lo B_hi        (three kind::f16 MMAs)
// into the same fp32 TMEM accumulator; the dropped A_lo B_lo term and the
// rounding of lo are ~2^-16 relative.
//
// Per CTA (one head, one span, all value columns plus the normaliser group):
// fp32 q, k, v tiles of a chunk land by TMA in a staging area as
// [col/4][token][4] tiles; they are split into hi/lo bf16 operand tiles (q, k
// for Q K^T; v for P [V,1] and the update). The state lives in TMEM; its
// hi/lo copies in shared memory (only the rows the readout reads: the last
// feature block is cut to a multiple of 16 rows) are the readout's B operand.
//
// The output pass runs three warp roles (span_output_tc32_kernel):
//   TMEM warps (0-7)     operand and state conversions; P = mask(T_n(A))
//                        written into TMEM over the scores (the P [V,1] MMAs
//                        read A from TMEM); the output, staged per warp and
//                        stored by TMA
//   builder warps (8-15) readout feature tiles (128 tokens x 64 features of
//                        a block) into a two-buffer TMEM area (the readout
//                        MMAs read A from TMEM); update feature tiles (64
//                        tokens x 128 features of a block, or the last
//                        block's few rows for all 128 tokens) through a ring
//                        of 32 KB shared-memory slots (hi and lo halves)
//   issuer warp (16)     TMA loads and MMAs
// The span pass (span_state_tc32_kernel) has 8 workers (v conversion, update
// tiles) and the issuer. All hand-offs are mbarriers with bounded waits, as
// in prefill_tc.cuh.
#pragma once
#include <cuda.h>
#include "common.cuh"
#include "tc_ptx.cuh"
#include "feature_build.cuh"
#include "prefill_tc.cuh"

namespace tsa {

template <int DK, int NT>
struct Tc32Shape {
  static constexpr int D = feat_dim(DK, NT);
  static constexpr int NB = (D + 127) / 128;
  // rows of the last block that the readout reads (a multiple of 16)
  static constexpr int LAST_ROWS = round_up(D - 128 * (NB - 1), 16);
  static constexpr int ROWS = 128 * (NB - 1) + LAST_ROWS;
  __host__ __device__ static constexpr int rows(int f) { return f < NB - 1 ? 128 : LAST_ROWS; }
  // 64-feature readout uses of block f
  __host__ __device__ static constexpr int halves(int f) { return (rows(f) + 63) / 64; }
  // The last block's update tile holds all 128 tokens of its few rows (at
  // most 64) in one ring slot: feature group g8 of token t at
  // (t/8)*GL*128 + g8*128 + (t%8)*16 bytes (hi; lo 16 KB further).
  static constexpr int GL = LAST_ROWS / 8;
  static constexpr bool COMPACT = LAST_ROWS <= 64;
  // update tiles of block f: two 64-token tiles, or the one compact tile
  __host__ __device__ static constexpr int upd_tiles(int f) { return (COMPACT && f == NB - 1) ? 1 : 2; }
  __host__ __device__ static constexpr int n_upd() { return 2 * NB - (COMPACT ? 1 : 0); }
};

// Shared memory of the fp32 kernels (byte offsets, host and device).
struct Tc32Smem {
  size_t qs, ks, vs, qh, ql, kh, kl, vh, vl, ring0, sh, sl, bar, total;
  int ring, nm;
  // span_pass: the span pass's own layout, without the q staging, the q/k
  // operand tiles and the state copies; sh and sl then hold its second v
  // tile buffer (hi, lo), and the space saved can take a third ring slot.
  __host__ __device__ Tc32Smem(int dk, int dv, int nm_, int rows, int ring_slots, bool span_pass = false) {
    ring = ring_slots;
    nm = nm_;
    const size_t x32 = (size_t)128 * dk * 4, x16 = (size_t)128 * dk * 2, v16 = (size_t)128 * nm_ * 2;
    if (span_pass) {
      qs = ks = 0;
      vs = ks + x32;
      qh = ql = kh = kl = vs;   // unused
      vh = vs + (size_t)128 * dv * 4;
      vl = vh + v16;
      sh = vl + v16;
      sl = sh + v16;
      ring0 = sl + v16;
      bar = ring0 + (size_t)ring * 32768;
      total = bar + 256;
      return;
    }
    qs = 0;
    ks = qs + x32;
    vs = ks + x32;
    qh = vs + (size_t)128 * dv * 4;
    ql = qh + x16;
    kh = ql + x16;
    kl = kh + x16;
    vh = kl + x16;
    vl = vh + v16;
    ring0 = vl + v16;
    sh = ring0 + (size_t)ring * 32768;
    sl = sh + (size_t)rows * nm_ * 2;
    bar = sl + (size_t)rows * nm_ * 2;
    total = bar + 256;
  }
  __host__ __device__ size_t slot(int r) const { return ring0 + (size_t)r * 32768; }
};

// mbarriers of the fp32 kernels (shared memory) and arrival counts. Slots
// 0-15 are those of prefill_tc.cuh's TcBars (ring sfull[3] / sempty[3], qk,
// odone, conv, chunk, drain keep their meaning); the slots of TcBars that
// these kernels do not use carry their own barriers:
//   0  stg_full   staging tiles (fp32 q, k, v) of the chunk landed   (1 + tx)
//   1  stg_free   the staging is read (workers; output pass: TMEM and
//                 builder warps)                                  (8 or 16)
//   2  tiles      hi/lo q, k operand tiles written                     (8)
//   3  ostored    output stores have read their staging               (8)
//   12 pready     P written into TMEM over the scores A                (8)
//   16 (the TMEM allocation word and the abort flag)
//   17 stload     the span's initial state copied into the ring area (1 + tx)
//   18-19 rofull  readout feature tile r of the TMEM buffers written    (8)
//   20-21 roempty ... and read by its MMAs (the span pass: vfree, its v
//                 tile buffer r free again)                            (1)
//   22 (a flag: the initial-state copy has been issued)
struct Tc32Bars {
  uint64_t* b;
  __device__ uint64_t* stg_full() const { return b + 0; }
  __device__ uint64_t* stg_free() const { return b + 1; }
  __device__ uint64_t* tiles() const { return b + 2; }
  // every worker warp's output store has read its staging piece    (8)
  __device__ uint64_t* ostored() const { return b + 3; }
  // every worker warp wrote its P pieces into TMEM (the ring's ofree slot,
  // which these kernels do not otherwise use)                        (8)
  __device__ uint64_t* pready() const { return b + 12; }
  // the span's initial state copied into the ring area            (1 + tx)
  __device__ uint64_t* stload() const { return b + 17; }
  // set once that copy has been issued (the drain waits for it then)
  __device__ volatile int* copy_issued() const { return reinterpret_cast<volatile int*>(b + 22); }
  // span pass: v tile buffer r free again (its MMAs are done)         (1)
  __device__ uint64_t* vfree(int r) const { return b + 20 + r; }
  // readout feature tile r of the TMEM double buffer written           (8)
  __device__ uint64_t* rofull(int r) const { return b + 18 + r; }
  // ... and read by its MMAs                                          (1)
  __device__ uint64_t* roempty(int r) const { return b + 20 + r; }
  __device__ TcBars ring_bars() const { return TcBars{b}; }
  // stg_users: warps that read the staging (8, or 16 in the output kernel)
  __device__ void init(uint64_t wait_ns, uint32_t stg_users = 8) const {
    const uint32_t cnt[16] = {1, stg_users, 8, 8, 8, 8, 8, 1, 1, 1, 1, 1, 8, 8, 1, 1};
    for (int k = 0; k < 16; ++k) tc::mbar_init(b + k, cnt[k]);
    for (int r = 0; r < 2; ++r) {
      tc::mbar_init(rofull(r), 8);
      tc::mbar_init(roempty(r), 1);
    }
    tc::mbar_init(stload(), 1);
    *copy_issued() = 0;
    *TcBars{b}.abort_flag() = 0;
    *TcBars{b}.wait_limit() = wait_ns;
    tc::mbar_fence_init();
  }
};

// The output kernel's warps: 8 TMEM warps (0-7: operand and state
// conversions, P, the output), 8 builder warps (8-15: feature tiles) and the
// MMA issuer (16).
// (17 warps put 5 on one SM sub-partition, whose 16,384 registers then
// allow 96 per thread)
constexpr int TC32_OUT_THREADS = 544;
constexpr int TC32_BUILDER0 = 256;   // first builder thread
constexpr int TC32_ISSUER_WARP = 16;

// The output kernel stages each chunk's output tile (128 x W fp32) in the
// state copies' area and writes it with TMA stores when that area holds it.
__host__ __device__ constexpr bool tc32_out_tma(int rows, int nm, int W) {
  return (size_t)rows * nm * 4 >= (size_t)128 * W * 4;
}

// TMEM columns of the output kernel: the state blocks (nb x nm), O (nm), the
// scores A / P (128), then 1 or 2 readout feature tiles of 64 columns (hi and
// lo bf16 pairs of 64 features).
__host__ __device__ constexpr int tc32_ro_bufs(int nb, int nm) {
  return nb * nm + nm + 128 + 128 <= 512 ? 2 : (nb * nm + nm + 128 + 64 <= 512 ? 1 : 0);
}

// A worker warp's side of a ring of n slots with explicit barriers (full:
// the warps wrote the slot; empty: its MMAs are done).
struct Tc32Ring {
  uint32_t eph = 0, pend = 0;
  int s = 0, n = 2;
  __device__ __forceinline__ bool acquire(const TcBars& B, uint64_t* empty) {
    if (!((pend >> s) & 1u)) return true;
    const bool ok = tc_wait_warp(B, empty, (eph >> s) & 1u);
    eph ^= 1u << s;
    pend &= ~(1u << s);
    return ok;
  }
  __device__ __forceinline__ void release_tmem(uint64_t* full, int lane) {
    tc::tmem_wait_st();
    tc_warp_arrive(full, lane);
    pend |= 1u << s;
    s = (s + 1 == n) ? 0 : s + 1;
  }
};

// hi and lo bf16 pairs of two fp32 values.
__device__ __forceinline__ void tc32_split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = tc::pack_bf16x2(a, b);
  const float ha = __uint_as_float(hi << 16), hb = __uint_as_float(hi & 0xFFFF0000u);
  lo = tc::pack_bf16x2(a - ha, b - hb);
}
__device__ __forceinline__ void tc32_split8(const float* v, uint4& hi, uint4& lo) {
  tc32_split2(v[0], v[1], hi.x, lo.x);
  tc32_split2(v[2], v[3], hi.y, lo.y);
  tc32_split2(v[4], v[5], hi.z, lo.z);
  tc32_split2(v[6], v[7], hi.w, lo.w);
}

// Features [F*128 + 32*G, +32) of one token in fp32, split and stored: group
// e (8 features at block offset a = 32*G + 8*e) goes to ((a & mask) / 8) * 128
// bytes past `hi` and `lo` (mask 63 for a 64-wide tile, 127 for 128-wide).
template <int DK, int NT, int F, int G, int E>
struct Phi32Groups {
  static __device__ __forceinline__ void run(const float (&x)[DK + 1], uint8_t* hi, uint8_t* lo, int mask) {
    Phi32Groups<DK, NT, F, G, E - 1>::run(x, hi, lo, mask);
    constexpr int a = 32 * G + 8 * (E - 1);
    constexpr int A = F * 128 + a;
    float v[8];
    v[0] = feat_value<DK, NT, A + 0>(x); v[1] = feat_value<DK, NT, A + 1>(x);
    v[2] = feat_value<DK, NT, A + 2>(x); v[3] = feat_value<DK, NT, A + 3>(x);
    v[4] = feat_value<DK, NT, A + 4>(x); v[5] = feat_value<DK, NT, A + 5>(x);
    v[6] = feat_value<DK, NT, A + 6>(x); v[7] = feat_value<DK, NT, A + 7>(x);
    uint4 h, l;
    tc32_split8(v, h, l);
    const int off = ((a & mask) >> 3) * 128;
    *reinterpret_cast<uint4*>(hi + off) = h;
    *reinterpret_cast<uint4*>(lo + off) = l;
  }
};
template <int DK, int NT, int F, int G>
struct Phi32Groups<DK, NT, F, G, 0> {
  static __device__ __forceinline__ void run(const float (&)[DK + 1], uint8_t*, uint8_t*, int) {}
};

// Features [F*128 + 32*G, +32) of one token in fp32, split into hi and lo
// bf16 pairs in registers: pair e (features 2e, 2e + 1 of the quarter) in
// hi[e] and lo[e] (element 2e in the low half).
template <int DK, int NT, int F, int G, int E>
struct Phi32Reg {
  static __device__ __forceinline__ void run(const float (&x)[DK + 1], uint32_t (&hi)[16], uint32_t (&lo)[16]) {
    Phi32Reg<DK, NT, F, G, E - 1>::run(x, hi, lo);
    constexpr int A = F * 128 + 32 * G + 2 * (E - 1);
    tc32_split2(feat_value<DK, NT, A>(x), feat_value<DK, NT, A + 1>(x), hi[E - 1], lo[E - 1]);
  }
};
template <int DK, int NT, int F, int G>
struct Phi32Reg<DK, NT, F, G, 0> {
  static __device__ __forceinline__ void run(const float (&)[DK + 1], uint32_t (&)[16], uint32_t (&)[16]) {}
};

// Runtime (block f, quarter g) -> instantiation; one call site per kernel.
template <int DK, int NT, int F = 0>
__device__ __forceinline__ void build_phi32_regs(int f, int g, const float (&x)[DK + 1], uint32_t (&hi)[16],
                                                 uint32_t (&lo)[16]) {
  if constexpr (F < Tc32Shape<DK, NT>::NB) {
    if (f == F) {
      switch (g) {
        case 0: Phi32Reg<DK, NT, F, 0, 16>::run(x, hi, lo); break;
        case 1: Phi32Reg<DK, NT, F, 1, 16>::run(x, hi, lo); break;
        case 2: Phi32Reg<DK, NT, F, 2, 16>::run(x, hi, lo); break;
        default: Phi32Reg<DK, NT, F, 3, 16>::run(x, hi, lo); break;
      }
      return;
    }
    build_phi32_regs<DK, NT, F + 1>(f, g, x, hi, lo);
  }
}

// One group of 8 features (block F, group G8: features F*128 + 8*G8 ..) of one
// token, split and stored at `off` bytes past hi and lo.
template <int DK, int NT, int F, int G8>
__device__ __forceinline__ void phi32_group(const float (&x)[DK + 1], uint8_t* hi, uint8_t* lo, int off) {
  constexpr int A = F * 128 + 8 * G8;
  float v[8];
  v[0] = feat_value<DK, NT, A + 0>(x); v[1] = feat_value<DK, NT, A + 1>(x);
  v[2] = feat_value<DK, NT, A + 2>(x); v[3] = feat_value<DK, NT, A + 3>(x);
  v[4] = feat_value<DK, NT, A + 4>(x); v[5] = feat_value<DK, NT, A + 5>(x);
  v[6] = feat_value<DK, NT, A + 6>(x); v[7] = feat_value<DK, NT, A + 7>(x);
  uint4 h, l;
  tc32_split8(v, h, l);
  *reinterpret_cast<uint4*>(hi + off) = h;
  *reinterpret_cast<uint4*>(lo + off) = l;
}

// Groups gb + g0, gb + g0 + stride, ... below ge of the last feature block
// (fewer than 128 rows), so that every builder thread of a tile takes a share
// of its few rows.
template <int DK, int NT, int G8 = 0>
__device__ __forceinline__ void build_phi32_last(int gb, int ge, int g0, int stride, const float (&x)[DK + 1],
                                                 uint8_t* hi, uint8_t* lo, int mask) {
  using S = Tc32Shape<DK, NT>;
  if constexpr (G8 < S::LAST_ROWS / 8) {
    if (G8 >= gb && G8 < ge && (G8 - gb) % stride == g0)
      phi32_group<DK, NT, S::NB - 1, G8>(x, hi, lo, (((8 * G8) & mask) >> 3) * 128);
    build_phi32_last<DK, NT, G8 + 1>(gb, ge, g0, stride, x, hi, lo, mask);
  }
}

// Runtime (block f, quarter g) -> instantiation; one call site per kernel.
template <int DK, int NT, int F = 0>
__device__ __forceinline__ void build_phi32(int f, int g, const float (&x)[DK + 1], uint8_t* hi, uint8_t* lo,
                                            int mask) {
  if constexpr (F < Tc32Shape<DK, NT>::NB) {
    if (f == F) {
      switch (g) {
        case 0: Phi32Groups<DK, NT, F, 0, 4>::run(x, hi, lo, mask); break;
        case 1: Phi32Groups<DK, NT, F, 1, 4>::run(x, hi, lo, mask); break;
        case 2: Phi32Groups<DK, NT, F, 2, 4>::run(x, hi, lo, mask); break;
        default: Phi32Groups<DK, NT, F, 3, 4>::run(x, hi, lo, mask); break;
      }
      return;
    }
    build_phi32<DK, NT, F + 1>(f, g, x, hi, lo, mask);
  }
}

// Staging loads of one chunk: fp32 q (if tq), k and the W value columns, each
// as a [col/4][token][4] tile (4-D tensor maps; box (4, 128, cols/4, 1)), so
// that consecutive threads (tokens) read consecutive 16-byte pieces.
__device__ __forceinline__ void tc32_issue_staging(const Tc32Smem& L, uint8_t* smem, uint64_t* bar,
                                                   const CUtensorMap* tq, const CUtensorMap* tk,
                                                   const CUtensorMap* tv, long long t0, int head, int c0, int W,
                                                   int dk) {
  if (!tc::elect_one()) return;
  tc::mbar_arrive_expect_tx(bar, (uint32_t)((tq ? 2 : 1) * 128 * dk * 4 + 128 * W * 4));
  if (tq) tc::tma_load_4d(smem + L.qs, tq, bar, 0, (int)t0, 0, head);
  tc::tma_load_4d(smem + L.ks, tk, bar, 0, (int)t0, 0, head);
  tc::tma_load_4d(smem + L.vs, tv, bar, 0, (int)t0, c0 / 4, head);
}

// Three-term split product into one accumulator: A_hi B_hi + A_hi B_lo + A_lo B_hi.
__device__ __forceinline__ void mma3(uint32_t d, uint64_t ah, uint64_t al, uint64_t bh, uint64_t bl, uint32_t id,
                                     uint32_t acc) {
  tc::mma_bf16_elect(d, ah, bh, id, acc);
  tc::mma_bf16_elect(d, ah, bl, id, 1u);
  tc::mma_bf16_elect(d, al, bh, id, 1u);
}

// The same with A in TMEM (hi and lo halves at a_hi and a_lo).
__device__ __forceinline__ void mma3_ts(uint32_t d, uint32_t ah, uint32_t al, uint64_t bh, uint64_t bl, uint32_t id,
                                        uint32_t acc) {
  tc::mma_bf16_ts_elect(d, ah, bh, id, acc);
  tc::mma_bf16_ts_elect(d, ah, bl, id, 1u);
  tc::mma_bf16_ts_elect(d, al, bh, id, 1u);
}

// P in TMEM, written over the scores A: the worker warp of half h owns keys
// [32h, 32h + 32) and [64 + 32h, 64 + 32h + 32) of its rows and puts the hi and
// lo bf16 pairs of each 32-key piece in the piece's own 32 columns (hi in the
// first 16, lo in the last 16). Keys [16k, 16k + 16) are then 8 columns at
// tc32_p_col(k) (hi) and tc32_p_col(k) + 16 (lo) past the start of A.
__host__ __device__ constexpr int tc32_p_col(int k) { return 32 * (k / 2) + 8 * (k % 2); }

// Workers: fp32 staging ([col/4][t][4]) -> hi/lo operand tiles. q, k:
// [e/8][t][8] (K-major); v: [c/8][t][8] (MN-major), W value columns (the
// ones group stays as set up). Thread (t = tid & 127, half = tid >> 7)
// converts half of its token's row.
__device__ __forceinline__ void tc32_convert_rows(const uint8_t* xs, uint8_t* th, uint8_t* tl, int cols, int t,
                                                  int half) {
  for (int g = half * (cols / 16); g < (half + 1) * (cols / 16); ++g) {
    float v[8];
    const float4 a = *reinterpret_cast<const float4*>(xs + (2 * g) * 2048 + t * 16);
    const float4 b = *reinterpret_cast<const float4*>(xs + (2 * g + 1) * 2048 + t * 16);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    uint4 h, l;
    tc32_split8(v, h, l);
    *reinterpret_cast<uint4*>(th + g * 2048 + t * 16) = h;
    *reinterpret_cast<uint4*>(tl + g * 2048 + t * 16) = l;
  }
}
template <int DK>
__device__ __forceinline__ void tc32_load_x(const uint8_t* xs, int t, float (&x)[DK + 1]) {
#pragma unroll
  for (int e = 0; e < DK; e += 4) {
    const float4 a = *reinterpret_cast<const float4*>(xs + (e / 4) * 2048 + t * 16);
    x[e] = a.x; x[e + 1] = a.y; x[e + 2] = a.z; x[e + 3] = a.w;
  }
}

// TMEM state block f -> its hi/lo bf16 copies (rows_f rows, nm columns):
// element (a, c) at (c/8) * rows_f*16 + a*16 + (c%8)*2 of block f's region.
template <int DK, int NT>
__device__ __forceinline__ void tc32_convert_state(uint8_t* sh, uint8_t* sl, uint32_t tm, uint32_t lane_off, int nm,
                                                   int f, int i, int half) {
  using S = Tc32Shape<DK, NT>;
  const int rows = S::rows(f);
  const size_t boff = (size_t)f * 128 * nm * 2;
  for (int g = half; g < nm / 16; g += 2) {
    uint32_t rr[16];
    tc::tmem_ld16(tm + lane_off + f * nm + g * 16, rr);
    tc::tmem_wait_ld();
    if (i < rows) {
      float v[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(rr[e]);
      uint4 h0, l0, h1, l1;
      tc32_split8(v, h0, l0);
      tc32_split8(v + 8, h1, l1);
      const size_t o0 = boff + (size_t)(2 * g) * rows * 16 + i * 16, o1 = o0 + (size_t)rows * 16;
      *reinterpret_cast<uint4*>(sh + o0) = h0;
      *reinterpret_cast<uint4*>(sl + o0) = l0;
      *reinterpret_cast<uint4*>(sh + o1) = h1;
      *reinterpret_cast<uint4*>(sl + o1) = l1;
    }
  }
}

// Update MMAs of one tile (ring slot at shared address a) into the state
// block at TMEM column d: a 64-token tile (tokens 64h..) of a full block, or
// the compact 128-token tile of the last block's GL feature groups.
__device__ __forceinline__ void tc32_issue_update(uint32_t d, uint32_t a, uint64_t dVh, uint64_t dVl, uint32_t id_up,
                                                  bool compact, int GL, int h, bool acc0) {
  if (!compact) {
    const uint64_t dAh = tc::sdesc(a, 2048, 128), dAl = tc::sdesc(a + 16384, 2048, 128);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      mma3(d, dAh + (uint64_t)(k * 256), dAl + (uint64_t)(k * 256), dVh + (uint64_t)(64 * h + k * 16),
           dVl + (uint64_t)(64 * h + k * 16), id_up, (acc0 || k > 0) ? 1u : 0u);
  } else {
    // token groups GL*128 bytes apart (K direction), feature groups 128 apart
    const uint32_t lbo = (uint32_t)GL * 128u;
    const uint64_t dAh = tc::sdesc(a, lbo, 128), dAl = tc::sdesc(a + 16384, lbo, 128);
    for (int k = 0; k < 8; ++k)
      mma3(d, dAh + (uint64_t)(k * 2 * lbo / 16), dAl + (uint64_t)(k * 2 * lbo / 16), dVh + (uint64_t)(16 * k),
           dVl + (uint64_t)(16 * k), id_up, (acc0 || k > 0) ? 1u : 0u);
  }
}

// One worker thread's share (of 256) of an update tile: a 64-token tile of a
// full block (token 64h + (w & 63), quarter w >> 6), or the compact tile of
// the last block (token w & 127, groups (w >> 7), (w >> 7) + 2, ..).
// xk holds the thread's inputs for tokens (w & 63) and 64 + (w & 63).
template <int DK, int NT>
__device__ __forceinline__ void tc32_build_update(uint8_t* slot, int f, int h, int w, const float (&xk)[2][DK + 1]) {
  using S = Tc32Shape<DK, NT>;
  float x[DK + 1];
  if (S::upd_tiles(f) == 1) {
    const int t = w & 127;
#pragma unroll
    for (int e = 0; e <= DK; ++e) x[e] = ((w >> 6) & 1) ? xk[1][e] : xk[0][e];
    uint8_t* hi = slot + (t / 8) * (S::GL * 128) + (t % 8) * 16;
    build_phi32_last<DK, NT>(0, S::GL, w >> 7, 2, x, hi, hi + 16384, 127);
  } else {
    const int tq = w & 63, qq = w >> 6;
#pragma unroll
    for (int e = 0; e <= DK; ++e) x[e] = h ? xk[1][e] : xk[0][e];
    uint8_t* hi = slot + (tq / 8) * 2048 + (tq % 8) * 16;
    if (S::rows(f) < 128)   // a last block of more than 64 rows: over the 4 threads of a token
      build_phi32_last<DK, NT>(0, S::GL, qq, 4, x, hi, hi + 16384, 127);
    else
      build_phi32<DK, NT>(f, qq, x, hi, hi + 16384, 127);
  }
}

// ---------------------------------------------------------------------------
// span_state_tc32: the state sum of one span -> scratch (fp32 inputs).
// ---------------------------------------------------------------------------
template <int DK, int NT>
__global__ void __launch_bounds__(TC_THREADS, 1)
span_state_tc32_kernel(const TcParams p, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v) {
  using S = Tc32Shape<DK, NT>;
  constexpr int D = S::D, NB = S::NB, DPAD = round_up(D, 4);
  extern __shared__ __align__(1024) uint8_t smem[];
  const TcUnit u = tc_unit(p);
  const int W = u.W, nm = u.nm;
  const Tc32Smem L(DK, W, nm, S::ROWS, p.ring, p.span_layout != 0);
  const Tc32Bars X{reinterpret_cast<uint64_t*>(smem + L.bar)};
  const TcBars B = X.ring_bars();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wq = warp & 3, half = (warp >> 2) & 1;
  // v tiles in two buffers when sh/sl hold the second (the span-pass layout,
  // or the shared layout's state-copy area when it is large enough), so that
  // the workers convert the next chunk's v while this chunk's MMAs still
  // read the other
  const bool v2 = p.span_layout != 0 || S::ROWS >= 128;
  auto vh_b = [&](int vb) { return vb ? smem + L.sh : smem + L.vh; };
  auto vl_b = [&](int vb) { return vb ? smem + L.sh + (size_t)128 * nm * 2 : smem + L.vl; };

  tc::grid_dep_launch();   // the scan after this pass may be launched now
  if (warp == 0) tc::tmem_alloc(B.tmem_slot(), 512);
  if (tid == 0) X.init(p.wait_ns);
  if (warp == 0) {
    __syncwarp();   // the first inputs at once, overlapping the set-up
    if (u.n_chunks > 0)
      tc32_issue_staging(L, smem, X.stg_full(), nullptr, &tm_k, &tm_v, u.t_begin, u.head, u.c0, W, DK);
  }
  if (tid < TC_WORKERS) {
    for (int vb = 0; vb < (v2 ? 2 : 1); ++vb) {
      tc_write_ones(vh_b(vb), W, tid);
      for (int e = tid; e < 256; e += TC_WORKERS)
        *reinterpret_cast<uint4*>(vl_b(vb) + (W / 8 + (e & 1)) * 2048 + (e >> 1) * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
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
    const uint32_t id_up = tc::idesc_bf16(128, nm, true, true);
    TcIssuerRing ring;
    int req = u.n_chunks > 0 ? 1 : 0, got = 0;   // the first staging load was issued above
    bool ok = true;
    for (int c = 0; c < u.n_chunks && ok; ++c) {
      const long long t0 = u.t_begin + (long long)c * TC_C;
      const int vb = v2 ? (c & 1) : 0;
      const uint64_t dVh = tc::sdesc(tc::smem_u32(vh_b(vb)), 128, 2048);
      const uint64_t dVl = tc::sdesc(tc::smem_u32(vl_b(vb)), 128, 2048);
      if (!(ok = tc_wait_warp(B, X.tiles(), c & 1u))) break;
      ++got;
      if (c + 1 < u.n_chunks) {
        if (!(ok = tc_wait_warp(B, X.stg_free(), c & 1u))) break;
        tc32_issue_staging(L, smem, X.stg_full(), nullptr, &tm_k, &tm_v, t0 + TC_C, u.head, u.c0, W, DK);
        ++req;
      }
      for (int f = 0; f < NB && ok; ++f)
        for (int h = 0; h < S::upd_tiles(f); ++h, pos.next()) {
          if (!(ok = ring.take(B, pos.s))) break;
          tc32_issue_update(tm + f * nm, tc::smem_u32(smem + L.slot(pos.s)), dVh, dVl, id_up,
                            S::upd_tiles(f) == 1, S::GL, h, c > 0 || h > 0);
          tc::mma_commit_elect(B.sempty(pos.s));
        }
      if (!ok) break;
      if (v2) tc::mma_commit_elect(X.vfree(vb));
      tc::mma_commit_elect(B.chunk());
    }
    // drain: every MMA and every staging load that was requested
    tc::mma_commit_elect(B.drain());
    tc::mbar_wait(B.drain(), 0, TC_WAIT_NS);
    for (; got < req; ++got) tc::mbar_wait(X.stg_full(), got & 1u, TC_WAIT_NS);
  } else {
    const int tq = tid & 63;   // update inputs: tokens tq and 64 + tq
    TcWorkerRing ring;
    for (int c = 0; c < u.n_chunks; ++c) {
      const long long t0 = u.t_begin + (long long)c * TC_C;
      const int valid = (int)min((long long)TC_C, u.t_end - t0);
      const int vb = v2 ? (c & 1) : 0;
      if (!tc_wait_warp(B, X.stg_full(), c & 1u)) break;
      // the v buffer is free: (two buffers) the MMAs of chunk c - 2 are done,
      // one barrier per buffer so that each wait is for its next phase;
      // (one buffer) the MMAs of chunk c - 1 are done
      if (v2 && c >= 2 && !tc_wait_warp(B, X.vfree(vb), ((c >> 1) - 1) & 1u)) break;
      if (!v2 && c > 0 && !tc_wait_warp(B, B.chunk(), (c - 1) & 1u)) break;
      tc32_convert_rows(smem + L.vs, vh_b(vb), vl_b(vb), W, tid & 127, half);
      float xk[2][DK + 1];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        tc32_load_x<DK>(smem + L.ks, 64 * h + tq, xk[h]);
        xk[h][DK] = (64 * h + tq < valid) ? 1.0f : 0.0f;
      }
      tc::fence_proxy_async();
      tc_warp_arrive(X.stg_free(), lane);
      tc_warp_arrive(X.tiles(), lane);
      bool ok = true;
      for (int f = 0; f < NB && ok; ++f)
        for (int h = 0; h < S::upd_tiles(f); ++h, pos.next()) {
          if (!(ok = ring.acquire(B, pos.s))) break;
          tc32_build_update<DK, NT>(smem + L.slot(pos.s), f, h, tid, xk);
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
    tc_store_state<D, DPAD, NB>(dst, tm, lane_off, nm, W, u.c0, p.dv, u.slice == 0, wq, lane, half);
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
// span_output_tc32: outputs of one span (fp32 inputs), state carried in TMEM.
// Per chunk: the workers split the staged q, k, v into hi/lo tiles (and keep
// their inputs in registers); the issuer runs Q K^T; the workers write P in
// two key halves; the issuer runs P [V,1] and the readouts, the workers write
// the output once O is complete, then the update tiles; after every MMA of
// the chunk the workers split the updated state into its hi/lo copies.
// ---------------------------------------------------------------------------
template <int DK, int NT>
__global__ void __launch_bounds__(TC32_OUT_THREADS, 1)
span_output_tc32_kernel(const TcParams p, const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_o) {
  using S = Tc32Shape<DK, NT>;
  constexpr int D = S::D, NB = S::NB, DPAD = round_up(D, 4);
  extern __shared__ __align__(1024) uint8_t smem[];
  const TcUnit u = tc_unit(p);
  const int W = u.W, nm = u.nm;
  const Tc32Smem L(DK, W, nm, S::ROWS, p.ring);
  const Tc32Bars X{reinterpret_cast<uint64_t*>(smem + L.bar)};
  const TcBars B = X.ring_bars();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wq = warp & 3, half = (warp >> 2) & 1;
  const bool single = (p.n_spans == 1);
  const size_t st_elems = (size_t)DPAD * (p.dv + 1);
  TSA_TRACE_DECL
  TSA_TRACE_EVENT(30, 0);
  // the span's initial state: the span pass's prefix (several spans), the
  // caller's state (ACCUMULATE) or zero
  const float* st_src = nullptr;
  if (!single) st_src = p.scratch + ((size_t)u.head * p.n_spans + u.span) * st_elems;
  else if (p.accumulate) st_src = p.states + (size_t)u.head * st_elems;
  const uint32_t st_bytes = (uint32_t)(st_elems * 4);
  // one bulk copy into the (still idle) ring area when it fits there
  const bool st_bulk = st_src != nullptr && st_bytes % 16 == 0 && st_bytes <= (uint32_t)p.ring * 32768u;

  if (warp == 0) tc::tmem_alloc(B.tmem_slot(), 512);
  if (tid == 0) X.init(p.wait_ns, 16);
  if (warp == 0) {
    // the first chunk's inputs at once (ready before this call's first
    // launch), overlapping the set-up below
    __syncwarp();
    if (u.n_chunks > 0)
      tc32_issue_staging(L, smem, X.stg_full(), &tm_q, &tm_k, &tm_v, u.t_begin, u.head, u.c0, W, DK);
  }
  if (tid < TC_WORKERS) {
    tc_write_ones(smem + L.vh, W, tid);
    for (int e = tid; e < 256; e += TC_WORKERS)
      *reinterpret_cast<uint4*>(smem + L.vl + (W / 8 + (e & 1)) * 2048 + (e >> 1) * 16) = make_uint4(0u, 0u, 0u, 0u);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = *B.tmem_slot();
  const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
  const uint32_t col_O = (uint32_t)(NB * nm);
  const uint32_t col_A = col_O + (uint32_t)nm;   // A has its own columns (no overlap with O)
  const uint32_t col_R = col_A + 128u;            // readout feature tiles, RB x 64 columns
  const int RB = tc32_ro_bufs(NB, nm);
  const int i = wq * 32 + lane;   // TMEM lane = query row / feature row of a block
  const bool out_tma = tc32_out_tma(S::ROWS, nm, W);

  TSA_TRACE_EVENT(31, 0);
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  TSA_TRACE_EVENT(33, 0);
  TcRingPos pos;
  pos.R = p.ring;

  if (warp == TC32_ISSUER_WARP) {
    // ------------------------------ issuer ---------------------------------
    const uint32_t id_qk = tc::idesc_bf16(128, 128, false, false);
    const uint32_t id_pv = tc::idesc_bf16(128, nm, false, true);
    const uint32_t id_up = tc::idesc_bf16(128, nm, true, true);
    const uint64_t dQh = tc::sdesc(tc::smem_u32(smem + L.qh), 2048, 128);
    const uint64_t dQl = tc::sdesc(tc::smem_u32(smem + L.ql), 2048, 128);
    const uint64_t dKh = tc::sdesc(tc::smem_u32(smem + L.kh), 2048, 128);
    const uint64_t dKl = tc::sdesc(tc::smem_u32(smem + L.kl), 2048, 128);
    const uint64_t dVh = tc::sdesc(tc::smem_u32(smem + L.vh), 128, 2048);
    const uint64_t dVl = tc::sdesc(tc::smem_u32(smem + L.vl), 128, 2048);
    TcIssuerRing ring;
    int ro_s = 0;
    uint32_t ro_ph = 0;
    int req = u.n_chunks > 0 ? 1 : 0, got = 0;   // the first staging load was issued above
    bool ok = true;
    for (int c = 0; c < u.n_chunks && ok; ++c) {
      const long long t0 = u.t_begin + (long long)c * TC_C;
      const bool need_update = single || (c + 1 < u.n_chunks);
      // the workers' tile conversion follows their reading of O and of A
      if (!(ok = tc_wait_warp(B, X.tiles(), c & 1u))) break;
      ++got;
      TSA_TRACE_EVENT(1, c);
      tc::fence_after_sync();
#pragma unroll
      for (int k = 0; k < DK / 16; ++k)
        mma3(tm + col_A, dQh + (uint64_t)(k * 256), dQl + (uint64_t)(k * 256), dKh + (uint64_t)(k * 256),
             dKl + (uint64_t)(k * 256), id_qk, k > 0 ? 1u : 0u);
      tc::mma_commit_elect(B.qk());
      // the state copies for this chunk's readouts (one conversion per chunk)
      if (!(ok = tc_wait_warp(B, B.conv(), c & 1u))) break;
      TSA_TRACE_EVENT(2, c);
      // O = phi(Q_f) [S_f, z_f] summed over blocks, 64 features at a time,
      // the feature tiles read from TMEM
      for (int f = 0; f < NB && ok; ++f) {
        const int rows = S::rows(f);
        const uint32_t sb = (uint32_t)((size_t)f * 128 * nm * 2);
        const uint64_t dSh = tc::sdesc(tc::smem_u32(smem + L.sh) + sb, 128, (uint32_t)rows * 16);
        const uint64_t dSl = tc::sdesc(tc::smem_u32(smem + L.sl) + sb, 128, (uint32_t)rows * 16);
        for (int h = 0; h < S::halves(f); ++h) {
          if (!(ok = tc_wait_warp(B, X.rofull(ro_s), (ro_ph >> ro_s) & 1u))) break;
          ro_ph ^= 1u << ro_s;
          tc::fence_after_sync();
          const uint32_t a = tm + col_R + 64u * (uint32_t)ro_s;
          const int ks = min(64, rows - 64 * h) / 16;
          for (int k = 0; k < ks; ++k) {
            const uint32_t ah = a + (uint32_t)tc32_p_col(k);
            mma3_ts(tm + col_O, ah, ah + 16u, dSh + (uint64_t)(64 * h + 16 * k), dSl + (uint64_t)(64 * h + 16 * k),
                    id_pv, (f > 0 || h > 0 || k > 0) ? 1u : 0u);
          }
          tc::mma_commit_elect(X.roempty(ro_s));
          ro_s = (ro_s + 1 == RB) ? 0 : ro_s + 1;
        }
      }
      if (!ok) break;
      // the workers have converted the staged chunk: fetch the next one
      if (c + 1 < u.n_chunks) {
        if (!(ok = tc_wait_warp(B, X.stg_free(), c & 1u))) break;
        tc32_issue_staging(L, smem, X.stg_full(), &tm_q, &tm_k, &tm_v, t0 + TC_C, u.head, u.c0, W, DK);
        ++req;
      }
      // O += P [V, 1], P from TMEM, 16 keys per step
      if (!(ok = tc_wait_warp(B, X.pready(), c & 1u))) break;
      tc::fence_after_sync();
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t ph = tm + col_A + (uint32_t)tc32_p_col(k);
        mma3_ts(tm + col_O, ph, ph + 16u, dVh + (uint64_t)(16 * k), dVl + (uint64_t)(16 * k), id_pv, 1u);
      }
      // (testing only: with dbg_withhold the first chunk's O is never
      // published, so the TMEM warps' bounded wait for it runs out)
      if (!(p.dbg_withhold && c == 0)) tc::mma_commit_elect(B.odone());
      TSA_TRACE_EVENT(3, c);
      // S_f += phi(K_f)^T [V, 1], 64 tokens at a time
      if (need_update) {
        for (int f = 0; f < NB && ok; ++f)
          for (int h = 0; h < S::upd_tiles(f); ++h, pos.next()) {
            if (!(ok = ring.take(B, pos.s))) break;
            tc32_issue_update(tm + f * nm, tc::smem_u32(smem + L.slot(pos.s)), dVh, dVl, id_up,
                              S::upd_tiles(f) == 1, S::GL, h, true);
            tc::mma_commit_elect(B.sempty(pos.s));
          }
        if (!ok) break;
      }
      tc::mma_commit_elect(B.chunk());
      TSA_TRACE_EVENT(4, c);
    }
    tc::mma_commit_elect(B.drain());
    tc::mbar_wait(B.drain(), 0, TC_WAIT_NS);
    for (; got < req; ++got) tc::mbar_wait(X.stg_full(), got & 1u, TC_WAIT_NS);
    if (*X.copy_issued()) tc::mbar_wait(X.stload(), 0, TC_WAIT_NS);   // the initial-state copy, too
  } else if (tid < TC_WORKERS) {
    // ---------------------------- TMEM warps -------------------------------
    // q, k, v and the state -> hi/lo operands, P, the output; thread = TMEM
    // lane i (query row / feature row), its half of the columns
    const int t = tid & 127;
    const int row_hi = wq * 32 + 31;
    float* og = static_cast<float*>(p.out) + (size_t)u.head * p.N * p.dv + u.c0;
    for (int c = 0; c < u.n_chunks; ++c) {
      const long long t0 = u.t_begin + (long long)c * TC_C;
      const int valid = (int)min((long long)TC_C, u.t_end - t0);
      TSA_TRACE_EVENT(10, c);
      // q, k -> hi/lo tiles for Q K^T (the previous Q K^T is done: its P was
      // read; the previous output is written: O may be overwritten)
      if (!tc_wait_warp(B, X.stg_full(), c & 1u)) break;
      tc32_convert_rows(smem + L.qs, smem + L.qh, smem + L.ql, DK, t, half);
      tc32_convert_rows(smem + L.ks, smem + L.kh, smem + L.kl, DK, t, half);
      tc::fence_proxy_async();
      tc_warp_arrive(X.tiles(), lane);
      TSA_TRACE_EVENT(12, c);
      if (c == 0) {
        // the span's initial state -> TMEM, then its hi/lo copies (here, not
        // before the chunk loop, so that the builders, the q K^T and P of the
        // first chunk overlap its arrival)
        // the grid this one depends on (the scan) is done: its prefixes, or
        // the caller's state, may be read; one bulk copy into the ring area
        tc::grid_dep_wait();
        const float* src = st_src;
        if (st_bulk) {
          if (warp == 0 && tc::elect_one()) {
            *X.copy_issued() = 1;
            tc::mbar_arrive_expect_tx(X.stload(), st_bytes);
            tc::bulk_load(smem + L.ring0, st_src, st_bytes, X.stload());
          }
          if (!tc_wait_warp(B, X.stload(), 0u)) break;
          src = reinterpret_cast<const float*>(smem + L.ring0);
        }
        for (int f = 0; f < NB; ++f) {
          const int a = f * 128 + i;
          for (int g = half; g < nm / 16; g += 2) {
            uint32_t r[16];
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
              const int cc = g * 16 + 4 * e4;
              float4 x = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
              if (src != nullptr && a < D) {
                if (cc < W && TSA_DCHECK_STATE((size_t)a * p.dv + u.c0 + cc, 4, (size_t)DPAD * p.dv))
                  x = *reinterpret_cast<const float4*>(src + (size_t)a * p.dv + u.c0 + cc);
                else if (cc == W) x.x = src[(size_t)DPAD * p.dv + a];
              }
              r[4 * e4] = __float_as_uint(x.x);
              r[4 * e4 + 1] = __float_as_uint(x.y);
              r[4 * e4 + 2] = __float_as_uint(x.z);
              r[4 * e4 + 3] = __float_as_uint(x.w);
            }
            tc::tmem_st16(tm + lane_off + f * nm + g * 16, r);
          }
        }
        tc::tmem_wait_st();
        TSA_TRACE_EVENT(32, 0);
        tc::fence_after_sync();
        for (int fb = 0; fb < NB; ++fb)
          tc32_convert_state<DK, NT>(smem + L.sh, smem + L.sl, tm, lane_off, nm, fb, i, half);
        tc::fence_proxy_async();
        tc_warp_arrive(B.conv(), lane);
      } else {
        // the previous chunk's state -> hi/lo copies for this chunk's readouts
        if (!tc_wait_warp(B, B.chunk(), (c - 1) & 1u)) break;
        if (out_tma) {
          // every warp's output store has read its piece of the area
          if (lane == 0) tc::bulk_wait_read();
          tc_warp_arrive(X.ostored(), lane);
          if (!tc_wait_warp(B, X.ostored(), (c - 1) & 1u)) break;
        }
        TSA_TRACE_EVENT(24, c);
        tc::fence_after_sync();
        for (int fb = 0; fb < NB; ++fb)
          tc32_convert_state<DK, NT>(smem + L.sh, smem + L.sl, tm, lane_off, nm, fb, i, half);
        tc::fence_proxy_async();
        tc_warp_arrive(B.conv(), lane);
        TSA_TRACE_EVENT(25, c);
      }
      // v -> hi/lo tiles (the previous chunk's MMAs, which read v, are done)
      tc32_convert_rows(smem + L.vs, smem + L.vh, smem + L.vl, W, t, half);
      tc::fence_proxy_async();
      tc_warp_arrive(X.stg_free(), lane);
      // P = mask(T_n(A)) written over A in TMEM (tc32_p_col): row i, the
      // warp's two 32-key pieces, while the readout MMAs run
      if (!tc_wait_warp(B, B.qk(), c & 1u)) break;
      TSA_TRACE_EVENT(13, c);
      tc::fence_after_sync();
      for (int kh2 = 0; kh2 < 2; ++kh2) {
        const int jb = 64 * kh2 + 32 * half;
        uint32_t ph[16], pl[16];
        if (jb <= row_hi) {   // warp-uniform: all 32 keys above the diagonal -> zeros
          uint32_t rr[32];
          tc::tmem_ld32(tm + lane_off + col_A + jb, rr);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j = jb + 2 * e;
            const float p0 = (j <= i && i < valid) ? taylor_T<NT>(__uint_as_float(rr[2 * e])) : 0.0f;
            const float p1 = (j + 1 <= i && i < valid) ? taylor_T<NT>(__uint_as_float(rr[2 * e + 1])) : 0.0f;
            tc32_split2(p0, p1, ph[e], pl[e]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) ph[e] = pl[e] = 0u;
        }
        tc::tmem_st16(tm + lane_off + col_A + jb, ph);
        tc::tmem_st16(tm + lane_off + col_A + jb + 16, pl);
      }
      tc::tmem_wait_st();
      tc_warp_arrive(X.pready(), lane);
      TSA_TRACE_EVENT(14, c);
      // out = O[:, :W] / O[:, W]; thread row i, its half of W
      if (!tc_wait_warp(B, B.odone(), c & 1u)) break;
      TSA_TRACE_EVENT(15, c);
      tc::fence_after_sync();
      {
        const int cw = W / 2;   // columns of this half: [half*cw, +cw), cw = 16, 32 or 64
        uint32_t rd[16];
        tc::tmem_ld16(tm + lane_off + col_O + W, rd);
        tc::tmem_wait_ld();
        const float inv = 1.0f / __uint_as_float(rd[0]);
        if (out_tma) {
          // the warp's 32 rows x cw columns -> its staging piece [cw/4][32][4]
          // in the state copies' area (idle from odone to the conversion),
          // then one TMA store; rows past the sequence end are clipped
          uint8_t* piece = smem + L.sh + (size_t)warp * 128 * cw;
          for (int e0 = 0; e0 < cw; e0 += 16) {
            uint32_t rr[16];
            tc::tmem_ld16(tm + lane_off + col_O + half * cw + e0, rr);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; e += 4)
              *reinterpret_cast<float4*>(piece + ((e0 + e) / 4) * 512 + lane * 16) =
                  make_float4(__uint_as_float(rr[e]) * inv, __uint_as_float(rr[e + 1]) * inv,
                              __uint_as_float(rr[e + 2]) * inv, __uint_as_float(rr[e + 3]) * inv);
          }
          tc::fence_proxy_async();
          __syncwarp();
          if (lane == 0 && t0 + wq * 32 < u.t_end) {
            tc::tma_store_4d(&tm_o, piece, 0, (int)(t0 + wq * 32), (u.c0 + half * cw) / 4, u.head);
            tc::bulk_commit();
          }
        } else {
          float* dst = og + (size_t)(t0 + i) * p.dv + half * cw;
          for (int e0 = 0; e0 < cw; e0 += 16) {
            uint32_t rr[16];
            tc::tmem_ld16(tm + lane_off + col_O + half * cw + e0, rr);
            tc::tmem_wait_ld();
            if (i < valid) {
#pragma unroll
              for (int e = 0; e < 16; e += 4)
                *reinterpret_cast<float4*>(dst + e0 + e) =
                    make_float4(__uint_as_float(rr[e]) * inv, __uint_as_float(rr[e + 1]) * inv,
                                __uint_as_float(rr[e + 2]) * inv, __uint_as_float(rr[e + 3]) * inv);
            }
          }
        }
      }
      TSA_TRACE_EVENT(16, c);
    }
  } else {
    // --------------------------- builder warps ------------------------------
    // readout tiles (token t = this thread's TMEM lane, quarter 2h + half of
    // a 64-feature half h) into TMEM, then update tiles (token 64h + tq,
    // quarter qq) through the shared-memory ring; the feature arithmetic has
    // one call site
    const int bt = tid - TC32_BUILDER0;
    const int t = bt & 127, tq = bt & 63, qq = bt >> 6;
    const int urow = (tq / 8) * 2048 + (tq % 8) * 16;    // 64-token, 128-wide tiles
    Tc32Ring ro;
    ro.n = RB;
    TcWorkerRing ring;
    for (int c = 0; c < u.n_chunks; ++c) {
      const long long t0 = u.t_begin + (long long)c * TC_C;
      const int valid = (int)min((long long)TC_C, u.t_end - t0);
      const bool need_update = single || (c + 1 < u.n_chunks);
      if (!tc_wait_warp(B, X.stg_full(), c & 1u)) break;
      TSA_TRACE_EVENT(11, c);
      float xk[2][DK + 1];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        tc32_load_x<DK>(smem + L.ks, 64 * h + tq, xk[h]);
        xk[h][DK] = (64 * h + tq < valid) ? 1.0f : 0.0f;
      }
      const int n_ro = [] { int n = 0; for (int f = 0; f < NB; ++f) n += S::halves(f); return n; }();
      const int nuse = n_ro + (need_update ? S::n_upd() : 0);
      int f = 0, h = 0;
      bool ok = true;
      for (int k = 0; k < nuse; ++k) {
        if (k == n_ro) {
          // q and k of the staging are read
          tc_warp_arrive(X.stg_free(), lane);
          f = 0;
          h = 0;
          // the first update tile goes where the initial state was copied:
          // wait until the TMEM warps have converted it
          if (c == 0 && !(ok = tc_wait_warp(B, B.conv(), 0u))) break;
        }
        const bool upd = (k >= n_ro);
        const int g = upd ? qq : 2 * h + half;
        TSA_TRACE_EVENT(20, k);
        if (!(ok = upd ? ring.acquire(B, pos.s) : ro.acquire(B, X.roempty(ro.s)))) break;
        TSA_TRACE_EVENT(21, k);
        if (upd && S::rows(f) < 128) {
          // the last block: its compact tile (or, above 64 rows, its rows
          // spread over the 4 threads of a token)
          tc32_build_update<DK, NT>(smem + L.slot(pos.s), f, h, bt, xk);
        } else if (32 * g < S::rows(f)) {
          float x[DK + 1];
          if (upd) {
#pragma unroll
            for (int e = 0; e <= DK; ++e) x[e] = h ? xk[1][e] : xk[0][e];
          } else {
            tc32_load_x<DK>(smem + L.qs, t, x);
            x[DK] = 1.0f;
          }
          uint32_t hv[16], lv[16];
          TSA_TRACE_EVENT(26, k);
          build_phi32_regs<DK, NT>(f, g, x, hv, lv);
          TSA_TRACE_EVENT(27, k);
          if (upd) {
            uint8_t* hi = smem + L.slot(pos.s) + urow;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int off = (4 * g + e) * 128;
              *reinterpret_cast<uint4*>(hi + off) = make_uint4(hv[4 * e], hv[4 * e + 1], hv[4 * e + 2], hv[4 * e + 3]);
              *reinterpret_cast<uint4*>(hi + 16384 + off) =
                  make_uint4(lv[4 * e], lv[4 * e + 1], lv[4 * e + 2], lv[4 * e + 3]);
            }
          } else {
            const uint32_t col = tm + lane_off + col_R + 64u * (uint32_t)ro.s + 32u * (uint32_t)half;
            tc::tmem_st16(col, hv);
            tc::tmem_st16(col + 16u, lv);
          }
        }
        TSA_TRACE_EVENT(22, k);
        if (upd) {
          ring.release(B, pos.s, lane);
          pos.next();
        } else {
          ro.release_tmem(X.rofull(ro.s), lane);
        }
        TSA_TRACE_EVENT(28, k);
        // next (f, h): readouts walk the block's 64-feature halves, updates
        // its update tiles
        if (++h == (upd ? S::upd_tiles(f) : S::halves(f))) { h = 0; ++f; }
      }
      if (!ok) break;
      if (!need_update) tc_warp_arrive(X.stg_free(), lane);
    }
  }
  if (out_tma && tid < TC_WORKERS && lane == 0) tc::bulk_wait_all();
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
  TSA_TRACE_EVENT(40, 0);
}

}  // namespace tsa
