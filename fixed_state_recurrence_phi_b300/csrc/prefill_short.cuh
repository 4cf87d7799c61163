// prefill_short.cuh -- prefill of short segments on the CUDA cores, with the
// head's whole state resident in shared memory.
//
// Appending a few tokens to existing states (Expanding Attention, arXiv
// 2610.20637 abstract: the states are additive across chunks, so a segment
// continues a sequence from the state of everything before it; Hacker News
// thread on the paper: the "+1" column carries the softmax normaliser). The
// segment is taken in blocks of LB = 16 tokens; with S the state of every
// token before the block:
//     num|den = phi(Q_b) S + mask(T_n(Q_b K_b^T)) [V_b, 1]      (j <= i)
//     out     = num / den
//     S      += phi(K_b)^T [V_b, 1]
// One CTA per head keeps S (D_pad x (d_v+1) fp32) in shared memory for the
// whole segment: it is read from HBM once (one bulk copy) and written once,
// by the last block's update, whatever the segment's length. A segment of a
// few tokens therefore costs about one pass over the states, like a decode
// step, rather than the chunked prefill's start-up on a 128-token chunk.
//
// Threads of a block (256):
//   inputs    x_t (with the constant 1.0 after the d_k inputs) and v_t; the
//             next block's are loaded into registers while this one computes
//   features  phi(q_t), phi(k_t) as [row a][token t]; T_n(q_t.k_j), j <= t
//   readout   phi(Q_b) S: each thread streams its feature rows of S once,
//             for all 16 tokens x 4 value columns (accumulated as token pairs);
//             the row groups of a warp are summed by shuffles, the warps'
//             partials in shared memory; den_t = phi(q_t).z per warp
//   output    partial sums + intra-block terms, divided, stored
//   update    S[a][4 columns] += sum_j phi(k_j)[a] v_j, with the thread's
//             values held in registers; z[a] += sum_j phi(k_j)[a]
// The kernel is bound by shared-memory bandwidth, so every element of S is
// read once per block by the readout and once (read and written) by the
// update, with the other operand held in registers.
#pragma once
#include "common.cuh"
#include "tc_ptx.cuh"

namespace tsa {

struct ShortParams {
  const void* q;    // [heads][N][DK]
  const void* k;    // [heads][N][DK]
  const void* v;    // [heads][N][DV]
  void* out;        // [heads][N][DV]
  float* states;    // [heads][DPAD*(DV+1)]
  int* err;         // device error word (set on a timed-out wait)
  long long N;
  int heads;
  int accumulate;
};

template <int DK, int NT, int DV>
struct ShortLayout {
  static constexpr int D = feat_dim(DK, NT);
  static constexpr int DPAD = round_up(D, 4);
  static constexpr int LB = 16;                        // tokens per block
  static constexpr int DKP = DK + 1;                   // x row: d_k inputs, then 1.0
  static constexpr int CG = DV / 4;                    // float4 column groups
  static constexpr int KW = 32 / CG;                   // feature-row groups per warp
  static constexpr int KG = 8 * KW;                    // feature-row groups of the readout
  static constexpr int ST = DPAD * (DV + 1);           // S [DPAD][DV], then z [DPAD]
  static constexpr int o_st = 0;
  static constexpr int o_fq = o_st + ST;                       // [DPAD][LB]
  static constexpr int o_fk = o_fq + DPAD * LB;                // [DPAD][LB]
  static constexpr int o_vv = o_fk + DPAD * LB;                // [LB][DV]
  static constexpr int o_xq = o_vv + LB * DV;                  // [LB][DKP]
  static constexpr int o_xk = o_xq + round_up(LB * DKP, 4);    // [LB][DKP]
  static constexpr int o_a = o_xk + round_up(LB * DKP, 4);     // [LB][LB]
  static constexpr int o_part = o_a + LB * LB;                 // [8 warps][LB][DV]
  static constexpr int o_den = o_part + 8 * LB * DV;           // [8 warps][LB]
  static constexpr int o_fc = o_den + 8 * LB;                  // feature codes [DPAD]
  static constexpr int o_fw = o_fc + DPAD;                     // feature weights [DPAD]
  static constexpr int o_bar = o_fw + DPAD;                    // one mbarrier
  static constexpr int floats = o_bar + 4;
  static constexpr size_t bytes = (size_t)floats * 4;
  // inputs per thread and block
  static constexpr int QPT = (LB * DK + 255) / 256;
  static constexpr int VPT = (LB * CG + 255) / 256;
  static_assert(DV % 4 == 0 && KW >= 1 && KW * CG == 32, "thread split");
  static_assert(LB * LB == 256, "one thread per intra-block pair");
};

// Shared memory of the layout above (host and device agree on it).
__host__ __device__ constexpr size_t short_smem_bytes(int dk, int nt, int dv) {
  const int dpad = round_up(feat_dim(dk, nt), 4);
  const int f = dpad * (dv + 1) + 2 * dpad * 16 + 16 * dv + 2 * round_up(16 * (dk + 1), 4) + 256 +
                8 * 16 * dv + 8 * 16 + 2 * dpad + 4;
  return (size_t)f * 4;
}
// Two CTAs per SM: one loads its state while the other computes.
constexpr size_t kShortSmemMax = 113 * 1024;
__host__ __device__ constexpr bool short_fits(int dk, int nt, int dv) {
  return (dv == 32 || dv == 64 || dv == 128) && short_smem_bytes(dk, nt, dv) <= kShortSmemMax;
}

constexpr uint64_t SHORT_WAIT_NS = 1000000000ull;   // 1 s for the state copy

// d += a * b on both lanes of a pair. Two scalar FMAs: the packed pair FMA
// (__ffma2_rn) measured slower in this kernel (71.7 against 63.6 us for 32
// tokens on 1,024 heads).
__device__ __forceinline__ void fma_pair(float2& d, float2 a, float2 b) {
  d.x = fmaf(a.x, b.x, d.x);
  d.y = fmaf(a.y, b.y, d.y);
}

template <typename T, int DK, int NT, int DV>
__global__ void __launch_bounds__(256, 2)
short_prefill_kernel(ShortParams p) {
  using L = ShortLayout<DK, NT, DV>;
  constexpr int D = L::D, DPAD = L::DPAD, LB = L::LB, DKP = L::DKP, CG = L::CG, KW = L::KW,
                KG = L::KG, QPT = L::QPT, VPT = L::VPT;
  static_assert(L::bytes == short_smem_bytes(DK, NT, DV), "layout size");
  static_assert(NT <= 4, "three-factor features (orders 0..3)");
  extern __shared__ __align__(16) float sm[];
  float* st = sm + L::o_st;
  float* z = st + DPAD * DV;
  float* fq = sm + L::o_fq;
  float* fk = sm + L::o_fk;
  float* vv = sm + L::o_vv;
  float* xq = sm + L::o_xq;
  float* xk = sm + L::o_xk;
  float* As = sm + L::o_a;
  float* part = sm + L::o_part;
  float* denp = sm + L::o_den;
  uint32_t* fc = reinterpret_cast<uint32_t*>(sm + L::o_fc);
  float* fw = sm + L::o_fw;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::o_bar);
  __shared__ int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int head = blockIdx.x;
  if (head >= p.heads || p.N <= 0) return;
  float* gst = p.states + (size_t)head * L::ST;
  const T* qg = static_cast<const T*>(p.q) + (size_t)head * p.N * DK;
  const T* kg = static_cast<const T*>(p.k) + (size_t)head * p.N * DK;
  const T* vg = static_cast<const T*>(p.v) + (size_t)head * p.N * DV;
  T* og = static_cast<T*>(p.out) + (size_t)head * p.N * DV;

  // the state before the segment: one bulk copy, in flight while the first
  // block's inputs and features are built; or zero
  if (tid == 0) {
    s_abort = 0;
    if (p.accumulate) {
      tc::mbar_init(bar, 1);
      tc::mbar_fence_init();
      tc::mbar_arrive_expect_tx(bar, (uint32_t)(L::ST * 4));
      tc::bulk_load(st, gst, (uint32_t)(L::ST * 4), bar);
    }
  }
  if (!p.accumulate) {
    float4* s4 = reinterpret_cast<float4*>(st);
    for (int e = tid; e < L::ST / 4; e += 256) s4[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int a = tid; a < DPAD; a += 256) {
    fc[a] = a < D ? __ldg(&g_feat<DK, NT>.code[a]) : 0u;
    fw[a] = a < D ? __ldg(&g_feat<DK, NT>.w[a]) : 0.f;
  }
  if (tid < LB) { xq[tid * DKP + DK] = 1.f; xk[tid * DKP + DK] = 1.f; }

  // one block's inputs, held in registers between their load and their store
  float rq[QPT], rk[QPT];
  float4 rv[VPT];
  auto load_in = [&](int b) {
    const long long t0 = (long long)b * LB;
#pragma unroll
    for (int i = 0; i < QPT; ++i) {
      const int e = tid + 256 * i, t = e / DK, ii = e % DK;
      rq[i] = rk[i] = 0.f;
      if (e < LB * DK && t0 + t < p.N) {
        rq[i] = Elem<T>::load1(qg + (t0 + t) * DK + ii);
        rk[i] = Elem<T>::load1(kg + (t0 + t) * DK + ii);
      }
    }
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int e = tid + 256 * i, t = e / CG, c4 = e % CG;
      rv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < LB * CG && t0 + t < p.N) rv[i] = Elem<T>::load4(vg + (t0 + t) * DV + 4 * c4);
    }
  };
  auto store_in = [&]() {
#pragma unroll
    for (int i = 0; i < QPT; ++i) {
      const int e = tid + 256 * i, t = e / DK, ii = e % DK;
      if (e < LB * DK) { xq[t * DKP + ii] = rq[i]; xk[t * DKP + ii] = rk[i]; }
    }
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int e = tid + 256 * i, t = e / CG, c4 = e % CG;
      if (e < LB * CG) *reinterpret_cast<float4*>(vv + t * DV + 4 * c4) = rv[i];
    }
  };
  load_in(0);
  store_in();

  const int nblk = (int)((p.N + LB - 1) / LB);
  for (int b = 0; b < nblk; ++b) {
    const long long t0 = (long long)b * LB;
    const int nb = (int)((p.N - t0) < LB ? (p.N - t0) : LB);
    __syncthreads();                       // this block's inputs are in place
    if (b + 1 < nblk) load_in(b + 1);      // in flight until the block ends

    // features [a][t] (phi(k_t) zero for tokens past the end, so that they
    // add nothing to the state) and the intra-block kernel values
    for (int e = tid; e < DPAD * LB; e += 256) {
      const int a = e / LB, t = e % LB;
      const uint32_t cd = fc[a];
      const int i = cd & 255, j = (cd >> 8) & 255, l = (cd >> 16) & 255;
      const float w = fw[a];
      const float* x1 = xq + t * DKP;
      const float* x2 = xk + t * DKP;
      const float f1 = w * x1[i] * x1[j] * x1[l];
      const float f2 = (t < nb) ? w * x2[i] * x2[j] * x2[l] : 0.f;
      fq[e] = f1;
      fk[e] = f2;
    }
    {
      const int t = tid / LB, j = tid % LB;
      float x = 0.f;
#pragma unroll
      for (int i = 0; i < DK; ++i) x = fmaf(xq[t * DKP + i], xk[j * DKP + i], x);
      As[t * LB + j] = (j <= t && j < nb) ? taylor_T<NT>(x) : 0.f;
    }
    if (b == 0 && p.accumulate && tid == 0) s_abort = tc::mbar_wait(bar, 0, SHORT_WAIT_NS) ? 0 : 1;
    __syncthreads();
    if (s_abort) {
      if (tid == 0) atomicExch(p.err, 3);
      return;
    }

    // den_t = phi(q_t).z: warp w takes the rows a = w, w + 8, ... for all
    // tokens (lane: token lane & 15, row half lane >> 4)
    {
      const int t = lane & 15, h = lane >> 4;
      float d = 0.f;
      for (int a = 2 * warp + h; a < DPAD; a += 16) d = fmaf(fq[a * LB + t], z[a], d);
      d += __shfl_xor_sync(0xffffffffu, d, 16);
      if (h == 0) denp[warp * LB + t] = d;
    }
    // phi(Q_b) S: lane (kq, cg) of warp w takes the feature rows
    // a = KW*w + kq + KG*i, all tokens, columns 4*cg..; ap[p][c] holds tokens
    // (2p, 2p+1) of column c
    {
      const int cg = lane % CG, kq = lane / CG;
      float2 ap[LB / 2][4];
#pragma unroll
      for (int pq = 0; pq < LB / 2; ++pq)
#pragma unroll
        for (int c = 0; c < 4; ++c) ap[pq][c] = make_float2(0.f, 0.f);
#pragma unroll 2
      for (int a = KW * warp + kq; a < DPAD; a += KG) {
        const float4 s = *reinterpret_cast<const float4*>(st + a * DV + 4 * cg);
        const float2 sd[4] = {make_float2(s.x, s.x), make_float2(s.y, s.y), make_float2(s.z, s.z),
                              make_float2(s.w, s.w)};
        const float4* f4 = reinterpret_cast<const float4*>(fq + a * LB);
#pragma unroll
        for (int qq = 0; qq < LB / 4; ++qq) {
          const float4 f = f4[qq];
          const float2 fa = make_float2(f.x, f.y), fb = make_float2(f.z, f.w);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            fma_pair(ap[2 * qq][c], fa, sd[c]);
            fma_pair(ap[2 * qq + 1][c], fb, sd[c]);
          }
        }
      }
      // sum the KW row groups of the warp by recursive halving of the token
      // pairs: afterwards this lane holds pairs base .. base + LB/2/KW - 1
      int base = 0;
#pragma unroll
      for (int m = CG, np = LB / 2; m < 32; m *= 2, np /= 2) {
        const bool hi = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < np / 2; ++i)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float2 keep = hi ? ap[i + np / 2][c] : ap[i][c];
            const float2 send = hi ? ap[i][c] : ap[i + np / 2][c];
            const float rx = __shfl_xor_sync(0xffffffffu, send.x, m);
            const float ry = __shfl_xor_sync(0xffffffffu, send.y, m);
            ap[i][c] = make_float2(keep.x + rx, keep.y + ry);
          }
        base += hi ? np / 2 : 0;
      }
      float* pw = part + warp * LB * DV + 4 * cg;
#pragma unroll
      for (int i = 0; i < LB / 2 / KW; ++i) {
        const int t = 2 * (base + i);
        *reinterpret_cast<float4*>(pw + t * DV) =
            make_float4(ap[i][0].x, ap[i][1].x, ap[i][2].x, ap[i][3].x);
        *reinterpret_cast<float4*>(pw + (t + 1) * DV) =
            make_float4(ap[i][0].y, ap[i][1].y, ap[i][2].y, ap[i][3].y);
      }
    }
    __syncthreads();

    // outputs: readout partials + intra-block terms, normalised
    for (int e = tid; e < LB * CG; e += 256) {
      const int t = e / CG, cg = e % CG;
      float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float4 x = *reinterpret_cast<const float4*>(part + (w * LB + t) * DV + 4 * cg);
        num.x += x.x; num.y += x.y; num.z += x.z; num.w += x.w;
      }
      float dn = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) dn += denp[w * LB + t];
      for (int j = 0; j <= t; ++j) {
        const float a = As[t * LB + j];
        const float4 x = *reinterpret_cast<const float4*>(vv + j * DV + 4 * cg);
        num.x = fmaf(a, x.x, num.x); num.y = fmaf(a, x.y, num.y);
        num.z = fmaf(a, x.z, num.z); num.w = fmaf(a, x.w, num.w);
        dn += a;
      }
      if (t < nb) {
        const float r = 1.0f / dn;
        Elem<T>::store4(og + (t0 + t) * DV + 4 * cg,
                        make_float4(num.x * r, num.y * r, num.z * r, num.w * r));
      }
    }
    // state update; the last block writes the final state to HBM
    {
      const bool last = (b == nblk - 1);
      const int cg = tid % CG, r0 = tid / CG;
      constexpr int RS = 256 / CG;
      // the thread's values of the block's tokens, held in registers
      float4 vr[LB];
#pragma unroll
      for (int j = 0; j < LB; ++j) vr[j] = *reinterpret_cast<const float4*>(vv + j * DV + 4 * cg);
      // two copies of the row loop, so that each stores to a known address
      // space (a store through a generic pointer could alias the next row's
      // shared-memory loads and would be ordered before them); two rows in
      // flight per thread
      auto rows = [&](float* dS, float* dz) {
#pragma unroll 2
        for (int a = r0; a < DPAD; a += RS) {
          float4 s = *reinterpret_cast<const float4*>(st + a * DV + 4 * cg);
          const float4* f4 = reinterpret_cast<const float4*>(fk + a * LB);
#pragma unroll
          for (int jj = 0; jj < LB / 4; ++jj) {
            const float4 f = f4[jj];
            const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float4 x = vr[4 * jj + u];
              s.x = fmaf(fv[u], x.x, s.x); s.y = fmaf(fv[u], x.y, s.y);
              s.z = fmaf(fv[u], x.z, s.z); s.w = fmaf(fv[u], x.w, s.w);
            }
          }
          *reinterpret_cast<float4*>(dS + a * DV + 4 * cg) = s;
        }
        for (int a = tid; a < DPAD; a += 256) {
          const float4* f4 = reinterpret_cast<const float4*>(fk + a * LB);
          float zz = z[a];
#pragma unroll
          for (int jj = 0; jj < LB / 4; ++jj) {
            const float4 f = f4[jj];
            zz += (f.x + f.y) + (f.z + f.w);
          }
          dz[a] = zz;
        }
      };
      if (last) rows(gst, gst + DPAD * DV);
      else rows(st, z);
    }
    __syncthreads();                       // block b's reads of x, v are done
    if (b + 1 < nblk) store_in();
  }
}

}  // namespace tsa
