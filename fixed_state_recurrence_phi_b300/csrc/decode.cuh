// decode.cuh -- one-token decode, state merge and state layout conversion.
//
// Decode (Expanding Attention, arXiv 2610.20637 abstract: each state is
// updated by one rank-one outer product per token, so per-token decoding cost
// does not depend on the context length; Hacker News thread: the "+1" column
// is the softmax normaliser). Per head:
//     S' = S + phi(k) [v; 1]^T ;   out = (phi(q)^T S')[:d_v] / (phi(q)^T S')[d_v]
// The step is bound by streaming the state once: each element is read, updated
// with the rank-one term and written back in the same pass, and the readout
// dot products are accumulated from the updated values held in registers.
#pragma once
#include "common.cuh"

namespace tsa {

struct DecodeParams {
  const void* q;   // [heads][DK]
  const void* k;   // [heads][DK]
  const void* v;   // [heads][DV]
  void* out;       // [heads][DV]
  float* states;   // [heads][DPAD*(DV+1)]
  int heads;
};

// One CTA (256 threads) per head. The S part [DPAD][DV] is walked as float4
// column groups: thread t owns column group cg = t % (DV/4) and rows
// r0 + RP*it, so its partial sums always belong to the same 4 columns.
// Small states (up to 160 x 64): 8 CTAs per SM (32 registers a thread), so
// that a batch of 1024 heads is one wave on 148 SMs; larger states keep the
// registers their longer walk needs.
__host__ __device__ constexpr int decode_min_ctas(int dk, int nt, int dv) {
  return round_up(feat_dim(dk, nt), 4) * dv <= 160 * 64 ? 8 : 1;
}
template <typename T, int DK, int NT, int DV>
__global__ void __launch_bounds__(256, decode_min_ctas(DK, NT, DV))
decode_kernel(DecodeParams p) {
  constexpr int D = feat_dim(DK, NT);
  constexpr int DPAD = round_up(D, 4);
  constexpr int CG = DV / 4;          // float4 column groups per row
  constexpr int RP = 256 / CG;        // rows per pass
  constexpr int NIT = (DPAD + RP - 1) / RP;
  constexpr int U0 = NIT < 4 ? NIT : 4;          // rows requested at entry
  constexpr int UNR = (NIT - U0) < 8 ? ((NIT - U0) > 0 ? NIT - U0 : 1) : 8;   // then per batch
  constexpr int NW = 8;
  static_assert(256 % CG == 0, "DV/4 must divide 256");

  __shared__ __align__(16) float vv[DV];
  __shared__ float xq[DK + 1], xk[DK + 1];
  __shared__ __align__(16) float phq[DPAD];
  __shared__ __align__(16) float phk[DPAD];
  __shared__ float red[NW][DV];
  __shared__ float redz[NW];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int head = blockIdx.x;
  if (head >= p.heads) return;

  const T* qg = static_cast<const T*>(p.q) + (size_t)head * DK;
  const T* kg = static_cast<const T*>(p.k) + (size_t)head * DK;
  const T* vg = static_cast<const T*>(p.v) + (size_t)head * DV;
  float* st = p.states + (size_t)head * DPAD * (DV + 1);
  const int cg = tid % CG, r0 = tid / CG;
  float4* S4 = reinterpret_cast<float4*>(st);

  // The first U0 state rows of this thread are requested before anything
  // else: they do not depend on the feature maps, so the state stream starts
  // at once and the feature maps are built while it is in flight.
  float4 s0[U0];
#pragma unroll
  for (int u = 0; u < U0; ++u) {
    const int a = r0 + RP * u;
    if (u < NIT && a < DPAD) s0[u] = S4[(size_t)a * CG + cg];
  }

  if (tid < DK) { xq[tid] = Elem<T>::load1(qg + tid); xk[tid] = Elem<T>::load1(kg + tid); }
  if (tid == 0) { xq[DK] = 1.0f; xk[DK] = 1.0f; }
  if (tid < DV) vv[tid] = Elem<T>::load1(vg + tid);
  __syncthreads();
  for (int a = tid; a < DPAD; a += 256) {
    float fq = 0.f, fk = 0.f;
    if (a < D) {
      const uint32_t cd = __ldg(&g_feat<DK, NT>.code[a]);
      const int i = cd & 255, j = (cd >> 8) & 255, l = (cd >> 16) & 255;
      const float w = __ldg(&g_feat<DK, NT>.w[a]);
      fq = w * xq[i] * xq[j] * xq[l];
      fk = w * xk[i] * xk[j] * xk[l];
      if constexpr (NT > 4) {
        const int m = cd >> 24;
        fq *= xq[m];
        fk *= xk[m];
      }
    }
    phq[a] = fq; phk[a] = fk;
  }
  __syncthreads();

  const float4 v4 = *reinterpret_cast<const float4*>(vv + cg * 4);
  float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
  // S += phi(k) [v]^T row by row, partial phi(q)^T S on the way
  auto row = [&](int a, float4 x) {
    const float fk = phk[a], fq = phq[a];
    x.x = fmaf(fk, v4.x, x.x); x.y = fmaf(fk, v4.y, x.y);
    x.z = fmaf(fk, v4.z, x.z); x.w = fmaf(fk, v4.w, x.w);
    part.x = fmaf(fq, x.x, part.x); part.y = fmaf(fq, x.y, part.y);
    part.z = fmaf(fq, x.z, part.z); part.w = fmaf(fq, x.w, part.w);
    S4[(size_t)a * CG + cg] = x;
  };
#pragma unroll
  for (int u = 0; u < U0; ++u) {
    const int a = r0 + RP * u;
    if (u < NIT && a < DPAD) row(a, s0[u]);
  }
  for (int it0 = U0; it0 < NIT; it0 += UNR) {
    float4 s[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int a = r0 + RP * (it0 + u);
      if (it0 + u < NIT && a < DPAD) s[u] = S4[(size_t)a * CG + cg];
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int a = r0 + RP * (it0 + u);
      if (it0 + u < NIT && a < DPAD) row(a, s[u]);
    }
  }
  // normaliser column z (DPAD floats after the S part)
  float pz = 0.f;
  {
    float4* z4 = reinterpret_cast<float4*>(st + (size_t)DPAD * DV);
    for (int e = tid; e < DPAD / 4; e += 256) {
      float4 x = z4[e];
      const float4 fk = *reinterpret_cast<const float4*>(phk + 4 * e);
      const float4 fq = *reinterpret_cast<const float4*>(phq + 4 * e);
      x.x += fk.x; x.y += fk.y; x.z += fk.z; x.w += fk.w;
      pz = fmaf(fq.x, x.x, pz); pz = fmaf(fq.y, x.y, pz);
      pz = fmaf(fq.z, x.z, pz); pz = fmaf(fq.w, x.w, pz);
      z4[e] = x;
    }
  }
  // reduce partials: lanes sharing cg within the warp, then across warps
#pragma unroll
  for (int off = 16; off >= CG; off >>= 1) {
    part.x += __shfl_xor_sync(0xffffffffu, part.x, off);
    part.y += __shfl_xor_sync(0xffffffffu, part.y, off);
    part.z += __shfl_xor_sync(0xffffffffu, part.z, off);
    part.w += __shfl_xor_sync(0xffffffffu, part.w, off);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) pz += __shfl_xor_sync(0xffffffffu, pz, off);
  if (CG >= 32 || lane < CG) {
    const int c = (CG >= 32) ? tid % CG : lane;
    red[warp][c * 4 + 0] = part.x; red[warp][c * 4 + 1] = part.y;
    red[warp][c * 4 + 2] = part.z; red[warp][c * 4 + 3] = part.w;
  }
  if (lane == 0) redz[warp] = pz;
  __syncthreads();
  if (tid < DV) {
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) { num += red[w][tid]; den += redz[w]; }
    Elem<T>::store1(static_cast<T*>(p.out) + (size_t)head * DV + tid, num / den);
  }
}

// a += b, float4 grid-stride.
__global__ void __launch_bounds__(256)
state_merge_kernel(float4* __restrict__ a, const float4* __restrict__ b, size_t n4) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    float4 x = a[i];
    const float4 y = b[i];
    x.x += y.x; x.y += y.y; x.z += y.z; x.w += y.w;
    a[i] = x;
  }
}

// dst[h][a][c] (c <= dv, column dv = z) from the padded per-head layout.
__global__ void __launch_bounds__(256)
state_canonical_kernel(const float* __restrict__ st, float* __restrict__ dst, int heads, int D,
                       int dpad, int dv) {
  const size_t total = (size_t)heads * D * (dv + 1);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % (dv + 1));
    const size_t r = i / (dv + 1);
    const int a = (int)(r % D);
    const size_t h = r / D;
    const float* hs = st + h * (size_t)dpad * (dv + 1);
    dst[i] = (c < dv) ? hs[(size_t)a * dv + c] : hs[(size_t)dpad * dv + a];
  }
}

}  // namespace tsa
