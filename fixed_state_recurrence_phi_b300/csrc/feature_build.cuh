// feature_build.cuh -- compile-time generation of the feature map phi for the
// tensor-core path.
//
// phi(x) = [1 | x_i | x_i x_j / sqrt(a!) | x_i x_j x_l / sqrt(a!)] in the
// canonical order of common.cuh (orders ascending, indices non-decreasing), so
// that <phi_m(q), phi_m(k)> = (q.k)^m / m! (Expanding Attention, arXiv
// 2610.20637 abstract: symmetric tensor-power inner products, the m-th block
// C(d+m-1, m) wide).
//
// One thread owns one token and holds its d inputs in registers; every feature
// index, factor index and weight is a compile-time constant, so each feature
// costs one multiply once the compiler has shared the run products x_i x_j (and
// x_i x_j w) between the features of a run. Features are written as bf16, 8 at
// a time (16 bytes), into the core-matrix tiles read by tcgen05.mma.
#pragma once
#include "common.cuh"
#include "tc_ptx.cuh"

namespace tsa {

template <int DK, int NT>
struct FeatConst {
  static constexpr FeatTab<DK, NT> tab = make_feat_tab<DK, NT>();
  static constexpr int D = feat_dim(DK, NT);
  static constexpr int NB = (D + 127) / 128;   // 128-feature blocks (MMA M = 128)
};

// Feature A of the token with inputs x[0..DK-1]; x[DK] is the value of the
// order-0 feature (1, or 0 for a masked token whose other inputs are 0).
template <int DK, int NT, int A>
__device__ __forceinline__ float feat_value(const float (&x)[DK + 1]) {
  using FC = FeatConst<DK, NT>;
  if constexpr (A >= FC::D) {
    return 0.0f;
  } else {
    constexpr uint32_t cd = FC::tab.code[A];
    constexpr int i = cd & 255, j = (cd >> 8) & 255, l = (cd >> 16) & 255;
    constexpr float w = FC::tab.w[A];
    if constexpr (i == DK) {
      return x[DK];
    } else if constexpr (j == DK) {
      return x[i];
    } else if constexpr (l == DK) {
      if constexpr (w == 1.0f) return x[i] * x[j];
      else return (x[i] * w) * x[j];
    } else {
      if constexpr (w == 1.0f) return (x[i] * x[j]) * x[l];
      else return ((x[i] * x[j]) * w) * x[l];
    }
  }
}

template <int DK, int NT, int A>
__device__ __forceinline__ uint4 feat8(const float (&x)[DK + 1]) {
  uint4 r;
  r.x = tc::pack_bf16x2(feat_value<DK, NT, A + 0>(x), feat_value<DK, NT, A + 1>(x));
  r.y = tc::pack_bf16x2(feat_value<DK, NT, A + 2>(x), feat_value<DK, NT, A + 3>(x));
  r.z = tc::pack_bf16x2(feat_value<DK, NT, A + 4>(x), feat_value<DK, NT, A + 5>(x));
  r.w = tc::pack_bf16x2(feat_value<DK, NT, A + 6>(x), feat_value<DK, NT, A + 7>(x));
  return r;
}

// Write the G groups of 8 features starting at A0 (a multiple of 8) for one
// token. `pq` / `pk` point at the token's row inside a feature tile whose
// 8-feature groups are 128 bytes apart.
template <int DK, int NT, bool WITH_Q, int A0, int G>
struct PhiGroups {
  static __device__ __forceinline__ void run(const float (&xq)[DK + 1], const float (&xk)[DK + 1],
                                             uint8_t* pq, uint8_t* pk) {
    PhiGroups<DK, NT, WITH_Q, A0, G - 1>::run(xq, xk, pq, pk);
    constexpr int a = A0 + 8 * (G - 1);
    constexpr int grp = (a % 128) / 8;
    if constexpr (WITH_Q) *reinterpret_cast<uint4*>(pq + grp * 128) = feat8<DK, NT, a>(xq);
    *reinterpret_cast<uint4*>(pk + grp * 128) = feat8<DK, NT, a>(xk);
  }
};
template <int DK, int NT, bool WITH_Q, int A0>
struct PhiGroups<DK, NT, WITH_Q, A0, 0> {
  static __device__ __forceinline__ void run(const float (&)[DK + 1], const float (&)[DK + 1], uint8_t*,
                                             uint8_t*) {}
};

// Features [128 f + 64 half, +64) of block f for one token (runtime f and half
// select one of the compile-time instantiations).
template <int DK, int NT, bool WITH_Q, int F = 0>
__device__ __forceinline__ void build_phi_half(int f, int half, const float (&xq)[DK + 1],
                                               const float (&xk)[DK + 1], uint8_t* pq, uint8_t* pk) {
  if constexpr (F < FeatConst<DK, NT>::NB) {
    if (f == F) {
      if (half == 0) PhiGroups<DK, NT, WITH_Q, F * 128, 8>::run(xq, xk, pq, pk);
      else PhiGroups<DK, NT, WITH_Q, F * 128 + 64, 8>::run(xq, xk, pq, pk);
      return;
    }
    build_phi_half<DK, NT, WITH_Q, F + 1>(f, half, xq, xk, pq, pk);
  }
}

}  // namespace tsa
