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
// index, factor index and weight is a compile-time constant. A feature is
// m * y with y its last input factor and m the run product x_i x_j w shared by
// the features of a run; two features come from one bf16x2 multiply, whose
// packed operands the compiler shares along the run. Features are written as
// bf16, 8 at a time (16 bytes), into the core-matrix tiles read by tcgen05.mma.
#pragma once
#include <cuda_bf16.h>
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

// Feature A as a product m * y of two factors: y is the last input factor of
// the monomial (exact in bf16, the inputs being bf16), m the rest including
// the weight.
template <int DK, int NT, int A>
__device__ __forceinline__ void feat_factors(const float (&x)[DK + 1], float& m, float& y) {
  using FC = FeatConst<DK, NT>;
  if constexpr (A >= FC::D) {
    m = 0.0f; y = 0.0f;
  } else {
    constexpr uint32_t cd = FC::tab.code[A];
    constexpr int i = cd & 255, j = (cd >> 8) & 255, l = (cd >> 16) & 255;
    constexpr float w = FC::tab.w[A];
    if constexpr (i == DK) { m = x[DK]; y = 1.0f; }
    else if constexpr (j == DK) { m = 1.0f; y = x[i]; }
    else if constexpr (l == DK) { m = (w == 1.0f) ? x[i] : x[i] * w; y = x[j]; }
    else { m = (w == 1.0f) ? x[i] * x[j] : (x[i] * x[j]) * w; y = x[l]; }
  }
}

// Two features in one bf16x2 multiply: (m_a, m_b) * (y_a, y_b). The packed
// factor pairs repeat along a run of monomials and are shared by the compiler.
template <int DK, int NT, int A>
__device__ __forceinline__ uint32_t feat2(const float (&x)[DK + 1]) {
  float ma, ya, mb, yb;
  feat_factors<DK, NT, A>(x, ma, ya);
  feat_factors<DK, NT, A + 1>(x, mb, yb);
  const uint32_t m = tc::pack_bf16x2(ma, mb), y = tc::pack_bf16x2(ya, yb);
  const __nv_bfloat162 r = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&m),
                                   *reinterpret_cast<const __nv_bfloat162*>(&y));
  return *reinterpret_cast<const uint32_t*>(&r);
}

template <int DK, int NT, int A>
__device__ __forceinline__ uint4 feat8(const float (&x)[DK + 1]) {
  uint4 r;
  r.x = feat2<DK, NT, A + 0>(x);
  r.y = feat2<DK, NT, A + 2>(x);
  r.z = feat2<DK, NT, A + 4>(x);
  r.w = feat2<DK, NT, A + 6>(x);
  return r;
}

// Write the G groups of 8 features starting at A0 (a multiple of 8) for one
// token into the feature tile of every CTA of the cluster: `local` points at
// the token's row in this CTA's tile (8-feature groups 128 bytes apart), and
// `remote[r]` is the shared::cluster address of the same row in CTA r (used for
// r != R, this CTA's rank).
template <int DK, int NT, int NS, int R, int A0, int G>
struct PhiGroups {
  static __device__ __forceinline__ void run(const float (&x)[DK + 1], uint8_t* local, const uint32_t* remote) {
    PhiGroups<DK, NT, NS, R, A0, G - 1>::run(x, local, remote);
    constexpr int a = A0 + 8 * (G - 1);
    constexpr int grp = (a % 128) / 8;
    const uint4 v = feat8<DK, NT, a>(x);
    *reinterpret_cast<uint4*>(local + grp * 128) = v;
#pragma unroll
    for (int r = 0; r < NS; ++r)
      if (r != R) tc::st_cluster_v4(remote[r] + grp * 128, v);
  }
};
template <int DK, int NT, int NS, int R, int A0>
struct PhiGroups<DK, NT, NS, R, A0, 0> {
  static __device__ __forceinline__ void run(const float (&)[DK + 1], uint8_t*, const uint32_t*) {}
};

// Groups of 8 (of the 16 in a 128-wide tile) that CTA r of a cluster of NS
// builds: [tc_group0(NS, r), tc_group0(NS, r + 1)); each half of the CTA's
// workers takes one part of that range.
__host__ __device__ constexpr int tc_group0(int ns, int r) { return (16 * r + ns - 1) / ns; }
__host__ __device__ constexpr int tc_group_mid(int ns, int r) {
  return tc_group0(ns, r) + (tc_group0(ns, r + 1) - tc_group0(ns, r) + 1) / 2;
}

// This CTA's share of feature block f for one token (runtime f and half pick a
// compile-time instantiation).
template <int DK, int NT, int NS, int R, int F = 0>
__device__ __forceinline__ void build_phi_part(int f, int half, const float (&x)[DK + 1], uint8_t* local,
                                               const uint32_t* remote) {
  if constexpr (F < FeatConst<DK, NT>::NB) {
    if (f == F) {
      constexpr int g0 = tc_group0(NS, R), gm = tc_group_mid(NS, R), g1 = tc_group0(NS, R + 1);
      if (half == 0) PhiGroups<DK, NT, NS, R, F * 128 + 8 * g0, gm - g0>::run(x, local, remote);
      else PhiGroups<DK, NT, NS, R, F * 128 + 8 * gm, g1 - gm>::run(x, local, remote);
      return;
    }
    build_phi_part<DK, NT, NS, R, F + 1>(f, half, x, local, remote);
  }
}

// Runtime rank -> instantiation.
template <int DK, int NT, int NS>
__device__ __forceinline__ void build_phi_rank(int rank, int f, int half, const float (&x)[DK + 1],
                                               uint8_t* local, const uint32_t* remote) {
  if constexpr (NS == 1) {
    build_phi_part<DK, NT, 1, 0>(f, half, x, local, remote);
  } else if constexpr (NS == 2) {
    if (rank == 0) build_phi_part<DK, NT, 2, 0>(f, half, x, local, remote);
    else build_phi_part<DK, NT, 2, 1>(f, half, x, local, remote);
  } else if constexpr (NS == 3) {
    if (rank == 0) build_phi_part<DK, NT, 3, 0>(f, half, x, local, remote);
    else if (rank == 1) build_phi_part<DK, NT, 3, 1>(f, half, x, local, remote);
    else build_phi_part<DK, NT, 3, 2>(f, half, x, local, remote);
  } else {
    static_assert(NS >= 1 && NS <= 4, "cluster size");
    if (rank == 0) build_phi_part<DK, NT, 4, 0>(f, half, x, local, remote);
    else if (rank == 1) build_phi_part<DK, NT, 4, 1>(f, half, x, local, remote);
    else if (rank == 2) build_phi_part<DK, NT, 4, 2>(f, half, x, local, remote);
    else build_phi_part<DK, NT, 4, 3>(f, half, x, local, remote);
  }
}

}  // namespace tsa
