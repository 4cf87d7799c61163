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
  static_assert(NT <= 4, "the tensor-core feature builders read three factors (orders 0..3)");
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

// ---- the same features from the packed bf16 inputs ---------------------------
// A token's inputs as they arrive, two bf16 per 32-bit word: xp[e] holds
// x[2e] (low half) and x[2e + 1] (high half); x0 is the value of the order-0
// feature (1, or 0 for a masked token). Only these words live in registers:
// an input's fp32 value is one shift or mask of its word, and the bf16 pair of
// two inputs one byte permutation of their words, so a feature pair costs the
// multiplier pair's conversion (shared along a run of monomials that differ
// only in their last index), at most one permutation and one bf16x2
// multiply. Results are bitwise equal to feat2: the multiplier is still
// formed in fp32 and rounded once, and the pair holds the same bf16 inputs.

template <int I>
__device__ __forceinline__ float in_f32(const uint32_t* xp) {
  return __uint_as_float((I % 2) ? (xp[I / 2] & 0xFFFF0000u) : (xp[I / 2] << 16));
}

// Index of the last input factor of feature A (-1: the order-0 feature, or
// past the end) and whether its multiplier is exactly 1 (order 1).
template <int DK, int NT, int A>
struct FeatY {
  using FC = FeatConst<DK, NT>;
  static constexpr bool live = A < FC::D;
  static constexpr uint32_t cd = live ? FC::tab.code[A] : 0u;
  static constexpr int i = cd & 255, j = (cd >> 8) & 255, l = (cd >> 16) & 255;
  static constexpr int y = (!live || i == DK) ? -1 : (j == DK ? i : (l == DK ? j : l));
  static constexpr bool unit_m = live && i != DK && j == DK;
};

// Multiplier m of feature A (the monomial without its last input factor, with
// the weight), in fp32.
template <int DK, int NT, int A>
__device__ __forceinline__ float feat_m(const uint32_t* xp, float x0) {
  using Y = FeatY<DK, NT, A>;
  if constexpr (!Y::live) {
    return 0.0f;
  } else {
    constexpr float w = FeatConst<DK, NT>::tab.w[A];
    if constexpr (Y::i == DK) return x0;
    else if constexpr (Y::j == DK) return 1.0f;
    else if constexpr (Y::l == DK) return (w == 1.0f) ? in_f32<Y::i>(xp) : in_f32<Y::i>(xp) * w;
    else if constexpr (w == 1.0f) return in_f32<Y::i>(xp) * in_f32<Y::j>(xp);
    else return (in_f32<Y::i>(xp) * in_f32<Y::j>(xp)) * w;
  }
}

// The bf16 pair (y_a, y_b) of the last input factors (y = -1: the value 1).
template <int YA, int YB>
__device__ __forceinline__ uint32_t in_pair(const uint32_t* xp) {
  if constexpr (YA >= 0 && YB == YA + 1 && YA % 2 == 0) {
    return xp[YA / 2];
  } else if constexpr (YA >= 0 && YB >= 0) {
    constexpr uint32_t sel = ((YB % 2) ? 0x7600u : 0x5400u) | ((YA % 2) ? 0x32u : 0x10u);
    return __byte_perm(xp[YA / 2], xp[YB / 2], sel);
  } else {
    const uint32_t lo = (YA >= 0) ? (((YA % 2) ? (xp[YA / 2] >> 16) : xp[YA / 2]) & 0xFFFFu) : 0x3F80u;
    const uint32_t hi = (YB >= 0) ? (((YB % 2) ? (xp[YB / 2] >> 16) : xp[YB / 2]) & 0xFFFFu) : 0x3F80u;
    return lo | (hi << 16);
  }
}

template <int DK, int NT, int A>
__device__ __forceinline__ uint32_t feat2p(const uint32_t* xp, float x0) {
  using Ya = FeatY<DK, NT, A>;
  using Yb = FeatY<DK, NT, A + 1>;
  if constexpr (!Ya::live) {
    return 0u;
  } else if constexpr (Ya::unit_m && (Yb::unit_m || !Yb::live)) {
    // order 1: the inputs themselves
    return Yb::live ? in_pair<Ya::y, Yb::y>(xp) : (in_pair<Ya::y, Ya::y>(xp) & 0xFFFFu);
  } else {
    const uint32_t m = tc::pack_bf16x2(feat_m<DK, NT, A>(xp, x0), feat_m<DK, NT, A + 1>(xp, x0));
    const uint32_t y = in_pair<Ya::y, (Yb::live ? Yb::y : -1)>(xp);
    const __nv_bfloat162 r = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&m),
                                     *reinterpret_cast<const __nv_bfloat162*>(&y));
    return *reinterpret_cast<const uint32_t*>(&r);
  }
}

template <int DK, int NT, int A>
__device__ __forceinline__ uint4 feat8p(const uint32_t* xp, float x0) {
  uint4 r;
  r.x = feat2p<DK, NT, A + 0>(xp, x0);
  r.y = feat2p<DK, NT, A + 2>(xp, x0);
  r.z = feat2p<DK, NT, A + 4>(xp, x0);
  r.w = feat2p<DK, NT, A + 6>(xp, x0);
  return r;
}

// Write the G groups of 8 features starting at A0 (a multiple of 8) for one
// token into its row of the feature tile: `row` points at the token's row,
// 8-feature groups 128 bytes apart.
template <int DK, int NT, int A0, int G>
struct PhiGroups {
  static __device__ __forceinline__ void run(const float (&x)[DK + 1], uint8_t* row) {
    PhiGroups<DK, NT, A0, G - 1>::run(x, row);
    constexpr int a = A0 + 8 * (G - 1);
    constexpr int grp = (a % 128) / 8;
    *reinterpret_cast<uint4*>(row + grp * 128) = feat8<DK, NT, a>(x);
  }
};
template <int DK, int NT, int A0>
struct PhiGroups<DK, NT, A0, 0> {
  static __device__ __forceinline__ void run(const float (&)[DK + 1], uint8_t*) {}
};

// Half `half` (groups 8*half .. 8*half + 7) of feature block f for one token;
// the runtime block index picks a compile-time instantiation (one call site
// per kernel keeps one copy of the feature code).
template <int DK, int NT, int F = 0>
__device__ __forceinline__ void build_phi_half(int f, int half, const float (&x)[DK + 1], uint8_t* row) {
  if constexpr (F < FeatConst<DK, NT>::NB) {
    if (f == F) {
      if (half == 0) PhiGroups<DK, NT, F * 128, 8>::run(x, row);
      else PhiGroups<DK, NT, F * 128 + 64, 8>::run(x, row);
      return;
    }
    build_phi_half<DK, NT, F + 1>(f, half, x, row);
  }
}

// Quarter `qtr` (groups 4*qtr .. 4*qtr + 3) of feature block f for one token.
template <int DK, int NT, int F = 0>
__device__ __forceinline__ void build_phi_quarter(int f, int qtr, const float (&x)[DK + 1], uint8_t* row) {
  if constexpr (F < FeatConst<DK, NT>::NB) {
    if (f == F) {
      switch (qtr) {
        case 0: PhiGroups<DK, NT, F * 128, 4>::run(x, row); break;
        case 1: PhiGroups<DK, NT, F * 128 + 32, 4>::run(x, row); break;
        case 2: PhiGroups<DK, NT, F * 128 + 64, 4>::run(x, row); break;
        default: PhiGroups<DK, NT, F * 128 + 96, 4>::run(x, row); break;
      }
      return;
    }
    build_phi_quarter<DK, NT, F + 1>(f, qtr, x, row);
  }
}

}  // namespace tsa
