// common.cuh -- compile-time feature tables and small device helpers shared by
// the libtsa kernels.
//
// Feature map (Expanding Attention, arXiv 2610.20637 abstract: each Taylor term
// (q.k)^m/m! is an inner product of tensor powers; the m-th state is
// C(d+m-1, m) wide): features are the monomials x^a with |a| = m < n, indices
// non-decreasing, orders concatenated in ascending m, each scaled by
// 1/sqrt(a!) so that <phi_m(q), phi_m(k)> = (q.k)^m / m!.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace tsa {

__host__ __device__ constexpr int binom(int n, int k) {
  if (k < 0 || k > n) return 0;
  long long r = 1;
  for (int i = 1; i <= k; ++i) r = r * (n - k + i) / i;
  return (int)r;
}

__host__ __device__ constexpr int feat_dim(int dk, int nt) {
  int s = 0;
  for (int m = 0; m < nt; ++m) s += binom(dk + m - 1, m);
  return s;
}

__host__ __device__ constexpr int round_up(int x, int m) { return (x + m - 1) / m * m; }

// 1/sqrt(a!) for the multi-index factorials that occur up to degree 4
// (a! = 1, 2, 6, 24 for one repeated index, 2 * 2 = 4 for two pairs).
constexpr float kInvSqrt2 = 0.70710678118654752440f;   // a! = 2
constexpr float kInvSqrt6 = 0.40824829046386301637f;   // a! = 6
constexpr float kInvSqrt24 = 0.20412414523193150818f;  // a! = 24

__host__ __device__ constexpr float inv_sqrt_factorial(int f) {
  return f == 1 ? 1.0f : f == 2 ? kInvSqrt2 : f == 4 ? 0.5f : f == 6 ? kInvSqrt6 : kInvSqrt24;
}

// The most orders any table is built for (degree NT - 1 <= 4).
constexpr int kMaxTerms = 5;

// One entry per feature: four factor indices packed in bytes 0..3; the index
// DK names the constant 1.0 stored after the d_k inputs, so an order-m feature
// is  w * x[i] * x[j] * x[l] * x[m']  with (4 - m) of the indices equal to DK.
// Up to order 3 byte 3 is always DK, so kernels built for NT <= 4 read three
// factors only.
template <int DK, int NT>
struct FeatTab {
  static constexpr int D = feat_dim(DK, NT);
  uint32_t code[D];
  float w[D];
};

template <int DK, int NT>
constexpr FeatTab<DK, NT> make_feat_tab() {
  static_assert(NT >= 1 && NT <= kMaxTerms, "orders 0..4 supported");
  FeatTab<DK, NT> t{};
  int a = 0;
  const uint32_t one = (uint32_t)DK;
  // a multi-index given by non-decreasing factor indices (DK = no factor)
  auto put = [&](uint32_t i, uint32_t j, uint32_t l, uint32_t m) {
    t.code[a] = i | (j << 8) | (l << 16) | (m << 24);
    // a! from the run lengths of the real indices
    const uint32_t f[4] = {i, j, l, m};
    int fact = 1, run = 1;
    for (int u = 1; u < 4; ++u) {
      if (f[u] != one && f[u] == f[u - 1]) {
        ++run;
        fact *= run;
      } else {
        run = 1;
      }
    }
    t.w[a] = inv_sqrt_factorial(fact);
    ++a;
  };
  put(one, one, one, one);
  if (NT > 1)
    for (int i = 0; i < DK; ++i) put((uint32_t)i, one, one, one);
  if (NT > 2)
    for (int i = 0; i < DK; ++i)
      for (int j = i; j < DK; ++j) put((uint32_t)i, (uint32_t)j, one, one);
  if (NT > 3)
    for (int i = 0; i < DK; ++i)
      for (int j = i; j < DK; ++j)
        for (int l = j; l < DK; ++l) put((uint32_t)i, (uint32_t)j, (uint32_t)l, one);
  if (NT > 4)
    for (int i = 0; i < DK; ++i)
      for (int j = i; j < DK; ++j)
        for (int l = j; l < DK; ++l)
          for (int m = l; m < DK; ++m) put((uint32_t)i, (uint32_t)j, (uint32_t)l, (uint32_t)m);
  return t;
}

// The table of each (d_k, n) lives in constant memory, built at compile time.
template <int DK, int NT>
__constant__ FeatTab<DK, NT> c_feat = make_feat_tab<DK, NT>();
// The same table in global memory, for reads where every thread of a warp
// takes a different entry (coalesced through L1 rather than serialised by
// the constant cache).
template <int DK, int NT>
__device__ const FeatTab<DK, NT> g_feat = make_feat_tab<DK, NT>();

// Truncated exponential T_n(x) = sum_{m<n} x^m/m!, evaluated in Horner form
// 1 + x(1 + x/2(1 + x/3(...))).
template <int NT>
__device__ __forceinline__ float taylor_T(float x) {
  float p = 1.0f;
#pragma unroll
  for (int m = NT - 1; m >= 1; --m) p = fmaf(x * (1.0f / (float)m), p, 1.0f);
  return p;
}

// ---- element access for fp32 / bf16 tensors -------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float4 load4(const float* p) {
    return *reinterpret_cast<const float4*>(p);
  }
  static __device__ __forceinline__ float2 load2(const float* p) {
    return *reinterpret_cast<const float2*>(p);
  }
  static __device__ __forceinline__ float load1(const float* p) { return *p; }
  static __device__ __forceinline__ void store4(float* p, float4 v) {
    *reinterpret_cast<float4*>(p) = v;
  }
  static __device__ __forceinline__ void store2(float* p, float2 v) {
    *reinterpret_cast<float2*>(p) = v;
  }
  static __device__ __forceinline__ void store1(float* p, float v) { *p = v; }
};
template <> struct Elem<__nv_bfloat16> {
  using bf = __nv_bfloat16;
  static __device__ __forceinline__ float4 load4(const bf* p) {
    uint2 u = *reinterpret_cast<const uint2*>(p);
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&u.x);
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&u.y);
    float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    return make_float4(fa.x, fa.y, fb.x, fb.y);
  }
  static __device__ __forceinline__ float2 load2(const bf* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
  }
  static __device__ __forceinline__ float load1(const bf* p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ void store4(bf* p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
  }
  static __device__ __forceinline__ void store2(bf* p, float2 v) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
  }
  static __device__ __forceinline__ void store1(bf* p, float v) { *p = __float2bfloat16_rn(v); }
};

}  // namespace tsa
