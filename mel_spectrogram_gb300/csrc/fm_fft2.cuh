// Register DFTs on two independent transforms at once (sm_100+ packed f32x2).
//
// A cx2 holds one complex value of each of two frames in structure-of-arrays
// form: re = (re_a, re_b), im = (im_a, im_b). Every butterfly, twiddle and
// power step is then one packed add/mul/fma for both frames, which halves the
// instruction count of the transform. Multiplication by -i or +i folds into
// the add that follows it (a +- i b swaps the roles of re and im), so no
// component swap is ever materialised.
#pragma once

#include <cuda_runtime.h>

#include "fm_fft.cuh"

namespace fm {

struct cx2 {
  float2 re, im;
};

__device__ __forceinline__ float2 dup(float s) { return make_float2(s, s); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
// a - b as one packed subtraction (sub.rn.f32x2): PTX has no packed negation, so
// adding a negated pair would cost two scalar sign flips first
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;"
      : "=l"(r)
      : "l"(*reinterpret_cast<const unsigned long long*>(&a)), "l"(*reinterpret_cast<const unsigned long long*>(&b)));
  return *reinterpret_cast<const float2*>(&r);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

__device__ __forceinline__ cx2 cadd(cx2 a, cx2 b) { return {add2(a.re, b.re), add2(a.im, b.im)}; }
__device__ __forceinline__ cx2 csub(cx2 a, cx2 b) { return {sub2(a.re, b.re), sub2(a.im, b.im)}; }
__device__ __forceinline__ cx2 cscale(cx2 a, float2 s) { return {mul2(a.re, s), mul2(a.im, s)}; }
// a - i b and a + i b
__device__ __forceinline__ cx2 add_mi(cx2 a, cx2 b) { return {add2(a.re, b.im), sub2(a.im, b.re)}; }
__device__ __forceinline__ cx2 add_pi(cx2 a, cx2 b) { return {sub2(a.re, b.im), add2(a.im, b.re)}; }
// v * w for w = c + i d given as (c, c) and (d, d)
__device__ __forceinline__ cx2 cmul(cx2 v, float2 c, float2 d) {
  return {fma2(v.im, make_float2(-d.x, -d.y), mul2(v.re, c)), fma2(v.re, d, mul2(v.im, c))};
}

// v * W_L^E with W_L = exp(-2 pi i / L)
template <int E, int L>
__device__ __forceinline__ cx2 twiddle(cx2 v) {
  constexpr int e = ((E % L) + L) % L;
  if constexpr (e == 0) {
    return v;
  } else if constexpr ((8 * e) % L == 0) {
    constexpr int oct = 8 * e / L;
    constexpr float r = 0.70710678118654752440f;
    const float2 R = dup(r);
    if constexpr (oct == 2) return {v.im, mul2(v.re, dup(-1.0f))};
    else if constexpr (oct == 4) return {mul2(v.re, dup(-1.0f)), mul2(v.im, dup(-1.0f))};
    else if constexpr (oct == 6) return {mul2(v.im, dup(-1.0f)), v.re};
    else if constexpr (oct == 1) return {mul2(add2(v.re, v.im), R), mul2(sub2(v.im, v.re), R)};
    else if constexpr (oct == 3) return {mul2(sub2(v.im, v.re), R), mul2(add2(v.re, v.im), dup(-r))};
    else if constexpr (oct == 5) return {mul2(add2(v.re, v.im), dup(-r)), mul2(sub2(v.re, v.im), R)};
    else return {mul2(sub2(v.re, v.im), R), mul2(add2(v.re, v.im), R)};
  } else {
    constexpr float c = (float)cx_cos_turn(e, L);
    constexpr float s = (float)cx_sin_turn(e, L);
    // W = c - i s: (re c + im s, im c - re s)
    return {fma2(v.im, dup(s), mul2(v.re, dup(c))), fma2(v.re, dup(-s), mul2(v.im, dup(c)))};
  }
}

template <int R>
__device__ __forceinline__ void butterfly(cx2 (&a)[R]);

template <>
__device__ __forceinline__ void butterfly<2>(cx2 (&a)[2]) {
  const cx2 t = a[0];
  a[0] = cadd(t, a[1]);
  a[1] = csub(t, a[1]);
}

template <>
__device__ __forceinline__ void butterfly<3>(cx2 (&a)[3]) {
  constexpr float h = 0.86602540378443864676f;
  const cx2 b = cadd(a[1], a[2]);
  const cx2 d = cscale(csub(a[1], a[2]), dup(h));
  const cx2 m = {fma2(b.re, dup(-0.5f), a[0].re), fma2(b.im, dup(-0.5f), a[0].im)};
  a[0] = cadd(a[0], b);
  a[1] = add_mi(m, d);
  a[2] = add_pi(m, d);
}

template <>
__device__ __forceinline__ void butterfly<4>(cx2 (&a)[4]) {
  const cx2 s02 = cadd(a[0], a[2]), d02 = csub(a[0], a[2]);
  const cx2 s13 = cadd(a[1], a[3]), d13 = csub(a[1], a[3]);
  a[0] = cadd(s02, s13);
  a[2] = csub(s02, s13);
  a[1] = add_mi(d02, d13);
  a[3] = add_pi(d02, d13);
}

template <>
__device__ __forceinline__ void butterfly<5>(cx2 (&a)[5]) {
  constexpr float c1 = 0.30901699437494742410f, c2 = -0.80901699437494742410f;
  constexpr float s1 = 0.95105651629515357212f, s2 = 0.58778525229247312917f;
  const cx2 b1 = cadd(a[1], a[4]), d1 = csub(a[1], a[4]);
  const cx2 b2 = cadd(a[2], a[3]), d2 = csub(a[2], a[3]);
  const cx2 a0 = a[0];
  const cx2 t1 = {fma2(b2.re, dup(c2), fma2(b1.re, dup(c1), a0.re)), fma2(b2.im, dup(c2), fma2(b1.im, dup(c1), a0.im))};
  const cx2 t2 = {fma2(b2.re, dup(c1), fma2(b1.re, dup(c2), a0.re)), fma2(b2.im, dup(c1), fma2(b1.im, dup(c2), a0.im))};
  const cx2 u1 = {fma2(d2.re, dup(s2), mul2(d1.re, dup(s1))), fma2(d2.im, dup(s2), mul2(d1.im, dup(s1)))};
  const cx2 u2 = {fma2(d2.re, dup(-s1), mul2(d1.re, dup(s2))), fma2(d2.im, dup(-s1), mul2(d1.im, dup(s2)))};
  a[0] = cadd(a0, cadd(b1, b2));
  a[1] = add_mi(t1, u1);
  a[4] = add_pi(t1, u1);
  a[2] = add_mi(t2, u2);
  a[3] = add_pi(t2, u2);
}

template <int L>
__device__ __forceinline__ void dft(cx2 (&x)[L]);

// Prime-factor DFT for coprime L = R * L2, as the float2 version in
// fm_fft.cuh: no twiddle multiplies between the two stages.
template <int L, int R, int L2>
__device__ __forceinline__ void dft_pfa(cx2 (&x)[L]) {
  constexpr int ka = L2 * cx_mod_inverse(L2 % R, R) % L, kb = R * cx_mod_inverse(R % L2, L2) % L;
  cx2 y[R][L2];
#pragma unroll
  for (int n1 = 0; n1 < R; ++n1)
#pragma unroll
    for (int n2 = 0; n2 < L2; ++n2) y[n1][n2] = x[(L2 * n1 + R * n2) % L];
#pragma unroll
  for (int n1 = 0; n1 < R; ++n1) dft<L2>(y[n1]);
#pragma unroll
  for (int k2 = 0; k2 < L2; ++k2) {
    cx2 t[R];
#pragma unroll
    for (int n1 = 0; n1 < R; ++n1) t[n1] = y[n1][k2];
    dft<R>(t);
#pragma unroll
    for (int k1 = 0; k1 < R; ++k1) x[(ka * k1 + kb * k2) % L] = t[k1];
  }
}

// L-point DFT: butterflies, the prime-factor split for coprime power-of-two
// and odd parts, otherwise decimation in time, L = R * L2: n = R n2 + n1,
// k = k2 + L2 k1.
template <int L>
__device__ __forceinline__ void dft(cx2 (&x)[L]) {
  if constexpr (L == 1) {
    return;
  } else if constexpr (L == 2 || L == 3 || L == 4 || L == 5) {
    butterfly<L>(x);
  } else if constexpr (CoprimeSplit<L>::R != 0) {
    dft_pfa<L, CoprimeSplit<L>::R, CoprimeSplit<L>::L2>(x);
  } else {
    constexpr int R = FirstFactor<L>::value;
    static_assert(R != 0, "DFT size must factor into 2, 3, 4 and 5");
    constexpr int L2 = L / R;
    cx2 y[R][L2];
#pragma unroll
    for (int n1 = 0; n1 < R; ++n1)
#pragma unroll
      for (int n2 = 0; n2 < L2; ++n2) y[n1][n2] = x[R * n2 + n1];
#pragma unroll
    for (int n1 = 0; n1 < R; ++n1) dft<L2>(y[n1]);
    static_for<1, R>([&](auto n1c) {
      constexpr int n1 = decltype(n1c)::value;
      static_for<1, L2>([&](auto k2c) {
        constexpr int k2 = decltype(k2c)::value;
        y[n1][k2] = twiddle<n1 * k2, L>(y[n1][k2]);
      });
    });
#pragma unroll
    for (int k2 = 0; k2 < L2; ++k2) {
      cx2 t[R];
#pragma unroll
      for (int n1 = 0; n1 < R; ++n1) t[n1] = y[n1][k2];
      butterfly<R>(t);
#pragma unroll
      for (int k1 = 0; k1 < R; ++k1) x[k2 + L2 * k1] = t[k1];
    }
  }
}

}  // namespace fm
