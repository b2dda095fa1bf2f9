// Register-resident complex DFTs for the mel kernel (sm_103a).
//
// Small DFTs are written out as radix-2/3/4/5 butterflies; larger ones are
// composed by decimation in time with compile-time twiddles. The twiddle
// constants come from a Taylor series in double evaluated by the compiler
// (no device trigonometry, no tables), and the eighth-turn twiddles are
// applied exactly (swaps and sign flips, or a single 1/sqrt(2) scale).
#pragma once

#include <cuda_runtime.h>

#include <type_traits>

namespace fm {

// ---------------------------------------------------------------------------
// Compile-time trigonometry: Taylor series in double on the reduced angle
// 2 pi a / d in (-pi, pi]; 30 terms leave an error far below float rounding.
// ---------------------------------------------------------------------------
constexpr double kPi = 3.141592653589793238462643383279502884;

constexpr double cx_sin_series(double x) {
  double term = x, sum = x;
  for (int i = 1; i < 30; ++i) {
    term *= -x * x / ((2.0 * i) * (2.0 * i + 1.0));
    sum += term;
  }
  return sum;
}
constexpr double cx_cos_series(double x) {
  double term = 1.0, sum = 1.0;
  for (int i = 1; i < 30; ++i) {
    term *= -x * x / ((2.0 * i - 1.0) * (2.0 * i));
    sum += term;
  }
  return sum;
}
constexpr double cx_turn_angle(long long a, long long d) {
  a %= d;
  if (a < 0) a += d;
  if (2 * a > d) a -= d;
  return 2.0 * kPi * (double)a / (double)d;
}
constexpr double cx_cos_turn(long long a, long long d) { return cx_cos_series(cx_turn_angle(a, d)); }
constexpr double cx_sin_turn(long long a, long long d) { return cx_sin_series(cx_turn_angle(a, d)); }

template <int B, int E, typename F>
__device__ __forceinline__ void static_for(F&& f) {
  if constexpr (B < E) {
    f(std::integral_constant<int, B>{});
    static_for<B + 1, E>(f);
  }
}

// ---------------------------------------------------------------------------
// Complex helpers (float2 = re, im)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 csub(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }
__device__ __forceinline__ float2 cscale(float2 a, float s) { return make_float2(a.x * s, a.y * s); }
// a * w for w = (cos, -sin) stored as a plain complex number
__device__ __forceinline__ float2 cmul(float2 a, float2 w) {
  return make_float2(fmaf(a.x, w.x, -a.y * w.y), fmaf(a.x, w.y, a.y * w.x));
}
__device__ __forceinline__ float2 mul_neg_i(float2 v) { return make_float2(v.y, -v.x); }
__device__ __forceinline__ float2 mul_pos_i(float2 v) { return make_float2(-v.y, v.x); }

// v * W_L^E, W_L = exp(-2 pi i / L), with exact handling of the eighth turns.
template <int E, int L>
__device__ __forceinline__ float2 twiddle(float2 v) {
  constexpr int e = ((E % L) + L) % L;
  if constexpr (e == 0) {
    return v;
  } else if constexpr ((8 * e) % L == 0) {
    constexpr int oct = 8 * e / L;
    constexpr float r = 0.70710678118654752440f;
    if constexpr (oct == 2) return mul_neg_i(v);
    else if constexpr (oct == 4) return make_float2(-v.x, -v.y);
    else if constexpr (oct == 6) return mul_pos_i(v);
    else if constexpr (oct == 1) return make_float2((v.x + v.y) * r, (v.y - v.x) * r);
    else if constexpr (oct == 3) return make_float2((v.y - v.x) * r, -(v.x + v.y) * r);
    else if constexpr (oct == 5) return make_float2(-(v.x + v.y) * r, (v.x - v.y) * r);
    else return make_float2((v.x - v.y) * r, (v.x + v.y) * r);
  } else {
    constexpr float c = (float)cx_cos_turn(e, L);
    constexpr float s = (float)cx_sin_turn(e, L);
    return make_float2(fmaf(v.x, c, v.y * s), fmaf(v.y, c, -v.x * s));
  }
}

// ---------------------------------------------------------------------------
// Small DFTs in registers: A[k] = sum_n a[n] W_R^{nk}, natural order in/out.
// ---------------------------------------------------------------------------
template <int R>
__device__ __forceinline__ void butterfly(float2 (&a)[R]);

template <>
__device__ __forceinline__ void butterfly<2>(float2 (&a)[2]) {
  const float2 t = a[0];
  a[0] = cadd(t, a[1]);
  a[1] = csub(t, a[1]);
}

template <>
__device__ __forceinline__ void butterfly<3>(float2 (&a)[3]) {
  constexpr float h = 0.86602540378443864676f;  // sin(2 pi / 3)
  const float2 b = cadd(a[1], a[2]);
  const float2 d = cscale(csub(a[1], a[2]), h);
  const float2 m = make_float2(fmaf(-0.5f, b.x, a[0].x), fmaf(-0.5f, b.y, a[0].y));
  a[0] = cadd(a[0], b);
  a[1] = cadd(m, mul_neg_i(d));
  a[2] = cadd(m, mul_pos_i(d));
}

template <>
__device__ __forceinline__ void butterfly<4>(float2 (&a)[4]) {
  const float2 s02 = cadd(a[0], a[2]), d02 = csub(a[0], a[2]);
  const float2 s13 = cadd(a[1], a[3]), d13 = csub(a[1], a[3]);
  a[0] = cadd(s02, s13);
  a[2] = csub(s02, s13);
  a[1] = cadd(d02, mul_neg_i(d13));
  a[3] = cadd(d02, mul_pos_i(d13));
}

template <>
__device__ __forceinline__ void butterfly<5>(float2 (&a)[5]) {
  constexpr float c1 = 0.30901699437494742410f;   // cos(2 pi/5)
  constexpr float c2 = -0.80901699437494742410f;  // cos(4 pi/5)
  constexpr float s1 = 0.95105651629515357212f;   // sin(2 pi/5)
  constexpr float s2 = 0.58778525229247312917f;   // sin(4 pi/5)
  const float2 b1 = cadd(a[1], a[4]), d1 = csub(a[1], a[4]);
  const float2 b2 = cadd(a[2], a[3]), d2 = csub(a[2], a[3]);
  const float2 a0 = a[0];
  const float2 t1 = make_float2(fmaf(c2, b2.x, fmaf(c1, b1.x, a0.x)), fmaf(c2, b2.y, fmaf(c1, b1.y, a0.y)));
  const float2 t2 = make_float2(fmaf(c1, b2.x, fmaf(c2, b1.x, a0.x)), fmaf(c1, b2.y, fmaf(c2, b1.y, a0.y)));
  const float2 u1 = make_float2(fmaf(s2, d2.x, s1 * d1.x), fmaf(s2, d2.y, s1 * d1.y));
  const float2 u2 = make_float2(fmaf(-s1, d2.x, s2 * d1.x), fmaf(-s1, d2.y, s2 * d1.y));
  a[0] = cadd(a0, cadd(b1, b2));
  a[1] = cadd(t1, mul_neg_i(u1));
  a[4] = cadd(t1, mul_pos_i(u1));
  a[2] = cadd(t2, mul_neg_i(u2));
  a[3] = cadd(t2, mul_pos_i(u2));
}

template <int L>
struct FirstFactor {
  static constexpr int value = (L % 4 == 0) ? 4 : (L % 2 == 0) ? 2 : (L % 5 == 0) ? 5 : (L % 3 == 0) ? 3 : 0;
};

// Coprime split L = R * L2 for the prime-factor (Good-Thomas) algorithm: R is
// the power-of-two part of L, L2 the odd part; R = 0 when either is 1.
template <int L>
struct CoprimeSplit {
  static constexpr int pow2 = L & -L;
  static constexpr int R = (pow2 > 1 && pow2 < L) ? pow2 : 0;
  static constexpr int L2 = R ? L / R : 0;
};

// a^-1 mod m for coprime a, m (m small; evaluated by the compiler)
constexpr int cx_mod_inverse(int a, int m) {
  for (int x = 1; x < m; ++x)
    if ((a * x) % m == 1) return x;
  return m == 1 ? 0 : -1;
}

template <int L>
__device__ __forceinline__ void dft(float2 (&x)[L]);

// Prime-factor DFT for coprime L = R * L2 (Good-Thomas): with the input map
// n = (L2 n1 + R n2) mod L and the Chinese-remainder output map
// k = (L2 (L2^-1 mod R) k1 + R (R^-1 mod L2) k2) mod L, the kernel W_L^{nk}
// factors into W_R^{n1 k1} W_L2^{n2 k2}: L2-point DFTs over n2, then R-point
// DFTs over n1, and no twiddle multiplies between them.
template <int L, int R, int L2>
__device__ __forceinline__ void dft_pfa(float2 (&x)[L]) {
  constexpr int ka = L2 * cx_mod_inverse(L2 % R, R) % L, kb = R * cx_mod_inverse(R % L2, L2) % L;
  float2 y[R][L2];
#pragma unroll
  for (int n1 = 0; n1 < R; ++n1)
#pragma unroll
    for (int n2 = 0; n2 < L2; ++n2) y[n1][n2] = x[(L2 * n1 + R * n2) % L];
#pragma unroll
  for (int n1 = 0; n1 < R; ++n1) dft<L2>(y[n1]);
#pragma unroll
  for (int k2 = 0; k2 < L2; ++k2) {
    float2 t[R];
#pragma unroll
    for (int n1 = 0; n1 < R; ++n1) t[n1] = y[n1][k2];
    dft<R>(t);
#pragma unroll
    for (int k1 = 0; k1 < R; ++k1) x[(ka * k1 + kb * k2) % L] = t[k1];
  }
}

// L-point DFT: radix-2/3/4/5 butterflies; the prime-factor split when L has
// coprime power-of-two and odd parts; otherwise decimation in time,
// L = R * L2: n = R n2 + n1, k = k2 + L2 k1.
template <int L>
__device__ __forceinline__ void dft(float2 (&x)[L]) {
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
    float2 y[R][L2];
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
      float2 t[R];
#pragma unroll
      for (int n1 = 0; n1 < R; ++n1) t[n1] = y[n1][k2];
      butterfly<R>(t);
#pragma unroll
      for (int k1 = 0; k1 < R; ++k1) x[k2 + L2 * k1] = t[k1];
    }
  }
}

}  // namespace fm
