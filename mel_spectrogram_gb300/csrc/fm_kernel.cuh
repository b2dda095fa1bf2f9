// Fused mel-spectrogram kernel for sm_103a.
//
// One launch runs the whole path of the flashmel README ("How it works"):
// centre reflect padding and framing as index arithmetic, the periodic Hann
// window, the n_fft-point real DFT, |X|^power and the sparse triangular mel
// projection, with coalesced stores of [B][n_mels][n_frames].
//
// Work split. A tile is G consecutive frames of one signal. A persistent grid
// of CTAs walks the tiles. Inside a CTA, thread (role, g) with g = tid % G
// owns frame g of the tile and plays `role` = tid / G in each phase, so every
// role-dependent constant (window slice, twiddles, filter row) is uniform
// across the G lanes that share it.
//
// The real n_fft-point DFT of frame y is computed as the complex M = n_fft/2
// point DFT of z[n] = (y[2n] + i y[2n+1]) / 2, split four-step as M = P * Q:
//   pass 1 : role p (0..P-1) takes z[p + P q], q < Q, does a Q-point DFT in
//            registers and multiplies output k2 by W_M^{p k2};
//   pass 2 : role t does the P-point DFTs over p for its Q/P values of k2,
//            giving Z[k2 + Q k1];
//   split  : X[k] = S + U and X[M-k] = conj(S - U) with S = Z[k] + conj Z[M-k],
//            U = -i W_N^k (Z[k] - conj Z[M-k]) (the 1/2 sits in the window).
// Exchanges between the passes go through shared memory with a frame stride of
// M + 1 (odd) complex values, so the G lanes of a role hit distinct banks.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "fm_internal.h"

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

// L-point DFT by decimation in time, L = R * L2: n = R n2 + n1, k = k2 + L2 k1.
template <int L>
__device__ __forceinline__ void dft(float2 (&x)[L]) {
  if constexpr (L == 1) {
    return;
  } else if constexpr (L == 2 || L == 3 || L == 4 || L == 5) {
    butterfly<L>(x);
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

// ---------------------------------------------------------------------------
// Input load and output store by dtype (warp-uniform branches)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float load_sample(const void* in, int dt, long long i) {
  if (dt == FM_F32) return __ldg(static_cast<const float*>(in) + i);
  if (dt == FM_I16) return (float)__ldg(static_cast<const short*>(in) + i) * (1.0f / 32768.0f);
  return __half2float(__ldg(static_cast<const __half*>(in) + i));
}

__device__ __forceinline__ void store_out(void* out, int dt, long long i, float v) {
  if (dt == FM_F32) static_cast<float*>(out)[i] = v;
  else static_cast<__half*>(out)[i] = __float2half_rn(v);
}

__device__ __forceinline__ float apply_power(float m2, int mode, float p) {
  if (mode == 0) return m2;
  if (mode == 1) return sqrtf(m2);
  return powf(m2, 0.5f * p);
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int N, int P, int Q, int G>
__global__ void __launch_bounds__(P* G) mel_kernel(const KernelParams prm) {
  constexpr int M = N / 2;
  constexpr int THREADS = P * G;
  constexpr int GS = M + 1;        // complex stride between frames in xbuf (odd)
  constexpr int PS = M + 1;        // float stride between frames in the power tile (odd)
  constexpr int K2R = Q / P;       // k2 values per role in pass 2
  constexpr int PAIRS = M / 2 + 1; // (k, M-k) pairs, k = 0..M/2
  constexpr int PPR = (PAIRS + P - 1) / P;
  constexpr int SUBS = 32 / G;     // mels per warp in the projection
  static_assert(P * Q == M && Q % P == 0, "bad FFT split");
  static_assert(G == 32 || G == 16, "frames per tile must be 16 or 32");
  static_assert(THREADS % 32 == 0, "CTA must be whole warps");

  extern __shared__ __align__(16) unsigned char smem[];
  const int hop = prm.hop;
  const int n_mels = prm.n_mels;
  const SmemLayout lay = smem_layout(N, hop, n_mels, prm.nnz, G);
  float* s_win = reinterpret_cast<float*>(smem + lay.window);
  float2* s_twh = reinterpret_cast<float2*>(smem + lay.tw_half);
  float2* s_twf = reinterpret_cast<float2*>(smem + lay.tw_full);
  int* s_ms = reinterpret_cast<int*>(smem + lay.mel_start);
  int* s_ml = reinterpret_cast<int*>(smem + lay.mel_len);
  int* s_mo = reinterpret_cast<int*>(smem + lay.mel_off);
  float* s_mw = reinterpret_cast<float*>(smem + lay.mel_w);
  float* s_in = reinterpret_cast<float*>(smem + lay.in_tile);
  float2* s_x = reinterpret_cast<float2*>(smem + lay.xbuf);
  float* s_pw = reinterpret_cast<float*>(smem + lay.xbuf);  // aliases s_x after the split

  const int tid = threadIdx.x;
  const int g = tid % G;
  const int role = tid / G;
  const int warp = tid >> 5, lane = tid & 31;
  const int S = in_row_stride(hop);
  const int rows = in_rows(N, hop, G);

  // per-CTA constant tables, loaded once (the grid is persistent)
  for (int i = tid; i < N; i += THREADS) s_win[i] = prm.window[i];
  for (int i = tid; i < M; i += THREADS) s_twh[i] = prm.tw_half[i];
  for (int i = tid; i <= M; i += THREADS) s_twf[i] = prm.tw_full[i];
  for (int i = tid; i < n_mels; i += THREADS) {
    s_ms[i] = prm.mel_start[i];
    s_ml[i] = prm.mel_len[i];
    s_mo[i] = prm.mel_off[i];
  }
  for (int i = tid; i < prm.nnz; i += THREADS) s_mw[i] = prm.mel_w[i];

  for (long long tile = blockIdx.x; tile < prm.total_tiles; tile += gridDim.x) {
    const long long b = tile / prm.tiles_per_signal;
    const int t0 = (int)(tile - b * prm.tiles_per_signal) * G;
    const long long T = prm.T;
    const long long row_base = b * T;

    // ---- stage the tile's samples (reflect at the signal edges) -----------
    {
      const long long gstart = (long long)t0 * hop - prm.pad;  // signal index of tile position 0
      const bool interior = gstart >= 0 && gstart + (long long)rows * hop <= T;
      for (int r = warp; r < rows; r += THREADS / 32) {
        float* dst = s_in + r * S;
        const long long s0 = gstart + (long long)r * hop;
        if (interior) {
          for (int c = lane; c < hop; c += 32) dst[c] = load_sample(prm.in, prm.in_dtype, row_base + s0 + c);
        } else {
          for (int c = lane; c < hop; c += 32) {
            long long s = s0 + c;
            if (s < 0) s = -s;
            else if (s >= T) s = 2 * T - 2 - s;
            dst[c] = (s >= 0 && s < T) ? load_sample(prm.in, prm.in_dtype, row_base + s) : 0.0f;
          }
        }
      }
    }
    __syncthreads();

    float2* xrow = s_x + g * GS;

    // ---- pass 1: windowed Q-point DFTs over z[p + P q], twiddle W_M^{p k2} ----
    {
      const int p = role;
      float2 z[Q];
      int r = (2 * p) / hop;
      int c = 2 * p - r * hop;
      const float* base = s_in + g * S;
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        const float2 v = *reinterpret_cast<const float2*>(base + r * S + c);
        const float2 w = *reinterpret_cast<const float2*>(s_win + 2 * (p + P * q));
        z[q] = make_float2(v.x * w.x, v.y * w.y);
        c += 2 * P;
        while (c >= hop) {
          c -= hop;
          ++r;
        }
      }
      dft<Q>(z);
      xrow[p] = z[0];
#pragma unroll
      for (int k2 = 1; k2 < Q; ++k2) xrow[k2 * P + p] = cmul(z[k2], s_twh[p * k2]);
    }
    __syncthreads();

    // ---- pass 2: P-point DFTs over p, giving Z[k2 + Q k1] ------------------
    {
      float2 y[K2R][P];
#pragma unroll
      for (int j = 0; j < K2R; ++j) {
        const int k2 = role + j * P;
#pragma unroll
        for (int p = 0; p < P; ++p) y[j][p] = xrow[k2 * P + p];
        dft<P>(y[j]);
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < K2R; ++j) {
        const int k2 = role + j * P;
#pragma unroll
        for (int k1 = 0; k1 < P; ++k1) xrow[k2 + Q * k1] = y[j][k1];
      }
    }
    __syncthreads();

    // ---- real-FFT split and |X|^power into the power tile -------------------
    {
      float lo[PPR], hi[PPR];
#pragma unroll
      for (int i = 0; i < PPR; ++i) {
        const int k = role + i * P;
        lo[i] = hi[i] = 0.0f;
        if (k <= M / 2) {
          const float2 zk = xrow[k];
          const float2 zm = xrow[k == 0 ? 0 : M - k];
          const float2 s = make_float2(zk.x + zm.x, zk.y - zm.y);
          const float2 d = make_float2(zk.x - zm.x, zk.y + zm.y);
          const float2 u = mul_neg_i(cmul(d, s_twf[k]));
          const float2 xa = cadd(s, u), xb = csub(s, u);
          lo[i] = apply_power(fmaf(xa.x, xa.x, xa.y * xa.y), prm.power_mode, prm.power);
          hi[i] = apply_power(fmaf(xb.x, xb.x, xb.y * xb.y), prm.power_mode, prm.power);
        }
      }
      __syncthreads();
      float* prow = s_pw + g * PS;
#pragma unroll
      for (int i = 0; i < PPR; ++i) {
        const int k = role + i * P;
        if (k <= M / 2) {
          prow[k] = lo[i];
          prow[M - k] = hi[i];
        }
      }
    }
    __syncthreads();

    // ---- sparse mel projection, lane = frame, coalesced stores -------------
    {
      const int gg = lane % G;
      const int sub = lane / G;
      const int tf = t0 + gg;
      const bool valid = tf < prm.n_frames;
      const float* prow = s_pw + gg * PS;
      for (int m = warp * SUBS + sub; m < n_mels; m += (THREADS / 32) * SUBS) {
        const int st = s_ms[m], ln = s_ml[m], of = s_mo[m];
        float acc = 0.0f;
        for (int j = 0; j < ln; ++j) acc = fmaf(s_mw[of + j], prow[st + j], acc);
        if (valid) store_out(prm.out, prm.out_dtype, (b * n_mels + m) * (long long)prm.n_frames + tf, acc);
      }
    }
    // The next tile's staging writes only s_in; its pass 1 writes s_x after the
    // barrier that follows staging, so no barrier is needed here.
  }
}

}  // namespace fm

// Instantiate one variant: FM_DEFINE_VARIANT(name, N, P, Q, G)
#define FM_DEFINE_VARIANT(NAME, N, P, Q, G)                                              \
  namespace fm {                                                                         \
  template __global__ void mel_kernel<N, P, Q, G>(const KernelParams);                 \
  extern const Variant NAME = {N, P, Q, G, P * G, (const void*)&mel_kernel<N, P, Q, G>}; \
  }
