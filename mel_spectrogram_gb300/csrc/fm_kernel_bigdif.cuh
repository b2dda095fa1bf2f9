// Mel kernel for the large transforms, decimation-in-frequency build (sm_103a).
//
// The same path as mel_kernel_big (padding and framing as index arithmetic,
// periodic Hann, the complex M = n_fft/2 point DFT of the windowed pairs
// z[n] = (y[2n] + i y[2n+1]) / 2, its split, |X|^p and the CSR mel
// projection), with the M-point DFT factored the other way round,
// M = 16 MS, n = n1 MS + n2, k = k1 + 16 k2:
//   Z[k1 + 16 k2] = sum_n2 W_MS^{n2 k2} (W_M^{n2 k1} sum_n1 z[n1 MS + n2] W_16^{n1 k1})
//   step A : for every n2 < MS of every frame of the tile, the 16-point DFT
//            over n1, read straight from the signal (lanes take consecutive
//            n2, so each of the 16 loads is coalesced), times W_M^{n2 k1};
//            value k1 goes to position n2 of sub-frame k1;
//   step B : the MS-point DFT of every sub-frame, two autosorting passes
//            (RA x RB = MS) in the sub-frame's own shared memory; each warp
//            holds whole sub-frames, so the passes need warp barriers only;
//            afterwards position k2 of sub-frame k1 holds Z[k1 + 16 k2];
//   split  : as in mel_kernel_big, reading Z[k] from sub-frame k mod 16,
//            position k / 16;
//   mel    : mel_project_lanes (a lane per filter and frame) or
//            mel_project_taps (a warp per filter, lanes over its taps), as
//            the plan chose from the filter widths.
// Against the three-pass build, the load and the first pass are one step
// (the windowed samples make no round trip through shared memory) and a tile
// crosses five CTA barriers instead of ten. One group of 512 threads, tiles
// of 32768 / n_fft frames, samples read from global memory (no staging).
#pragma once

#include "fm_kernel_big.cuh"

namespace fm {

// Radices of the two sub-frame passes, MS = RA RB.
template <int MS>
struct DifRadices;
template <>
struct DifRadices<128> {
  static constexpr int RA = 16, RB = 8;
};
template <>
struct DifRadices<256> {
  static constexpr int RA = 16, RB = 16;
};
template <>
struct DifRadices<512> {
  static constexpr int RA = 16, RB = 32;
};

// Step A inputs of this thread: task t is (f, n2) = ((tid + t TH) / MS,
// (tid + t TH) % MS), its value n1 the windowed pair z[n1 MS + n2] of frame f
// (frame f starts at padded position s0 + f hop). Every global load of the
// tile is issued before the first one is used.
template <int N, int F, int TH, typename Raw>
__device__ __forceinline__ void dif_load(float2 (&v)[F * (N / 2 / kDifR0) / TH][kDifR0], const Raw* __restrict__ sig,
                                         long long T, long long s0, int hop, const float2* __restrict__ win2,
                                         const PadSpec& ps, int tid, unsigned* err) {
  constexpr int MS = N / 2 / kDifR0, TASKS = F * MS / TH;
  const bool interior = s0 >= 0 && s0 + (long long)(F - 1) * hop + N <= T;
#pragma unroll
  for (int t = 0; t < TASKS; ++t) {
    const int task = tid + t * TH, f = task / MS, n2 = task % MS;
#pragma unroll
    for (int n1 = 0; n1 < kDifR0; ++n1) {
      const long long s = s0 + (long long)f * hop + 2 * (n1 * MS + n2);
      if (interior) {
        v[t][n1] = FM_IN(s >= 0 && s + 1 < T, err) ? make_float2(raw_to_float(sig[s]), raw_to_float(sig[s + 1]))
                                                   : make_float2(0.0f, 0.0f);
      } else {
        v[t][n1] = make_float2(big_sample(sig, T, s, ps), big_sample(sig, T, s + 1, ps));
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TASKS; ++t) {
    const int n2 = (tid + t * TH) % MS;
#pragma unroll
    for (int n1 = 0; n1 < kDifR0; ++n1) {
      const float2 w = __ldg(win2 + n1 * MS + n2);
      v[t][n1] = make_float2(v[t][n1].x * w.x, v[t][n1].y * w.y);
    }
  }
}

// Real-FFT split and |X|^p for k = 0 .. M/2 of every frame into the power
// tile (float rows of M + 1 aliasing the buffer: all reads, barrier, writes),
// Z[k] of frame f at position k / 16 of sub-frame 16 f + k mod 16.
template <int M, int F, int TH, int MODE>
__device__ __forceinline__ void dif_split(const float2* s_x, float* s_pw, const float2* s_twn, float pw, int tid,
                                          Cap x_cap, Cap p_cap) {
  constexpr int MS = M / kDifR0, SFS = big_frame_stride(MS), PS = M + 1;
  constexpr int PAIRS = M / 2 + 1, TOTAL = F * PAIRS;
  constexpr int PER = (TOTAL + TH - 1) / TH;
  static_assert(kDifR0 == 16, "k / 16 and k mod 16 below");
  float lo[PER], hi[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int task = tid + i * TH;
    lo[i] = hi[i] = 0.0f;
    if (task < TOTAL) {
      const int f = task / PAIRS, k = task % PAIRS, km = (M - k) & (M - 1);
      const float2 zk = get<float2>(s_x, 0, (f * kDifR0 + (k & 15)) * SFS + big_phys(k >> 4), x_cap);
      const float2 zm = get<float2>(s_x, 0, (f * kDifR0 + (km & 15)) * SFS + big_phys(km >> 4), x_cap);
      // W_N^k from the two twiddle rows of W_N
      const float2 w = cmul(s_twn[k & (kBigTwFine - 1)], s_twn[kBigTwFine + (k >> 6)]);
      split_pair<MODE>(zk, zm, w, pw, lo[i], hi[i]);
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int task = tid + i * TH;
    if (task < TOTAL) {
      const int f = task / PAIRS, k = task % PAIRS;
      put(s_pw, 0, f * PS + k, lo[i], p_cap);
      put(s_pw, 0, f * PS + M - k, hi[i], p_cap);
    }
  }
  __syncthreads();
}

// The tile loop: tiles blockIdx.x + gridDim.x k of F = 32768 / n_fft frames.
template <int N, typename Raw>
__device__ __forceinline__ void run_tiles_dif(const KernelParams& prm, unsigned char* smem, int tid) {
  constexpr int M = N / 2, MS = M / kDifR0, F = big_frames(N), TH = kBigThreads, NWARPS = TH / 32;
  constexpr int RA = DifRadices<MS>::RA, RB = DifRadices<MS>::RB, SFS = big_frame_stride(MS);
  constexpr int TASKS = F * MS / TH;          // step A tasks per thread
  constexpr int SUB = F * kDifR0 / NWARPS;    // sub-frames per warp in step B
  static_assert(RA * RB == MS && (F * MS) % TH == 0 && (F * kDifR0) % NWARPS == 0, "radices and tasks");
  float2* s_x = reinterpret_cast<float2*>(smem);
  float* s_pw = reinterpret_cast<float*>(smem);
  const int warp = tid >> 5, lane = tid & 31;
  const Raw* in = static_cast<const Raw*>(prm.in);
  const float2* win2 = reinterpret_cast<const float2*>(prm.win);
  const long long T = prm.T;
  const TileSplitter split(prm.tiles_per_signal);
  const PadSpec pads = {prm.zpad, prm.cpad, prm.pad_mode};
  const BigLayout lay = big_layout(N, prm.n_mels, prm.nnz, true);
  const float2* s_tw = reinterpret_cast<const float2*>(smem + lay.tw);  // W_M rows, then W_N rows
  const float2* s_twn = s_tw + kBigTwFine + M / kBigTwFine;
  const int4* s_mel = reinterpret_cast<const int4*>(smem + lay.mel);
  const float* s_mw = reinterpret_cast<const float*>(smem + lay.mw);
  // buffer sizes for the debug build's index checks; a warp's sub-frames are
  // checked against what is left of the buffer after them
  const Cap x_cap = {F * kDifR0 * SFS, prm.err}, p_cap = {F * (M + 1), prm.err};
  float2* s_w = s_x + warp * SUB * SFS;
  const Cap w_cap = {x_cap.n - warp * SUB * SFS, prm.err};
  const long long out_total = prm.B * (long long)prm.n_mels * prm.n_frames;
  for (long long tile = blockIdx.x; tile < prm.total_tiles; tile += gridDim.x) {
    long long b;
    int tt;
    split(tile, b, tt);
    const int t0 = tt * F;
    // step A in registers: loads, 16-point DFTs over n1, W_M^{n2 k1}
    float2 v[TASKS][kDifR0];
    dif_load<N, F, TH, Raw>(v, in + b * T, T, (long long)t0 * prm.hop - prm.lead, prm.hop, win2, pads, tid,
                            prm.err);
#pragma unroll
    for (int t = 0; t < TASKS; ++t) {
      const int n2 = (tid + t * TH) % MS;
      dft<kDifR0>(v[t]);
#pragma unroll
      for (int k1 = 1; k1 < kDifR0; ++k1) v[t][k1] = cmul(v[t][k1], big_tw<M>(s_tw, n2 * k1));
    }
    __syncthreads();  // the previous tile's mel reads of the power tile are done
#pragma unroll
    for (int t = 0; t < TASKS; ++t) {
      const int task = tid + t * TH, f = task / MS, n2 = task % MS;
#pragma unroll
      for (int k1 = 0; k1 < kDifR0; ++k1) put(s_x, 0, (f * kDifR0 + k1) * SFS + big_phys(n2), v[t][k1], x_cap);
    }
    __syncthreads();
    // step B: this warp's SUB sub-frames, warp barriers only. Below MS = 512
    // the first pass runs on G1 sub-frames at a time (one butterfly a lane),
    // which keeps the 4096 and 8192 builds free of register spills.
    if constexpr (MS < 512) {
      constexpr int G1 = 32 * RA / MS;
#pragma unroll 1
      for (int sf = 0; sf < SUB; sf += G1)
        big_pass<MS, G1, 32, RA, 1, kDifR0>(s_w + sf * SFS, s_tw, lane, 0, {w_cap.n - sf * SFS, w_cap.err});
    } else {
      big_pass<MS, SUB, 32, RA, 1, kDifR0>(s_w, s_tw, lane, 0, w_cap);
    }
    big_pass<MS, SUB, 32, RB, RA, kDifR0>(s_w, s_tw, lane, 0, w_cap);
    __syncthreads();
    switch (prm.power_mode) {
      case 0: dif_split<M, F, TH, 0>(s_x, s_pw, s_twn, prm.power, tid, x_cap, p_cap); break;
      case 1: dif_split<M, F, TH, 1>(s_x, s_pw, s_twn, prm.power, tid, x_cap, p_cap); break;
      default: dif_split<M, F, TH, 2>(s_x, s_pw, s_twn, prm.power, tid, x_cap, p_cap); break;
    }
    const int n_valid = min(F, prm.n_frames - t0);
    const long long obase = b * prm.n_mels * (long long)prm.n_frames + t0;
    if (prm.out_dtype == FM_F32) {
      float* o = static_cast<float*>(prm.out) + obase;
      if (prm.mel_taps)
        mel_project_taps<F, NWARPS, M + 1>(s_pw, s_mel, s_mw, o, n_valid, prm.n_mels, prm.n_frames, warp, lane,
                                           p_cap, prm.nnz, out_total - obase);
      else
        mel_project_lanes<F, NWARPS, M + 1>(s_pw, s_mel, s_mw, o, n_valid, prm.n_mels, prm.n_frames, warp, lane,
                                            p_cap, prm.nnz, out_total - obase);
    } else {
      __half* o = static_cast<__half*>(prm.out) + obase;
      if (prm.mel_taps)
        mel_project_taps<F, NWARPS, M + 1>(s_pw, s_mel, s_mw, o, n_valid, prm.n_mels, prm.n_frames, warp, lane,
                                           p_cap, prm.nnz, out_total - obase);
      else
        mel_project_lanes<F, NWARPS, M + 1>(s_pw, s_mel, s_mw, o, n_valid, prm.n_mels, prm.n_frames, warp, lane,
                                            p_cap, prm.nnz, out_total - obase);
    }
  }
}

template <int N>
__global__ void __launch_bounds__(kBigThreads, 1) mel_kernel_bigdif(const KernelParams prm) {
  extern __shared__ __align__(16) unsigned char smem[];
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  big_tables<N>(prm, smem, big_layout(N, prm.n_mels, prm.nnz, true), tid);
  if (prm.in_dtype == FM_F32) run_tiles_dif<N, float>(prm, smem, tid);
  else if (prm.in_dtype == FM_I16) run_tiles_dif<N, short>(prm, smem, tid);
  else run_tiles_dif<N, __half>(prm, smem, tid);
}

}  // namespace fm

// Instantiate one decimation-in-frequency large-transform variant:
// FM_DEFINE_VARIANT_BIGDIF(name, N); P = 16 (the first DFTs), Q = the
// sub-frame length.
#define FM_DEFINE_VARIANT_BIGDIF(NAME, N)                                                             \
  namespace fm {                                                                                      \
  template __global__ void mel_kernel_bigdif<N>(const KernelParams);                                 \
  extern const Variant NAME = {N, kDifR0, N / 2 / kDifR0, big_frames(N), kBigThreads, 0, 2,           \
                               (const void*)&mel_kernel_bigdif<N>, kAnyHop, 1};                       \
  }
