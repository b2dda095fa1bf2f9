// Paired-frame complex transform for n_fft = 400 (sm_103a): the alternative
// that the flashmel README measured and removed on its hardware ("Where each
// case actually sits (Nsight Compute)", whisper bullet: two frames per
// complex FFT via conjugate symmetry, about 1.5x slower there), built here to
// be measured against the two-frame packed kernel on GB300. Plans take it
// only when the diagnostic switch FM_MEL_N400_KERNEL=c2c is set.
//
// Frames a = g and b = g + 16 of a 32-frame tile form one complex signal
// z[n] = w[n] (y_a[n] + i y_b[n]) (w carries the 1/2 that the real-FFT split
// of the other kernels uses, so Z below is half the DFT); by conjugate
// symmetry its N-point DFT Z gives both spectra:
//   X_a[k] = Z[k] + conj Z[N-k],   i X_b[k] = Z[k] - conj Z[N-k],
// so |X_a|^2 and |X_b|^2 are the squared moduli of those two sums.
// Four-step with N = P x Q = 20 x 20, one frame pair per thread and role:
//   pass 1 : role p, Q-point DFT of z[p + P q], times W_N^{p k2};
//   pass 2 : role t, P-point DFT over p for k2 = t: Z[t + Q k1], written
//            back to shared memory in natural order;
//   split  : role t separates the pairs (k, N - k), k = t + P i <= N/2;
//   mel    : the CSR projection of the one-frame-per-thread kernel.
// Scalar complex arithmetic: the pair already fills the real and imaginary
// lanes, so there is nothing left to pack.
#pragma once

#include "fm_kernel.cuh"

namespace fm {

constexpr int kC2cP = 20, kC2cQ = 20, kC2cN = 400;
constexpr int kC2cPairs = 16;                   // frame pairs per tile (32 frames)
constexpr int kC2cThreads = kC2cP * kC2cPairs;  // 320

// Shared-memory layout: pass-1 table (window times the int16 scale and the
// sample's tile offset, per role and step), W_N^j (j < N), filterbank, two
// staging buffers of rows of one hop, the exchange buffer (16 pairs x 401
// complex, odd stride; the power tile of 32 frames x 201 floats aliases it).
struct SmemLayoutC2c {
  size_t tab, tw, mel, mel_w, in_tile, in_tile_bytes, xbuf, total;
};
__host__ __device__ inline SmemLayoutC2c smem_layout_c2c(int hop, int n_mels, int nnz, int in_esize) {
  SmemLayoutC2c L;
  size_t o = 0;
  L.tab = o;    o = align16(o + sizeof(float2) * kC2cN);
  L.tw = o;     o = align16(o + sizeof(float2) * kC2cN);
  L.mel = o;    o = align16(o + sizeof(int4) * n_mels);
  L.mel_w = o;  o = align16(o + sizeof(float) * (nnz > 0 ? nnz : 1));
  L.in_tile_bytes = align16((size_t)in_esize * in_rows(kC2cN, hop, 2 * kC2cPairs) * in_row_stride(hop));
  L.in_tile = o; o += 2 * L.in_tile_bytes;
  L.xbuf = o;   o = align16(o + sizeof(float2) * kC2cPairs * (kC2cN + 1));
  L.total = o;
  return L;
}

template <typename Raw>
__device__ __forceinline__ float c2c_sample(const Raw* p) {
  if constexpr (sizeof(Raw) == 4) return *reinterpret_cast<const float*>(p);
  else if constexpr (std::is_same<Raw, short>::value) return (float)*p;  // int16 scale is in the window
  else return __half2float(*p);
}

template <int MODE>
__device__ __forceinline__ float c2c_power(float2 v, float pw) {
  const float m2 = fmaf(v.x, v.x, v.y * v.y);
  if constexpr (MODE == 0) return m2;
  else if constexpr (MODE == 1) return sqrtf(m2);
  else return powf(m2, 0.5f * pw);
}

template <int MODE, typename Raw>
__device__ __forceinline__ void run_tiles_c2c(const KernelParams& prm, unsigned char* smem,
                                              const SmemLayoutC2c& lay) {
  constexpr int P = kC2cP, Q = kC2cQ, N = kC2cN, GS = N + 1, PS = N / 2 + 1, G = 2 * kC2cPairs;
  constexpr int NWARPS = kC2cThreads / 32;
  const float2* s_tab = reinterpret_cast<const float2*>(smem + lay.tab);
  const float2* s_tw = reinterpret_cast<const float2*>(smem + lay.tw);
  const int4* s_mel = reinterpret_cast<const int4*>(smem + lay.mel);
  const float* s_mw = reinterpret_cast<const float*>(smem + lay.mel_w);
  float2* s_x = reinterpret_cast<float2*>(smem + lay.xbuf);
  float* s_pw = reinterpret_cast<float*>(smem + lay.xbuf);  // aliases s_x after the separation reads

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = tid % kC2cPairs, role = tid / kC2cPairs;
  const int hop = prm.hop, S = in_row_stride(hop), rows = in_rows(N, hop, G);
  const Raw* in = static_cast<const Raw*>(prm.in);
  const long long T = prm.T;
  const TileSplitter split(prm.tiles_per_signal);
  const PadSpec pads = {prm.zpad, prm.cpad, prm.pad_mode};
  auto in_buf = [&](int i) { return reinterpret_cast<Raw*>(smem + lay.in_tile + (size_t)i * lay.in_tile_bytes); };
  // buffer sizes for the debug build's index checks
  const Cap in_cap = {(int)(lay.in_tile_bytes / sizeof(Raw)), prm.err};
  const Cap x_cap = {kC2cPairs * GS, prm.err}, p_cap = {G * PS, prm.err};
  const long long out_total = prm.B * (long long)prm.n_mels * prm.n_frames;
  auto stage = [&](long long tile, int buf) {
    long long b;
    int tt;
    split(tile, b, tt);
    stage_tile<Raw, NWARPS>(in + b * T, T, (long long)tt * G * hop - prm.lead, rows, hop, S, in_buf(buf), warp,
                            lane, pads, in_cap);
    cp_async_commit();
  };

  long long tile = blockIdx.x;
  int buf = 0;
  if (tile < prm.total_tiles) stage(tile, 0);
  for (; tile < prm.total_tiles; tile += gridDim.x) {
    cp_async_wait_all();
    __syncthreads();  // this tile's samples are visible; the previous tile is fully done
    const long long next = tile + gridDim.x;
    if (next < prm.total_tiles) stage(next, buf ^ 1);

    // pass 1: z[p + P q] of frames g (real part) and g + 16 (imaginary part).
    // The two frames share one transform, so a frame past the signal's last
    // (in its last tile; its staged samples may be anything) contributes
    // exact zeros, chosen by select rather than multiplied away.
    long long b;
    int tt;
    split(tile, b, tt);
    const int t0 = tt * G;
    const bool va = t0 + g < prm.n_frames, vb = t0 + g + kC2cPairs < prm.n_frames;
    const Raw* fa = in_buf(buf) + g * S;
    const Raw* fb = fa + kC2cPairs * S;
    float2* xrow = s_x + g * GS;
    float2 z[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const float2 e = s_tab[role * Q + q];  // (window, offset of sample p + P q from the frame's row)
      const int o = __float_as_int(e.y);
      const bool in = FM_IN(g * S + o >= 0 && (g + kC2cPairs) * S + o < in_cap.n, prm.err);
      const float ya = in && va ? c2c_sample(fa + o) : 0.0f, yb = in && vb ? c2c_sample(fb + o) : 0.0f;
      z[q] = make_float2(ya * e.x, yb * e.x);
    }
    dft<Q>(z);
    put(xrow, g * GS, role, z[0], x_cap);
#pragma unroll
    for (int k2 = 1; k2 < Q; ++k2) put(xrow, g * GS, k2 * P + role, cmul(z[k2], s_tw[role * k2]), x_cap);
    __syncthreads();

    // pass 2: role t, k2 = t: Z[t + Q k1], back in natural order
    float2 y[P];
#pragma unroll
    for (int p = 0; p < P; ++p) y[p] = get(xrow, g * GS, role * P + p, x_cap);
    dft<P>(y);
    __syncthreads();  // every pass-1 value read before Z overwrites the row
#pragma unroll
    for (int k1 = 0; k1 < P; ++k1) put(xrow, g * GS, role + Q * k1, y[k1], x_cap);
    __syncthreads();

    // separation of the pairs (k, N - k), k = role + P i <= N / 2
    constexpr int PER = (N / 2) / P + 1;  // 11
    float pa[PER], pb[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int k = role + P * i;
      pa[i] = pb[i] = 0.0f;
      if (k <= N / 2) {
        const float2 zk = get(xrow, g * GS, k, x_cap);
        const float2 zm = get(xrow, g * GS, (N - k) % N, x_cap);
        pa[i] = c2c_power<MODE>(make_float2(zk.x + zm.x, zk.y - zm.y), prm.power);  // X_a[k]
        pb[i] = c2c_power<MODE>(make_float2(zk.x - zm.x, zk.y + zm.y), prm.power);  // i X_b[k]
      }
    }
    __syncthreads();  // every Z read before the power tile overwrites the buffer
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int k = role + P * i;
      if (k <= N / 2) {
        put(s_pw, 0, g * PS + k, pa[i], p_cap);
        put(s_pw, 0, (g + kC2cPairs) * PS + k, pb[i], p_cap);
      }
    }
    __syncthreads();

    const int n_valid = min(G, prm.n_frames - t0);
    const long long obase = b * prm.n_mels * (long long)prm.n_frames + t0;
    if (prm.out_dtype == FM_F32)
      mel_project<G, NWARPS, PS>(s_pw, s_mel, s_mw, static_cast<float*>(prm.out) + obase, n_valid, prm.n_mels,
                                 prm.n_frames, warp, lane, p_cap, prm.nnz, out_total - obase);
    else
      mel_project<G, NWARPS, PS>(s_pw, s_mel, s_mw, static_cast<__half*>(prm.out) + obase, n_valid, prm.n_mels,
                                 prm.n_frames, warp, lane, p_cap, prm.nnz, out_total - obase);
    buf ^= 1;
    // the next iteration's barrier orders these power-tile reads before the
    // next pass 1 overwrites the exchange buffer
  }
  cp_async_commit();  // nothing stays in flight past the end of the CTA
  cp_async_wait_all();
}

template <int N>
__global__ void __launch_bounds__(kC2cThreads) mel_kernel_c2c(const KernelParams prm) {
  static_assert(N == kC2cN, "the paired-frame kernel is built for n_fft 400");
  extern __shared__ __align__(16) unsigned char smem[];
  const int esize = prm.in_dtype == FM_F32 ? 4 : 2;
  const SmemLayoutC2c lay = smem_layout_c2c(prm.hop, prm.n_mels, prm.nnz, esize);
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  copy_table_async(smem + lay.tab, prm.c2c_tab, (int)sizeof(float2) * kC2cN, tid, kC2cThreads);
  copy_table_async(smem + lay.tw, prm.c2c_tw, (int)sizeof(float2) * kC2cN, tid, kC2cThreads);
  copy_table_async(smem + lay.mel, prm.mel, (int)sizeof(int4) * prm.n_mels, tid, kC2cThreads);
  copy_table_async(smem + lay.mel_w, prm.mel_w, (int)align16(sizeof(float) * (prm.nnz > 0 ? prm.nnz : 1)), tid,
                   kC2cThreads);
  pdl_wait();  // caller buffers only after the previous kernel in the stream is done
  // (the first barrier of the tile loop publishes the tables)
#define FM_C2C_RUN(MODE)                                                          \
  if (prm.in_dtype == FM_F32) run_tiles_c2c<MODE, float>(prm, smem, lay);          \
  else if (prm.in_dtype == FM_I16) run_tiles_c2c<MODE, short>(prm, smem, lay);     \
  else run_tiles_c2c<MODE, __half>(prm, smem, lay);
  if (prm.power_mode == 0) {
    FM_C2C_RUN(0)
  } else if (prm.power_mode == 1) {
    FM_C2C_RUN(1)
  } else {
    FM_C2C_RUN(2)
  }
#undef FM_C2C_RUN
}

}  // namespace fm
