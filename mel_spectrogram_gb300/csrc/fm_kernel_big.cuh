// Mel kernel for the large transforms (n_fft = 4096, 8192, 16384; sm_103a),
// and for n_fft 1024 and 2048 at hops too long for the one-frame kernel.
//
// Same path as the other kernels (padding and framing as index arithmetic,
// periodic Hann, real DFT through the complex M = n_fft/2 point DFT of
// z[n] = (y[2n] + i y[2n+1]) / 2 and its split, |X|^p, sparse mel projection),
// but a frame's M complex values no longer fit one thread's registers, so the
// complex DFT runs in shared memory as three mixed-radix autosorting
// (Stockham) passes over a tile of F frames:
//   load   : the windowed pairs z[n] of F consecutive frames, straight from
//            the signal (coalesced; edge frames through padded_source);
//   passes : radix R0, R1, R2 with M = R0 R1 R2. Pass i, with Ns the
//            product of the earlier radices, takes the R values
//            x[j + r M/R] of butterfly j, multiplies value r by
//            W_{Ns R}^{(j mod Ns) r}, does an R-point DFT in registers and
//            writes value r to x[(j / Ns) Ns R + (j mod Ns) + r Ns]; after the
//            last pass x holds Z[k] in natural order. Every thread holds all
//            its butterflies of a pass in registers (32 complex values), so a
//            pass is loads, barrier, stores, barrier, in place;
//   split  : X[k], X[M-k] from Z[k], Z[M-k] and W_N^k, |X|^p into a power
//            tile that aliases the buffer;
//   mel    : the CSR projection, lane = frame.
// A CTA holds 16 K complex values (32768 / n_fft frames), 139 KB of shared
// memory with one float2 of padding per 16 (strided accesses spread over the
// banks). With GB tile groups the CTA's threads and buffer split into GB
// groups that run their own tiles (32768 / n_fft / GB frames) on their own
// named barrier, sharing the twiddle rows and the filterbank; GB = 1 is one
// group of the whole CTA. Twiddles (float64-built tables) and the window are read
// from global memory through the read-only cache.
#pragma once

#include "fm_kernel.cuh"

namespace fm {

constexpr int kBigThreads = 512;

// Radices of the three autosorting passes, M = R0 R1 R2.
template <int M>
struct BigRadices;
template <>
struct BigRadices<512> {
  static constexpr int R0 = 8, R1 = 8, R2 = 8;
};
template <>
struct BigRadices<1024> {
  static constexpr int R0 = 16, R1 = 16, R2 = 4;
};
template <>
struct BigRadices<2048> {
  static constexpr int R0 = 16, R1 = 16, R2 = 8;
};
template <>
struct BigRadices<4096> {
  static constexpr int R0 = 16, R1 = 16, R2 = 16;
};
template <>
struct BigRadices<8192> {
  static constexpr int R0 = 16, R1 = 16, R2 = 32;
};

// frames per tile (F M = 16 K complex values per tile)
__host__ __device__ constexpr int big_frames(int n_fft) { return 32768 / n_fft; }
// float2 slots per frame in shared memory: M values, one pad per 16, one more
__host__ __device__ constexpr int big_frame_stride(int M) { return M + (M >> 4) + 1; }
__host__ __device__ constexpr size_t big_smem_bytes(int n_fft) {
  return sizeof(float2) * (size_t)big_frames(n_fft) * (size_t)big_frame_stride(n_fft / 2);
}
// The decimation-in-frequency build (mel_kernel_bigdif) keeps a tile as 16
// sub-frames of M/16 values per frame, each with its own padding.
constexpr int kDifR0 = 16;
__host__ __device__ constexpr size_t big_dif_smem_bytes(int n_fft) {
  return sizeof(float2) * (size_t)big_frames(n_fft) * kDifR0 * (size_t)big_frame_stride(n_fft / 2 / kDifR0);
}
// Twiddles from shared memory in two levels, W^t = W^(t mod 64) W^(64 floor(t / 64)):
// rows of 64 fine and M/64 (+1) coarse factors of W_M (the passes) and of W_N
// (the split), gathered from the plan's full tables when a CTA starts. A full
// table (64 KB at n_fft 16384) would not stay in L1 beside the transform.
constexpr int kBigTwFine = 64;
__host__ __device__ constexpr int big_tw_count(int M) { return 2 * kBigTwFine + M / kBigTwFine + M / kBigTwFine + 1; }

// Shared memory of the large-transform kernel after the transform buffer:
// the twiddle rows, the filterbank (descriptors and weights) and, when one
// tile's span fits, the staging buffer of the next tile's samples.
struct BigLayout {
  size_t tw, mel, mw, st;
};
__host__ __device__ inline BigLayout big_layout(int n_fft, int n_mels, int nnz, bool dif = false) {
  BigLayout L;
  size_t o = dif ? big_dif_smem_bytes(n_fft) : big_smem_bytes(n_fft);
  L.tw = o;   o = align16(o + sizeof(float2) * big_tw_count(n_fft / 2));
  L.mel = o;  o = align16(o + sizeof(int4) * n_mels);
  L.mw = o;   o = align16(o + sizeof(float) * (nnz > 0 ? nnz : 1));
  L.st = o;
  return L;
}

// Samples a tile of F frames covers, (F - 1) hop + n_fft: the span the kernel
// prefetches into a staging buffer (one per group) after the tables when it
// fits (KernelParams::big_span), 16-byte aligned.
__host__ __device__ constexpr long long big_span(int F, int n_fft, int hop) {
  return (long long)(F - 1) * hop + n_fft;
}
__host__ __device__ constexpr size_t big_staging_bytes(int F, int n_fft, int hop, int esize) {
  return (size_t)((big_span(F, n_fft, hop) * esize + 15) / 16 * 16);
}
// barrier over one tile group of n threads: the CTA barrier when the group is
// the whole CTA, a warp barrier when it is one warp, else named barrier `id`
__device__ __forceinline__ void big_sync(int id, int n) {
  if (n == kBigThreads) __syncthreads();
  else if (n == 32) __syncwarp();
  else asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ int big_phys(int i) { return i + (i >> 4); }

__device__ __forceinline__ float raw_to_float(float v) { return v; }
__device__ __forceinline__ float raw_to_float(short v) { return (float)v; }
__device__ __forceinline__ float raw_to_float(__half v) { return __half2float(v); }

// sample at padded position s of one signal (index arithmetic, zero where
// padded_source says so)
template <typename Raw>
__device__ __forceinline__ float big_sample(const Raw* __restrict__ sig, long long T, long long s, const PadSpec& ps) {
  const long long src = padded_source(s, T, ps);
  return src < 0 ? 0.0f : raw_to_float(sig[src]);
}

// Windowed pairs of F frames: frame f starts at signal index s0 + f hop;
// z[n] = (y[2n], y[2n+1]) times (w[2n], w[2n+1]) (the window carries the 1/2 of
// the split, the STFT normalisation and the int16 scale).
// Every global load of the tile is issued before the first one is used (the
// loop has a compile-time trip count), so the tile waits for one memory
// latency rather than one per few pairs.
template <int N, int F, int TH, typename Raw>
__device__ __forceinline__ void big_load(float2* s_x, const Raw* __restrict__ sig, long long T, long long s0,
                                         int hop, const float2* __restrict__ win2, const PadSpec& ps, int tid,
                                         Cap x_cap) {
  constexpr int M = N / 2, FS = big_frame_stride(M);
  constexpr int PER = F * M / TH;
  static_assert((F * M) % TH == 0, "pairs must divide evenly over the threads");
  const bool interior = s0 >= 0 && s0 + (long long)(F - 1) * hop + N <= T;
  float2 v[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int idx = tid + i * TH, f = idx / M, n = idx % M;
    const long long s = s0 + (long long)f * hop + 2 * n;
    if (interior) {
      v[i] = FM_IN(s >= 0 && s + 1 < T, x_cap.err) ? make_float2(raw_to_float(sig[s]), raw_to_float(sig[s + 1]))
                                                   : make_float2(0.0f, 0.0f);
    } else {
      v[i] = make_float2(big_sample(sig, T, s, ps), big_sample(sig, T, s + 1, ps));
    }
  }
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int idx = tid + i * TH, f = idx / M, n = idx % M;
    const float2 w = __ldg(win2 + n);
    put(s_x, 0, f * FS + big_phys(n), make_float2(v[i].x * w.x, v[i].y * w.y), x_cap);
  }
}

// The same from a staging buffer that holds the tile's padded samples
// (st[i] = the sample at padded position s0 + i, see stage_run).
template <int N, int F, int TH, typename Raw>
__device__ __forceinline__ void big_load_staged(float2* s_x, const Raw* st, int hop, const float2* __restrict__ win2,
                                                int tid, Cap x_cap, Cap st_cap) {
  constexpr int M = N / 2, FS = big_frame_stride(M);
  constexpr int PER = F * M / TH;
#pragma unroll 8
  for (int i = 0; i < PER; ++i) {
    const int idx = tid + i * TH, f = idx / M, n = idx % M;
    const Raw* p = st + f * hop + 2 * n;
    const float2 w = __ldg(win2 + n);
    const float2 v = FM_IN(f * hop + 2 * n + 1 < st_cap.n, st_cap.err) ? make_float2(raw_to_float(p[0]), raw_to_float(p[1]))
                                                                      : make_float2(0.0f, 0.0f);
    put(s_x, 0, f * FS + big_phys(n), make_float2(v.x * w.x, v.y * w.y), x_cap);
  }
}

// One radix-R autosorting pass over the F frames (Ns = product of the
// earlier radices).
// W_M^t from the two twiddle rows of W_M (fine: t mod 64, coarse: t / 64)
template <int M>
__device__ __forceinline__ float2 big_tw(const float2* s_tw, int t) {
  return cmul(s_tw[t & (kBigTwFine - 1)], s_tw[kBigTwFine + (t >> 6)]);
}

// TWS: the rows hold W_{TWS M} (a sub-transform of M points reads W_M^t as
// W_{TWS M}^{TWS t}).
template <int M, int F, int TH, int R, int NS, int TWS = 1>
__device__ __forceinline__ void big_pass(float2* s_x, const float2* s_tw, int tid, int bar, Cap x_cap) {
  constexpr int J = M / R;  // butterflies per frame
  constexpr int FS = big_frame_stride(M);
  static_assert((F * J) % TH == 0, "butterflies must divide evenly over the threads");
  constexpr int TASKS = F * J / TH;
  float2 v[TASKS][R];
#pragma unroll
  for (int t = 0; t < TASKS; ++t) {
    const int task = tid + t * TH;
    const int f = task / J, j = task % J;
    const float2* xf = s_x + f * FS;
#pragma unroll
    for (int r = 0; r < R; ++r) v[t][r] = get<float2>(xf, f * FS, big_phys(j + r * J), x_cap);
    if constexpr (NS > 1) {
      const int e = (j % NS) * (M / (NS * R));  // W_{Ns R}^{(j mod Ns) r} = W_M^{e r}, e r < M
#pragma unroll
      for (int r = 1; r < R; ++r) v[t][r] = cmul(v[t][r], big_tw<M>(s_tw, e * r * TWS));
    }
    dft<R>(v[t]);
  }
  big_sync(bar, TH);  // every read of this pass before any write
#pragma unroll
  for (int t = 0; t < TASKS; ++t) {
    const int task = tid + t * TH;
    const int f = task / J, j = task % J;
    float2* xf = s_x + f * FS;
    const int d = (j / NS) * NS * R + (j % NS);
#pragma unroll
    for (int r = 0; r < R; ++r) put(xf, f * FS, big_phys(d + r * NS), v[t][r], x_cap);
  }
  big_sync(bar, TH);
}

// Real-FFT split and |X|^p for k = 0 .. M/2 of every frame, into the power
// tile (float rows of M + 1, aliasing the buffer: all reads, barrier, writes).
template <int M, int F, int TH, int MODE>
__device__ __forceinline__ void big_split(float2* s_x, float* s_pw, const float2* s_twn, float pw, int tid, int bar,
                                          Cap x_cap, Cap p_cap) {
  constexpr int FS = big_frame_stride(M), PS = M + 1;
  constexpr int PAIRS = M / 2 + 1, TOTAL = F * PAIRS;
  constexpr int PER = (TOTAL + TH - 1) / TH;
  float lo[PER], hi[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int task = tid + i * TH;
    lo[i] = hi[i] = 0.0f;
    if (task < TOTAL) {
      const int f = task / PAIRS, k = task % PAIRS;
      const float2 zk = get<float2>(s_x, 0, f * FS + big_phys(k), x_cap);
      const float2 zm = get<float2>(s_x, 0, f * FS + big_phys((M - k) & (M - 1)), x_cap);
      // W_N^k from the two twiddle rows of W_N
      const float2 w = cmul(s_twn[k & (kBigTwFine - 1)], s_twn[kBigTwFine + (k >> 6)]);
      split_pair<MODE>(zk, zm, w, pw, lo[i], hi[i]);
    }
  }
  big_sync(bar, TH);
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int task = tid + i * TH;
    if (task < TOTAL) {
      const int f = task / PAIRS, k = task % PAIRS;
      put(s_pw, 0, f * PS + k, lo[i], p_cap);
      put(s_pw, 0, f * PS + M - k, hi[i], p_cap);
    }
  }
  big_sync(bar, TH);
}

// Sum over the warp of each of acc[0 .. V-1] (V a power of two <= 32):
// steps over lane offsets 16, 8, ... first halve the values a lane holds (the
// lanes with the offset bit set keep the upper half, the others the lower,
// each adding its partner's copy), then the remaining offsets sum one value.
// Afterwards lane v (32 / V) holds the sum of acc[v]; V - 1 + 5 - log2(V)
// shuffles in a chain five deep.
template <int V>
__device__ __forceinline__ float warp_sum_each(float (&acc)[V], int lane) {
  static_assert(V >= 1 && V <= 32 && (V & (V - 1)) == 0, "V a power of two");
  int o = 16;
#pragma unroll
  for (int n = V; n > 1; n >>= 1, o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float give = up ? acc[i] : acc[i + n / 2];
      const float keep = up ? acc[i + n / 2] : acc[i];
      acc[i] = keep + __shfl_xor_sync(0xffffffffu, give, o);
    }
  }
#pragma unroll
  for (; o >= 1; o >>= 1) acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], o);
  return acc[0];
}

// Sparse mel projection with the lanes over a filter's taps: filter m goes to
// warp m mod NWARPS (filter widths grow with m, so every warp gets a like
// share of the taps); its taps are read 32 at a time (consecutive bins and
// weights, no bank conflicts), each lane keeping one partial sum per frame,
// and warp_sum_each adds them up; lane f (32 / F) stores frame f. The cost of
// a filter is its ceil(taps / 32) loads plus a shuffle sum, against the
// widest filter's taps one by one when a lane holds a filter
// (mel_project_lanes), which is why the plan picks between the two from the
// filter widths. p_cap, nnz, out_left: as mel_project.
template <int F, int NWARPS, int PS, typename OutT>
__device__ __forceinline__ void mel_project_taps(const float* s_pw, const int4* __restrict__ s_mel,
                                                 const float* __restrict__ s_mw, OutT* out_tile, int n_valid,
                                                 int n_mels, long long n_frames, int warp, int lane, Cap p_cap,
                                                 int nnz, long long out_left) {
  constexpr int L = 32 / F;
  const int f_out = lane / L;
  const bool writer = lane % L == 0 && f_out < n_valid;
  for (int m = warp; m < n_mels; m += NWARPS) {
    const int4 md = s_mel[m];
    float acc[F];
#pragma unroll
    for (int f = 0; f < F; ++f) acc[f] = 0.0f;
    for (int j = lane; j < md.y; j += 32) {
      const float w = FM_IN(md.z + j >= 0 && md.z + j < nnz, p_cap.err) ? s_mw[md.z + j] : 0.0f;
#pragma unroll
      for (int f = 0; f < F; ++f) acc[f] = fmaf(w, get(s_pw, 0, f * PS + md.x + j, p_cap), acc[f]);
    }
    const float sum = warp_sum_each<F>(acc, lane);
    if (writer && FM_IN(f_out + (long long)m * n_frames < out_left, p_cap.err))
      store_out(out_tile + (long long)m * n_frames + f_out, sum);
  }
}

// Sparse mel projection with a lane per filter and frame (the mapping of
// mel_project), its taps read eight ahead into registers and summed into two
// partial sums, so that the widest filter's lane waits for one shared-memory
// latency per eight taps rather than per tap.
template <int G, int NWARPS, int PS, typename OutT>
__device__ __forceinline__ void mel_project_lanes(const float* s_pw, const int4* __restrict__ s_mel,
                                                  const float* __restrict__ s_mw, OutT* out_tile, int n_valid,
                                                  int n_mels, long long n_frames, int warp, int lane, Cap p_cap,
                                                  int nnz, long long out_left) {
  constexpr int SUBS = 32 / G;
  const int gg = lane % G, sub = lane / G;
  const int poff = gg * PS;
  const bool valid = gg < n_valid;
  for (int m = warp * SUBS + sub; m < n_mels; m += NWARPS * SUBS) {
    const int4 md = s_mel[m];
    float a0 = 0.0f, a1 = 0.0f;
    int j = 0;
    for (; j + 8 <= md.y; j += 8) {
      float w[8], p[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        w[u] = FM_IN(md.z + j + u >= 0 && md.z + j + u < nnz, p_cap.err) ? s_mw[md.z + j + u] : 0.0f;
        p[u] = get(s_pw, 0, poff + md.x + j + u, p_cap);
      }
#pragma unroll
      for (int u = 0; u < 8; u += 2) {
        a0 = fmaf(w[u], p[u], a0);
        a1 = fmaf(w[u + 1], p[u + 1], a1);
      }
    }
    for (; j < md.y; ++j) {
      const float w = FM_IN(md.z + j >= 0 && md.z + j < nnz, p_cap.err) ? s_mw[md.z + j] : 0.0f;
      a0 = fmaf(w, get(s_pw, 0, poff + md.x + j, p_cap), a0);
    }
    if (valid && FM_IN(gg + (long long)m * n_frames < out_left, p_cap.err))
      store_out(out_tile + (long long)m * n_frames + gg, a0 + a1);
  }
}

// The tile loop of group grp (tid: the thread within the group): tiles
// blockIdx.x + gridDim.x * (grp + GB k) of F = 32768 / n_fft / GB frames, on
// the group's share of the transform buffer and its named barrier 1 + grp.
template <int N, int GB, typename Raw>
__device__ __forceinline__ void run_tiles_big(const KernelParams& prm, unsigned char* smem, int grp, int tid) {
  constexpr int M = N / 2, F = big_frames(N) / GB, TH = kBigThreads / GB, NWARPS = TH / 32;
  constexpr int R0 = BigRadices<M>::R0, R1 = BigRadices<M>::R1, R2 = BigRadices<M>::R2;
  static_assert(R0 * R1 * R2 == M && F * GB == big_frames(N) && TH % 32 == 0, "radices, frames and groups");
  float2* s_x = reinterpret_cast<float2*>(smem) + (size_t)grp * F * big_frame_stride(M);
  float* s_pw = reinterpret_cast<float*>(s_x);
  const int warp = tid >> 5, lane = tid & 31, bar = 1 + grp;
  const Raw* in = static_cast<const Raw*>(prm.in);
  const float2* win2 = reinterpret_cast<const float2*>(prm.win);
  const long long T = prm.T;
  const TileSplitter split(prm.tiles_per_signal);
  const PadSpec pads = {prm.zpad, prm.cpad, prm.pad_mode};
  // With staging buffers (prm.big_span > 0), the next tile's samples are
  // prefetched by cp.async while this tile's transform runs.
  const BigLayout lay = big_layout(N, prm.n_mels, prm.nnz);
  const float2* s_tw = reinterpret_cast<const float2*>(smem + lay.tw);  // W_M rows, then W_N rows
  const float2* s_twn = s_tw + kBigTwFine + M / kBigTwFine;
  const int4* s_mel = reinterpret_cast<const int4*>(smem + lay.mel);
  const float* s_mw = reinterpret_cast<const float*>(smem + lay.mw);
  const int span = prm.big_span;
  Raw* s_st = reinterpret_cast<Raw*>(smem + lay.st + (size_t)grp * ((span * sizeof(Raw) + 15) / 16 * 16));
  // buffer sizes for the debug build's index checks (the staging buffer holds
  // span samples, rounded up to 16 bytes)
  const Cap x_cap = {F * big_frame_stride(M), prm.err}, p_cap = {F * (M + 1), prm.err};
  const Cap st_cap = {span, prm.err};
  const long long out_total = prm.B * (long long)prm.n_mels * prm.n_frames;
  const long long first = (long long)blockIdx.x + (long long)gridDim.x * grp, stride = (long long)gridDim.x * GB;
  auto prefetch = [&](long long t) {
    long long bb;
    int tq;
    split(t, bb, tq);
    stage_run<Raw>(in + bb * T, T, (long long)tq * F * prm.hop - prm.lead, span, s_st, tid, TH, pads, st_cap);
    cp_async_commit();
  };
  if (span > 0 && first < prm.total_tiles) prefetch(first);
  for (long long tile = first; tile < prm.total_tiles; tile += stride) {
    long long b;
    int tt;
    split(tile, b, tt);
    const int t0 = tt * F;
    if (span > 0) cp_async_wait_all();  // this thread's copies of the tile have landed
    big_sync(bar, TH);  // the previous tile's mel reads are done; the staged tile is visible
    if (span > 0)
      big_load_staged<N, F, TH, Raw>(s_x, s_st, prm.hop, win2, tid, x_cap, st_cap);
    else
      big_load<N, F, TH, Raw>(s_x, in + b * T, T, (long long)t0 * prm.hop - prm.lead, prm.hop, win2, pads, tid,
                              x_cap);
    big_sync(bar, TH);
    if (span > 0 && tile + stride < prm.total_tiles) prefetch(tile + stride);  // staging read: reuse it
    big_pass<M, F, TH, R0, 1>(s_x, s_tw, tid, bar, x_cap);
    big_pass<M, F, TH, R1, R0>(s_x, s_tw, tid, bar, x_cap);
    big_pass<M, F, TH, R2, R0 * R1>(s_x, s_tw, tid, bar, x_cap);
    switch (prm.power_mode) {
      case 0: big_split<M, F, TH, 0>(s_x, s_pw, s_twn, prm.power, tid, bar, x_cap, p_cap); break;
      case 1: big_split<M, F, TH, 1>(s_x, s_pw, s_twn, prm.power, tid, bar, x_cap, p_cap); break;
      default: big_split<M, F, TH, 2>(s_x, s_pw, s_twn, prm.power, tid, bar, x_cap, p_cap); break;
    }
    const int n_valid = min(F, prm.n_frames - t0);
    const long long obase = b * prm.n_mels * (long long)prm.n_frames + t0;
    if (prm.out_dtype == FM_F32)
      mel_project<F, NWARPS, M + 1>(s_pw, s_mel, s_mw, static_cast<float*>(prm.out) + obase, n_valid,
                                    prm.n_mels, prm.n_frames, warp, lane, p_cap, prm.nnz, out_total - obase);
    else
      mel_project<F, NWARPS, M + 1>(s_pw, s_mel, s_mw, static_cast<__half*>(prm.out) + obase, n_valid,
                                    prm.n_mels, prm.n_frames, warp, lane, p_cap, prm.nnz, out_total - obase);
  }
  cp_async_wait_all();  // nothing stays in flight past the end of the CTA
}

// The plan's tables, once per CTA (the grid is persistent): the twiddle rows
// gathered from the full W_M and W_N tables, and the filterbank; then the
// wait for the previous kernel in the stream and a CTA barrier.
template <int N>
__device__ __forceinline__ void big_tables(const KernelParams& prm, unsigned char* smem, const BigLayout& lay,
                                           int tid) {
  constexpr int M = N / 2, ROWS = M / kBigTwFine;
  float2* s_tw = reinterpret_cast<float2*>(smem + lay.tw);
  for (int i = tid; i < kBigTwFine; i += kBigThreads) {
    s_tw[i] = prm.tw_half[i];                             // W_M^i
    s_tw[kBigTwFine + ROWS + i] = prm.tw_full[i];         // W_N^i
  }
  for (int i = tid; i < ROWS; i += kBigThreads) s_tw[kBigTwFine + i] = prm.tw_half[kBigTwFine * i];  // W_M^(64 i)
  for (int i = tid; i <= ROWS; i += kBigThreads)
    s_tw[2 * kBigTwFine + ROWS + i] = prm.tw_full[kBigTwFine * i];  // W_N^(64 i), 64 i <= M
  copy_table_async(smem + lay.mel, prm.mel, (int)sizeof(int4) * prm.n_mels, tid, kBigThreads);
  copy_table_async(smem + lay.mw, prm.mel_w, (int)align16(sizeof(float) * (prm.nnz > 0 ? prm.nnz : 1)), tid,
                   kBigThreads);
  cp_async_commit();
  cp_async_wait_all();
  pdl_wait();  // caller buffers only after the previous kernel in the stream is done
  __syncthreads();  // the tables are visible to every group
}

template <int N, int GB>
__global__ void __launch_bounds__(kBigThreads, 1) mel_kernel_big(const KernelParams prm) {
  extern __shared__ __align__(16) unsigned char smem[];
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  big_tables<N>(prm, smem, big_layout(N, prm.n_mels, prm.nnz), tid);
  constexpr int TH = kBigThreads / GB;
  const int grp = GB == 1 ? 0 : __shfl_sync(0xffffffffu, tid / TH, 0), gtid = tid % TH;
  if (prm.in_dtype == FM_F32) run_tiles_big<N, GB, float>(prm, smem, grp, gtid);
  else if (prm.in_dtype == FM_I16) run_tiles_big<N, GB, short>(prm, smem, grp, gtid);
  else run_tiles_big<N, GB, __half>(prm, smem, grp, gtid);
}

}  // namespace fm

// Instantiate one large-transform variant: FM_DEFINE_VARIANT_BIG(name, N, GB),
// GB tile groups per CTA
#define FM_DEFINE_VARIANT_BIG(NAME, N, GB)                                                            \
  namespace fm {                                                                                      \
  template __global__ void mel_kernel_big<N, GB>(const KernelParams);                                \
  extern const Variant NAME = {N, 0, 0, big_frames(N) / GB, kBigThreads, 0, 2,                        \
                               (const void*)&mel_kernel_big<N, GB>, kAnyHop, GB};                     \
  }
