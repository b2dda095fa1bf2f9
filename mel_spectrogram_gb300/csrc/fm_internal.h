// Internal declarations shared by the C-ABI layer and the sm_103a kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fm_mel.h"

namespace fm {

// Index checks of the debug build (compiled with -DFM_BOUNDS_CHECK into
// libfm_mel_check.so). A guarded access is written `if (FM_IN(ok, err)) ...`
// with `ok` its index test against the buffer it touches: on a miss the
// kernel records FM_ERR_BOUNDS in the plan's error word (err) and skips the
// access, so a wrong index shows up as a status, never as a fault or a trap.
// In the normal build FM_IN is `true` and the tests compile away.
#ifdef FM_BOUNDS_CHECK
__device__ __forceinline__ bool fm_in_bounds(bool ok, unsigned* err) {
  if (!ok && err != nullptr) atomicExch(err, (unsigned)FM_ERR_BOUNDS);
  return ok;
}
#define FM_IN(ok, err) ::fm::fm_in_bounds((ok), (err))
#else
#define FM_IN(ok, err) true
#endif

// Everything one launch needs. Passed by value (it lives in the kernel's
// parameter constant bank), so the kernel reads it without global loads.
struct KernelParams {
  const void* in;  // [B][T] samples (f32 / int16 / f16)
  void* out;       // [B][n_mels][n_frames] (f32 / f16)
  long long B, T;
  int n_frames;
  int hop;
  // framing: frame t covers samples [t * hop - lead, t * hop - lead + n_fft)
  // of the signal; outside [0, T) the `zpad` zeros of torchaudio's `pad`, then
  // `cpad` centre-padding samples by pad_mode (FM_PAD_*), then nothing that a
  // valid frame reads
  int lead, zpad, cpad, pad_mode;
  int in_dtype, out_dtype;
  int n_mels;
  int nnz;
  int power_mode;  // 0: |X|^2, 1: |X|, 2: general exponent
  float power;
  int tiles_per_signal;
  long long total_tiles;
  // two-frames-per-thread kernel: slots [perm_t0, perm_t0 + perm_edges) take
  // the signals' first and last tiles and those tiles' slots take the tiles
  // displaced (0: every slot processes its own tile)
  int perm_edges;
  long long perm_t0;
  // pass-1 table, one float4 per (role p, q) at [p * Q + q]: the window at
  // samples 2n and 2n+1 (n = p + P q, times 1/2 for the real-FFT split and
  // times 2^-15 for int16 input) and, as int bits, the offset of sample 2n in
  // the staged tile relative to the frame's first row.
  const float4* p1;
  const float2* tw_half;  // W_{n_fft/2}^j, j < n_fft/2, stored (cos, -sin)
  const float2* tw_full;  // W_{n_fft}^k, k <= n_fft/2, stored (cos, -sin)
  const int4* mel;        // n_mels x {start, len, offset, 0}
  const float* mel_w;     // nnz
  const struct X2Tables* x2;  // two-frames-per-thread kernel only
  int x2_slots;               // its mel chunk slots (X2Tables::desc rows in use)
  unsigned* err;          // device error word (FM_ERR_KERNEL_TIMEOUT etc.)
  const float* win;       // the n_fft-point window (large-transform kernel only)
  int big_span;           // large-transform kernel: samples staged per tile in shared memory (0: none)
  int mel_taps;           // decimation-in-frequency large-transform kernel: 1 = a warp per filter with the
                          // lanes over its taps, 0 = a lane per filter and frame
  const float2* c2c_tab;  // paired-frame kernel: (window, tile offset) per role and step
  const float2* c2c_tw;   // paired-frame kernel: W_400^j, j < 400
  // Packed kernel: when tmap_ok, every signal is described to the TMA unit as
  // rows of one staged line (line * in_bytes / 8 elements of 8 bytes) that
  // start at sample tmap_off + y * line, tmap_rows rows per signal, and the
  // box is one whole staged tile at its padded row pitch (the pad columns lie
  // outside the rows and arrive zero-filled). An interior tile is then one
  // tensor copy.
  CUtensorMap tmap;  // 128-byte aligned by its type
  int tmap_ok, tmap_off, tmap_rows;
};

// Row stride (elements) of the staged input tile: rows hold `hop` samples; a
// stride of 2 (mod 4) elements makes the per-frame sample-pair reads of the
// lanes of a warp fall on distinct banks (float2 for f32, one word for
// 16-bit samples).
__host__ __device__ inline int in_row_stride(int hop) { return hop + ((hop % 4 == 0) ? 2 : 0); }
__host__ __device__ inline int in_rows(int n_fft, int hop, int frames_per_tile) {
  return frames_per_tile + (n_fft - 1) / hop;
}

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }
__host__ __device__ inline size_t align128(size_t x) { return (x + 127) & ~size_t(127); }

// Dynamic shared-memory layout of one CTA, in bytes from the base.
struct SmemLayout {
  size_t p1, tw_half, tw_full, mel, mel_w, in_tile, in_tile_bytes, xbuf, total;
};

__host__ __device__ inline SmemLayout smem_layout(int n_fft, int hop, int n_mels, int nnz, int frames_per_tile,
                                                  int in_esize, int n_in_buffers) {
  const int M = n_fft / 2;
  SmemLayout L;
  size_t o = 0;
  L.p1 = o;        o = align16(o + sizeof(float4) * M);
  L.tw_half = o;   o = align16(o + sizeof(float2) * M);
  L.tw_full = o;   o = align16(o + sizeof(float2) * (M + 1));
  L.mel = o;       o = align16(o + sizeof(int4) * n_mels);
  L.mel_w = o;     o = align16(o + sizeof(float) * (nnz > 0 ? nnz : 1));
  L.in_tile_bytes = align16((size_t)in_esize * in_rows(n_fft, hop, frames_per_tile) * in_row_stride(hop));
  L.in_tile = o;   o += L.in_tile_bytes * n_in_buffers;
  L.xbuf = o;      o = align16(o + sizeof(float2) * (size_t)frames_per_tile * (M + 1));
  L.total = o;
  return L;
}

// Constant tables of the two-frames-per-thread kernel, in one device block
// that each CTA copies into shared memory. Sized for n_fft <= 512 (M <= 256):
// every bin lies in at most two triangles, so nnz <= 2 (M + 1).
constexpr int kX2MaxM = 256;
constexpr int kX2MaxMels = 256;
constexpr int kX2MaxWarps = 16;
constexpr int kX2Unroll = 2;    // chunks per unrolled mel iteration
constexpr int kX2ProducerWarps = 1;  // the warp that stages every group's tiles
constexpr int kX2MaxSlots = 1024;  // mel chunk slots (4 chunks each) over all warps
struct X2Tables {
  float4 p1[kX2MaxM];        // as KernelParams::p1
  float4 tw_half[kX2MaxM];   // [p * Q + k2] = W_M^{p k2} as {c, c, d, d}, W = c + i d
  float4 tw_full[kX2MaxM + 1];
  // Mel work as four chunk streams per warp, one per quarter-warp. Every
  // filter is padded to an even length L >= 2 (zero weights; a run that would
  // pass bin M is shifted left) and cut into L/2 chunks of two bins; filters
  // are dealt to streams to balance their chunk counts, and the four streams
  // of warp w share slots [warp_begin[w], warp_begin[w + 1]), a multiple of
  // kX2Unroll long (padded with no-op chunks). Slot s, quarter h:
  //   desc[s][h] = {byte offset of the chunk's first bin row in the power
  //                 tile (bin * 128), filter index if the chunk ends its
  //                 filter (store and restart the sum), else -1};
  //   w4[s][h]   = {w0, w0, w1, w1}, the weights of the two bins.
  int warp_begin[kX2MaxWarps + 1];
  int2 desc[kX2MaxSlots][4];
  float4 w4[kX2MaxSlots][4];
};

// Line stride (elements) of the packed kernel's staged tile, for lines of
// `len` samples: each line starts on a 16-byte boundary (TMA bulk copies need
// it) and the stride is an odd multiple of 16 bytes. With 4-byte samples the
// frame starts of a half-warp's 16 lanes then fall on 8 distinct 16-byte bank
// groups, two lanes each, and the warp's two half-warps (8 bytes apart) read
// their 256 bytes in the minimum two wavefronts. That holds for lines of one
// hop (frame g on line g) and of two hops when the hop is a multiple of 32
// words (frames 2j and 2j + 1 on line j, 0 mod 32 banks apart). 2-byte
// samples take two wavefronts for 128 bytes either way.
__host__ __device__ constexpr int in_row_stride_x2_c(int len, int esize) {
  return ((((len + 16 / esize - 1) / (16 / esize)) | 1) * (16 / esize));
}
__host__ __device__ inline int in_row_stride_x2(int len, int esize) { return in_row_stride_x2_c(len, esize); }

// Layout of the two-frames-per-thread kernel (32-frame tiles): its tables
// (copied once per CTA from the X2Tables block) and the exchange buffer. The
// power tile occupies the lower half of the exchange buffer after pass 2, and
// the next tile's samples are staged into the upper half meanwhile, so a CTA
// needs no separate input buffer (when a tile fits there; otherwise one is
// appended).
struct SmemLayoutX2 {
  // group g's "tile staged" mbarrier at bars + 8 g and its "staging area free"
  // mbarrier at bars + 8 (groups + g); the (signal, tile in signal) of its
  // k-th tile at slots + 8 (2 g + k % 2), written by the producer; its
  // exchange buffer at xbuf + g group_stride and its staged tile at
  // in_tile + g group_stride
  size_t bars, slots, p1, tw_half, tw_full, desc, w4, xbuf, in_tile, in_tile_bytes, group_stride, total;
};

// Staged lines of the packed kernel: k_hops hops of samples per line (2 for
// a compile-time hop, else 1), `lines` of them per 32-frame tile.
__host__ __device__ inline int x2_lines(int n_fft, int hop, int k_hops) {
  return (in_rows(n_fft, hop, 32) + k_hops - 1) / k_hops;
}

// n_slots: mel chunk slots (four chunks each); groups: tile groups per CTA,
// which share the tables and own one exchange buffer (and tile) each
__host__ __device__ inline SmemLayoutX2 smem_layout_x2(int n_fft, int hop, int k_hops, int n_slots, int in_esize,
                                                       int groups) {
  const int M = n_fft / 2;
  const int ns = n_slots > 0 ? n_slots : 1;
  SmemLayoutX2 L;
  size_t o = 0;
  L.bars = o;      o = o + sizeof(unsigned long long) * 2 * groups;
  L.slots = o;     o = align16(o + sizeof(int2) * 2 * groups);
  L.p1 = o;        o = align16(o + sizeof(float4) * M);
  L.tw_half = o;   o = align16(o + sizeof(float4) * M);
  L.tw_full = o;   o = align16(o + sizeof(float4) * (M + 1));
  L.desc = o;      o = align16(o + sizeof(int2) * 4 * ns);
  L.w4 = o;        o = align16(o + sizeof(float4) * 4 * ns);
  // staging areas start on 128-byte boundaries (tensor TMA destinations)
  const size_t xq_bytes = align128(sizeof(float4) * 16 * (size_t)(M + 1));
  const size_t half = align128(xq_bytes / 2);  // >= the power tile, (M + 1) bins x 16 lanes x float2
  o = align128(o);
  L.xbuf = o;
  L.in_tile_bytes =
      align128((size_t)in_esize * x2_lines(n_fft, hop, k_hops) * in_row_stride_x2(k_hops * hop, in_esize));
  if (L.in_tile_bytes <= xq_bytes - half) {
    L.in_tile = L.xbuf + half;
    L.group_stride = xq_bytes;
  } else {
    L.in_tile = L.xbuf + xq_bytes;
    L.group_stride = xq_bytes + L.in_tile_bytes;
  }
  L.total = L.xbuf + groups * L.group_stride;
  return L;
}

// One compiled kernel: a fixed n_fft and its FFT split M = P * Q.
struct Variant {
  int n_fft;
  int P, Q;             // pass 1: P roles x Q-point DFTs; pass 2: Q x P-point DFTs (kind 2: P = 16, Q = M / 16
                        // for the decimation-in-frequency build, 0 for the three-pass build)
  int frames_per_tile;  // G: frames per tile = lanes per role
  int threads;          // P * G
  int in_buffers;       // 2: the next tile's input lands while this one computes
  int kind;             // 0: one frame per thread; 1: two frames per thread (packed); 2: shared-memory passes;
                        // 3: one complex transform per frame pair
  const void* fn;       // __global__ void(KernelParams)
  int hop;              // > 0: compiled for this hop only; else kEvenHops, kOddHops or kAnyHop
  int groups;           // kinds 1 and 2: independent tile groups per CTA; else 0
};

// Variant::hop values other than a compiled-in hop
constexpr int kEvenHops = 0;   // any even hop (samples staged and read in aligned pairs)
constexpr int kOddHops = -1;   // any odd hop (contiguous staging, pairs read as two samples)
constexpr int kAnyHop = -2;    // any hop (the large-transform kernel reads single samples)

// The kernels for (n_fft, hop) in order of preference (a hop-specialised build
// first): the first one, or with `after` the one that follows it; nullptr
// when there is none left. The plan takes the first whose shared memory fits.
const Variant* find_variant(int n_fft, int hop, const Variant* after = nullptr);

}  // namespace fm
