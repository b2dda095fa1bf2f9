// Internal declarations shared by the C-ABI layer and the sm_103a kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fm_mel.h"

namespace fm {

// Everything one launch needs. Passed by value (it lives in the kernel's
// parameter constant bank), so the kernel reads it without global loads.
struct KernelParams {
  const void* in;  // [B][T] samples (f32 / int16 / f16)
  void* out;       // [B][n_mels][n_frames] (f32 / f16)
  long long B, T;
  int n_frames;
  int hop;
  int pad;  // n_fft / 2
  int in_dtype, out_dtype;
  int n_mels;
  int nnz;
  int power_mode;  // 0: |X|^2, 1: |X|, 2: general exponent
  float power;
  int tiles_per_signal;
  long long total_tiles;
  const float* window;    // n_fft, periodic Hann * 1/2 (the 1/2 of the real-FFT split)
  const float2* tw_half;  // W_{n_fft/2}^j, j < n_fft/2, stored (cos, -sin)
  const float2* tw_full;  // W_{n_fft}^k, k <= n_fft/2, stored (cos, -sin)
  const int* mel_start;   // n_mels
  const int* mel_len;     // n_mels
  const int* mel_off;     // n_mels (+1)
  const float* mel_w;     // nnz
  unsigned* err;          // device error word (FM_ERR_KERNEL_TIMEOUT etc.)
};

// Row stride (floats) of the staged input tile: rows hold `hop` samples; a
// stride of 2 (mod 4) floats makes the per-frame float2 reads of a half-warp
// fall on 16 distinct bank pairs.
__host__ __device__ inline int in_row_stride(int hop) { return hop + ((hop % 4 == 0) ? 2 : 0); }
__host__ __device__ inline int in_rows(int n_fft, int hop, int frames_per_tile) {
  return frames_per_tile + (n_fft - 1) / hop;
}

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// Dynamic shared-memory layout of one CTA, in bytes from the base.
struct SmemLayout {
  size_t window, tw_half, tw_full, mel_start, mel_len, mel_off, mel_w, in_tile, xbuf, total;
};

__host__ __device__ inline SmemLayout smem_layout(int n_fft, int hop, int n_mels, int nnz,
                                                  int frames_per_tile) {
  const int M = n_fft / 2;
  SmemLayout L;
  size_t o = 0;
  L.window = o;    o = align16(o + sizeof(float) * n_fft);
  L.tw_half = o;   o = align16(o + sizeof(float2) * M);
  L.tw_full = o;   o = align16(o + sizeof(float2) * (M + 1));
  L.mel_start = o; o = align16(o + sizeof(int) * n_mels);
  L.mel_len = o;   o = align16(o + sizeof(int) * n_mels);
  L.mel_off = o;   o = align16(o + sizeof(int) * n_mels);
  L.mel_w = o;     o = align16(o + sizeof(float) * (nnz > 0 ? nnz : 1));
  L.in_tile = o;   o = align16(o + sizeof(float) * (size_t)in_rows(n_fft, hop, frames_per_tile) * in_row_stride(hop));
  L.xbuf = o;      o = align16(o + sizeof(float2) * (size_t)frames_per_tile * (M + 1));
  L.total = o;
  return L;
}

// One compiled kernel: a fixed n_fft and its FFT split M = P * Q.
struct Variant {
  int n_fft;
  int P, Q;             // pass 1: P roles x Q-point DFTs; pass 2: Q x P-point DFTs
  int frames_per_tile;  // G: frames per tile = lanes per role
  int threads;          // P * G
  const void* fn;       // __global__ void(KernelParams)
};

const Variant* find_variant(int n_fft);

}  // namespace fm
