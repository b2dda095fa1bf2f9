// Host-side table builders (double precision) used by the plan.
#pragma once

#include <cuda_runtime.h>

#include <vector>

#include "fm_mel.h"

namespace fm {

bool is_supported_nfft(int n_fft);

// Validates the filterbank arguments; f_max <= 0 is replaced by sr / 2.
fm_status check_filter_args(int sr, int n_fft, int n_mels, double f_min, double* f_max, int mel_scale,
                            int norm);

// Per-filter CSR of the triangular mel filterbank over bins k * sr / n_fft.
void build_filterbank(int sr, int n_fft, int n_mels, double f_min, double f_max, bool slaney,
                      bool slaney_norm, std::vector<int>& start, std::vector<int>& len,
                      std::vector<int>& off, std::vector<float>& weights);

// Periodic Hann (times 1/2 and the fm_normalized scale), zero-padded and
// centred to n_fft.
void build_window(int n_fft, int win_length, int normalized, std::vector<float>& window);

// tw[j] = exp(-2 pi i j / len), j < count, stored (cos, -sin).
void build_twiddles(int len, int count, std::vector<float2>& tw);

// The plan's device error word (the one fm_plan_poll_error reads), for the
// diagnostic kernels of the library; NULL for a NULL plan.
unsigned* plan_error_word(const fm_plan* plan);

}  // namespace fm
