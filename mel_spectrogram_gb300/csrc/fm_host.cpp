// Host-side plan tables, computed in double precision and rounded to float.
//
// flashmel 0.1.0, filters.py: make_window (periodic Hann, zero-padded and
// centred to n_fft) and pack_fbank (a triangular filter has contiguous
// support, so each row is stored as a start, a length and its weights). The
// filterbank follows torchaudio's melscale_fbanks, which that file calls; its
// formulas are the published HTK and Slaney mel scales.
#include <cmath>
#include <cstring>
#include <vector>

#include "fm_host.h"

namespace fm {

namespace {

constexpr double kTwoPi = 6.283185307179586476925286766559;

double hz_to_mel(double f, bool slaney) {
  if (!slaney) return 2595.0 * std::log10(1.0 + f / 700.0);
  const double f_sp = 200.0 / 3.0;  // Hz per mel below the break
  if (f < 1000.0) return f / f_sp;
  return 1000.0 / f_sp + std::log(f / 1000.0) * 27.0 / std::log(6.4);
}

double mel_to_hz(double m, bool slaney) {
  if (!slaney) return 700.0 * (std::pow(10.0, m / 2595.0) - 1.0);
  const double f_sp = 200.0 / 3.0;
  const double m_break = 1000.0 / f_sp;
  if (m < m_break) return m * f_sp;
  return 1000.0 * std::exp((m - m_break) * std::log(6.4) / 27.0);
}

}  // namespace

bool is_supported_nfft(int n_fft) {
  if (n_fft == 400) return true;
  for (int n = 64; n <= 16384; n *= 2)
    if (n == n_fft) return true;
  return false;
}

fm_status check_filter_args(int sr, int n_fft, int n_mels, double f_min, double* f_max, int mel_scale,
                            int norm) {
  if (sr <= 0 || n_fft < 2 || n_mels <= 0 || f_max == nullptr) return FM_ERR_INVALID_ARG;
  if (!(f_min >= 0.0) || !std::isfinite(f_min) || !std::isfinite(*f_max)) return FM_ERR_INVALID_ARG;
  if (mel_scale != FM_MEL_HTK && mel_scale != FM_MEL_SLANEY) return FM_ERR_INVALID_ARG;
  if (norm != FM_NORM_NONE && norm != FM_NORM_SLANEY) return FM_ERR_INVALID_ARG;
  const double nyq = 0.5 * (double)sr;
  if (*f_max <= 0.0) *f_max = nyq;
  if (*f_max > nyq * (1.0 + 1e-12) || *f_max <= f_min) return FM_ERR_INVALID_ARG;
  return FM_OK;
}

void build_filterbank(int sr, int n_fft, int n_mels, double f_min, double f_max, bool slaney,
                      bool slaney_norm, std::vector<int>& start, std::vector<int>& len,
                      std::vector<int>& off, std::vector<float>& weights) {
  const int n_freqs = n_fft / 2 + 1;
  // n_mels + 2 vertices equally spaced in mel between mel(f_min) and mel(f_max)
  const double m_lo = hz_to_mel(f_min, slaney), m_hi = hz_to_mel(f_max, slaney);
  std::vector<double> v(n_mels + 2);
  for (int i = 0; i < n_mels + 2; ++i) {
    const double m = (i == n_mels + 1) ? m_hi : m_lo + (m_hi - m_lo) * (double)i / (double)(n_mels + 1);
    v[i] = mel_to_hz(m, slaney);
  }
  start.assign(n_mels, 0);
  len.assign(n_mels, 0);
  off.assign(n_mels + 1, 0);
  weights.clear();
  std::vector<double> row(n_freqs);
  for (int m = 0; m < n_mels; ++m) {
    const double lo = v[m], mid = v[m + 1], hi = v[m + 2];
    const double scale = slaney_norm ? 2.0 / (hi - lo) : 1.0;
    int first = -1, last = -1;
    for (int k = 0; k < n_freqs; ++k) {
      const double f = (double)k * (double)sr / (double)n_fft;  // bin frequency
      const double up = (f - lo) / (mid - lo);
      const double down = (hi - f) / (hi - mid);
      double w = up < down ? up : down;
      if (!(w > 0.0)) w = 0.0;
      row[k] = w * scale;
      if (row[k] > 0.0) {
        if (first < 0) first = k;
        last = k;
      }
    }
    off[m] = (int)weights.size();
    if (first >= 0) {
      start[m] = first;
      len[m] = last - first + 1;
      for (int k = first; k <= last; ++k) weights.push_back((float)row[k]);
    }
  }
  off[n_mels] = (int)weights.size();
}

void build_window(int n_fft, int win_length, int normalized, std::vector<float>& window) {
  // periodic Hann of win_length samples, zero-padded and centred in n_fft;
  // times the STFT normalisation (1, 1/sqrt(sum w^2) or 1/sqrt(win_length),
  // flashmel filters.py make_window) and
  // times 1/2, the factor of the real-FFT split that the kernel leaves out.
  window.assign(n_fft, 0.0f);
  const int left = (n_fft - win_length) / 2;
  std::vector<double> w(win_length);
  double energy = 0.0;
  for (int n = 0; n < win_length; ++n) {
    w[n] = 0.5 - 0.5 * std::cos(kTwoPi * (double)n / (double)win_length);
    energy += w[n] * w[n];
  }
  double scale = 1.0;
  if (normalized == FM_NORMALIZED_WINDOW) scale = 1.0 / std::sqrt(energy);
  else if (normalized == FM_NORMALIZED_FRAME_LENGTH) scale = 1.0 / std::sqrt((double)win_length);
  for (int n = 0; n < win_length; ++n) window[left + n] = (float)(0.5 * scale * w[n]);
}

void build_twiddles(int len, int count, std::vector<float2>& tw) {
  // tw[j] = exp(-2 pi i j / len) stored (cos, -sin); j reduced exactly first
  tw.resize(count);
  for (int j = 0; j < count; ++j) {
    const double a = kTwoPi * (double)(j % len) / (double)len;
    tw[j].x = (float)std::cos(a);
    tw[j].y = (float)-std::sin(a);
  }
}

}  // namespace fm

extern "C" fm_status fm_mel_filterbank_csr(int sr, int n_fft, int n_mels, double f_min, double f_max,
                                           fm_mel_scale mel_scale, fm_norm norm, int32_t* start,
                                           int32_t* len, int32_t* off, float* weights, int64_t* nnz) {
  if (nnz == nullptr) return FM_ERR_INVALID_ARG;
  if (n_fft % 2 != 0) return FM_ERR_INVALID_ARG;
  fm_status st = fm::check_filter_args(sr, n_fft, n_mels, f_min, &f_max, mel_scale, norm);
  if (st != FM_OK) return st;
  std::vector<int> s, l, o;
  std::vector<float> w;
  fm::build_filterbank(sr, n_fft, n_mels, f_min, f_max, mel_scale == FM_MEL_SLANEY, norm == FM_NORM_SLANEY,
                       s, l, o, w);
  const int64_t cap = *nnz;
  *nnz = (int64_t)w.size();
  if (weights != nullptr && cap < (int64_t)w.size()) return FM_ERR_INVALID_ARG;
  if (start) std::memcpy(start, s.data(), sizeof(int32_t) * n_mels);
  if (len) std::memcpy(len, l.data(), sizeof(int32_t) * n_mels);
  if (off) std::memcpy(off, o.data(), sizeof(int32_t) * (n_mels + 1));
  if (weights && !w.empty()) std::memcpy(weights, w.data(), sizeof(float) * w.size());
  return FM_OK;
}
