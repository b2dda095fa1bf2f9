"""The oracle against its pins, and planted mistakes against the pins.

A pin only counts if a plausible mistake in the oracle would fail it, so the
second half plants such mistakes in a copy of the oracle (on the CPU) and
checks that at least one pin rejects each.
"""
from __future__ import annotations

import importlib.util
import math
import sys

import numpy as np
import pytest

import oracle.mel_oracle as real_oracle
from tests import oracle_pins as pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(real_oracle)


def _fresh_oracle():
    spec = importlib.util.spec_from_file_location("oracle_mutant", real_oracle.__file__)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _symmetric_hann(o):
    def hann(win_length, n_fft):
        n = np.arange(win_length, dtype=np.float64)
        w = 0.5 - 0.5 * np.cos(2.0 * math.pi * n / (win_length - 1))
        out = np.zeros(n_fft)
        left = (n_fft - win_length) // 2
        out[left : left + win_length] = w
        return out

    o.hann_periodic = hann


def _edge_repeating_pad(o):
    def pad_fn(x, pad):
        return np.concatenate([x[..., :pad][..., ::-1], x, x[..., -pad:][..., ::-1]], axis=-1)

    o.reflect_pad = pad_fn


def _off_by_one_frames(o):
    o.n_frames = lambda T, hop: (T + hop - 1) // hop


def _dft_wrong_sign_angle_index(o):
    orig = o.dft_onesided

    def dft(y):
        N = y.shape[-1]
        n = np.arange(N)[:, None]
        k = np.arange(N // 2 + 1)[None, :]
        ang = 2.0 * math.pi * ((k + 1) * n % N) / N  # transposed/shifted index
        return y @ np.cos(ang) - 1j * (y @ np.sin(ang))

    o.dft_onesided = dft
    del orig


def _falling_edge_foot(o):
    orig = o.mel_filterbank

    def fb(n_fft, sr, n_mels, f_min, f_max, scale="htk", norm=None):
        fk = o.bin_frequencies(n_fft, sr)[None, :]
        v = o.filter_vertices(f_min, f_max, n_mels, scale)
        lo, mid, hi = v[:-2, None], v[1:-1, None], v[2:, None]
        rising = (fk - lo) / (mid - lo)
        falling = (hi - fk) / (hi - lo)  # wrong denominator
        F = np.maximum(0.0, np.minimum(rising, falling))
        if norm == "slaney":
            F = F * (2.0 / (v[2:] - v[:-2]))[:, None]
        return F

    o.mel_filterbank = fb
    del orig


def _slaney_norm_base(o):
    orig = o.mel_filterbank

    def fb(n_fft, sr, n_mels, f_min, f_max, scale="htk", norm=None):
        F = orig(n_fft, sr, n_mels, f_min, f_max, scale, None)
        if norm == "slaney":
            v = o.filter_vertices(f_min, f_max, n_mels, scale)
            F = F * (2.0 / (v[1:-1] - v[:-2]))[:, None]  # half the base
        return F

    o.mel_filterbank = fb


def _htk_natural_log(o):
    orig = o.hz_to_mel

    def h2m(f, scale):
        if scale == "htk":
            return 2595.0 * np.log(1.0 + np.asarray(f, dtype=np.float64) / 700.0)
        return orig(f, scale)

    o.hz_to_mel = h2m


def _int16_scale(o):
    orig = o.to_float64

    def conv(x):
        x = np.asarray(x)
        if x.dtype == np.int16:
            return x.astype(np.float64) / 32767.0
        return orig(x)

    o.to_float64 = conv


def _power_half(o):
    orig = o.spectral_power

    def sp(X, power):
        return orig(X, power) * (0.5 if power == 2.0 else 1.0)

    o.spectral_power = sp


def _circular_shifted(o):
    orig = o.centre_pad

    def cp(x, pad, mode):
        if mode == "circular":
            T = x.shape[-1]
            return x[..., (np.arange(-pad, T + pad) + 1) % T]  # wraps one sample late
        return orig(x, pad, mode)

    o.centre_pad = cp


def _replicate_inner_sample(o):
    orig = o.centre_pad

    def cp(x, pad, mode):
        if mode == "replicate":
            T = x.shape[-1]
            return x[..., np.clip(np.arange(-pad, T + pad), 1, T - 2)]  # repeats the second sample
        return orig(x, pad, mode)

    o.centre_pad = cp


def _zero_pad_after_centring(o):
    def ps(x, n_fft, hop, win_length=None, power=2.0, center=True, pad_mode="reflect", pad=0, normalized=False):
        win_length = n_fft if win_length is None else win_length
        xd = o.to_float64(x)
        T = xd.shape[-1] + 2 * pad
        if center:
            xp = o.zero_pad(o.centre_pad(xd, n_fft // 2, pad_mode), pad)  # zeros outside the centre pad
            count = o.n_frames(T, hop)
        else:
            xp = o.zero_pad(xd, pad)
            count = o.n_frames_uncentred(T, n_fft, hop)
        frames = o.frame(xp, n_fft, hop, count)
        w = o.hann_periodic(win_length, n_fft)
        return np.swapaxes(o.spectral_power(o.dft_onesided(frames * w * o.window_norm(w, win_length, normalized)), power),
                           -1, -2)

    o.power_spectrogram = ps


def _window_norm_linear_sum(o):
    orig = o.window_norm

    def wn(w, win_length, normalized):
        if normalized in (True, "window"):
            return 1.0 / float(np.sum(w))
        return orig(w, win_length, normalized)

    o.window_norm = wn


def _uncentred_frame_count(o):
    o.n_frames_uncentred = lambda T, n_fft, hop: 1 + (T - n_fft + hop - 1) // hop


def _slaney_linear_slope(o):
    orig_h2m, orig_m2h = o.hz_to_mel, o.mel_to_hz

    def h2m(f, scale):
        if scale == "slaney":
            f = np.asarray(f, dtype=np.float64)
            return np.where(f >= 1000.0, orig_h2m(f, scale), f / 100.0)  # 10 mels per kHz instead of 15
        return orig_h2m(f, scale)

    def m2h(m, scale):
        if scale == "slaney":
            m = np.asarray(m, dtype=np.float64)
            return np.where(m >= 15.0, orig_m2h(m, scale), 100.0 * m)
        return orig_m2h(m, scale)

    o.hz_to_mel, o.mel_to_hz = h2m, m2h


def _slaney_log10(o):
    orig = o.hz_to_mel

    def h2m(f, scale):
        if scale == "slaney":
            f = np.asarray(f, dtype=np.float64)
            log = 15.0 + 27.0 * np.log10(np.maximum(f, 1e-300) / 1000.0) / np.log10(6.4) * 0.5  # half the step
            return np.where(f >= 1000.0, log, f / (200.0 / 3.0))
        return orig(f, scale)

    o.hz_to_mel = h2m


def _vertices_one_short(o):
    def fv(f_min, f_max, n_mels, scale):
        m = np.linspace(o.hz_to_mel(f_min, scale), o.hz_to_mel(f_max, scale), n_mels + 1)
        m = np.append(m, m[-1] + (m[-1] - m[-2]))  # n_mels + 1 steps squeezed, last vertex past f_max
        return o.mel_to_hz(m, scale)

    o.filter_vertices = fv


def _bin_grid_coarse(o):
    o.bin_frequencies = lambda n_fft, sr: np.arange(n_fft // 2 + 1, dtype=np.float64) * (float(sr) / (n_fft - 2))


def _window_left_aligned(o):
    def hann(win_length, n_fft):
        n = np.arange(win_length, dtype=np.float64)
        out = np.zeros(n_fft)
        out[:win_length] = 0.5 - 0.5 * np.cos(2.0 * math.pi * n / win_length)  # not centred
        return out

    o.hann_periodic = hann


def _frames_one_late(o):
    def frame(xp, n_fft, hop, count):
        idx = np.arange(count)[:, None] * hop + np.arange(n_fft)[None, :] + 1
        idx = np.minimum(idx, xp.shape[-1] - 1)
        return xp[..., idx]

    o.frame = frame


def _power_ignored(o):
    orig = o.spectral_power
    o.spectral_power = lambda X, power: orig(X, 2.0)


def _frame_length_norm_by_nfft(o):
    orig = o.window_norm

    def wn(w, win_length, normalized):
        if normalized == "frame_length":
            return 1.0 / math.sqrt(float(w.shape[-1]))  # the frame (torch.stft), not the window's length
        return orig(w, win_length, normalized)

    o.window_norm = wn


def _constant_pads_edge(o):
    orig = o.centre_pad

    def cp(x, pad, mode):
        if mode == "constant" and pad > 0:
            return orig(x, pad, "replicate")
        return orig(x, pad, mode)

    o.centre_pad = cp


def _f_max_ignored(o):
    orig = o.mel_filterbank
    o.mel_filterbank = lambda n_fft, sr, n_mels, f_min, f_max, scale="htk", norm=None: orig(
        n_fft, sr, n_mels, f_min, sr / 2.0, scale, norm)


def _f_min_ignored(o):
    orig = o.mel_filterbank
    o.mel_filterbank = lambda n_fft, sr, n_mels, f_min, f_max, scale="htk", norm=None: orig(
        n_fft, sr, n_mels, 0.0, f_max, scale, norm)


def _int16_unsigned(o):
    orig = o.to_float64

    def conv(x):
        x = np.asarray(x)
        if x.dtype == np.int16:
            return x.view(np.uint16).astype(np.float64) / 32768.0  # sign bit read as magnitude
        return orig(x)

    o.to_float64 = conv


def _reflect_right_repeats_edge(o):
    orig = o.reflect_pad

    def rp(x, pad):
        out = orig(x, pad)
        if pad > 0:
            T = x.shape[-1]
            out[..., pad + T :] = x[..., T - pad :][..., ::-1]  # right mirror repeats x[T-1]
        return out

    o.reflect_pad = rp


def _htk_break_1000(o):
    orig_h2m, orig_m2h = o.hz_to_mel, o.mel_to_hz

    def h2m(f, scale):
        if scale == "htk":
            return 2595.0 * np.log10(1.0 + np.asarray(f, dtype=np.float64) / 1000.0)
        return orig_h2m(f, scale)

    def m2h(m, scale):
        if scale == "htk":
            return 1000.0 * (10.0 ** (np.asarray(m, dtype=np.float64) / 2595.0) - 1.0)
        return orig_m2h(m, scale)

    o.hz_to_mel, o.mel_to_hz = h2m, m2h


def _filters_reversed(o):
    orig = o.mel_filterbank
    o.mel_filterbank = lambda *a, **k: orig(*a, **k)[::-1].copy()


def _normalized_ignored(o):
    o.window_norm = lambda w, win_length, normalized: 1.0


MUTANTS = [
    _symmetric_hann,
    _edge_repeating_pad,
    _off_by_one_frames,
    _dft_wrong_sign_angle_index,
    _falling_edge_foot,
    _slaney_norm_base,
    _htk_natural_log,
    _int16_scale,
    _power_half,
    _circular_shifted,
    _replicate_inner_sample,
    _zero_pad_after_centring,
    _window_norm_linear_sum,
    _uncentred_frame_count,
    _slaney_linear_slope,
    _slaney_log10,
    _vertices_one_short,
    _bin_grid_coarse,
    _window_left_aligned,
    _frames_one_late,
    _power_ignored,
    _frame_length_norm_by_nfft,
    _constant_pads_edge,
    _f_max_ignored,
    _f_min_ignored,
    _int16_unsigned,
    _reflect_right_repeats_edge,
    _htk_break_1000,
    _filters_reversed,
    _normalized_ignored,
]


@pytest.mark.parametrize("mutate", MUTANTS, ids=lambda m: m.__name__.strip("_"))
def test_pins_catch_planted_mistake(mutate):
    o = _fresh_oracle()
    mutate(o)
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(o)
        except (AssertionError, ValueError, IndexError):
            failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake {mutate.__name__}"


def test_mutants_do_not_leak():
    assert "oracle_mutant" not in sys.modules or sys.modules["oracle_mutant"] is not real_oracle
    pins.check_bin_centre_cosine(real_oracle)


def test_oracle_dft_at_the_large_sizes():
    """The oracle's DFT at the sizes of the large-transform kernels (4096 to
    16384, the huge workload's 16384 among them), where an angle 2 pi k n / N
    formed without reducing k n mod N first would lose digits: Parseval on
    random rows, and the closed form of a cosine on bin k0, whose one-sided
    spectrum is N/2 at k0 and zero elsewhere. The bound on the cosine, 1e-13 N,
    sits between the oracle's own error (3.9e-12 at 16384) and that of the
    same matrices built from the unreduced angle (1.2e-8). Run on the oracle
    itself only (each matrix pair is 1 GB at 16384, too heavy for the
    planted-mistake loop)."""
    rng = np.random.default_rng(16384)
    for N in (4096, 8192, 16384):
        y = rng.standard_normal((2, N))
        n = np.arange(N)
        k0 = N // 2 - 7 if N == 16384 else 3 * N // 8 + 5
        c = np.cos(2.0 * math.pi * ((k0 * n) % N) / N)
        X = real_oracle.dft_onesided(np.vstack([y, c[None, :]]))
        e = np.abs(X[:2]) ** 2
        lhs = e[:, 0] + 2.0 * e[:, 1 : N // 2].sum(axis=1) + e[:, N // 2]
        assert np.allclose(lhs, N * (y * y).sum(axis=1), rtol=1e-11), N
        expect = np.zeros(N // 2 + 1)
        expect[k0] = N / 2
        assert np.abs(X[2] - expect).max() <= 1e-13 * N, (N, np.abs(X[2] - expect).max())
