"""Pins for the float64 oracle: checks that do not restate its code.

Each ``check_*`` takes an oracle module (the real one, or a copy with a planted
mistake) and raises AssertionError if the module disagrees with something the
pages or the mathematics fix independently:

  * brute force: an explicit triple loop (mirrored list, complex exponentials),
    and one that spells out every pad mode, centring, `pad` and normalisation;
  * closed forms: an impulse, and a bin-centre cosine through the whole chain;
  * Parseval's identity for the one-sided DFT;
  * filterbank invariants: mel-equispaced vertices, support, partition of
    unity, Slaney unit area, and the published anchors in golden/anchors.json;
  * a library special case: torch.stft in float64 on the CPU.
"""
from __future__ import annotations

import cmath
import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- brute force
def brute_power(x, n_fft, hop, win_length, power=2.0):
    """Deliberately naive STFT power: explicit mirrored list and exponentials."""
    x = [float(v) for v in x]
    T = len(x)
    pad = n_fft // 2
    left = [x[pad - i] for i in range(pad)]  # x[pad], ..., x[1]
    right = [x[T - 2 - j] for j in range(pad)]  # x[T-2], x[T-3], ...
    xp = left + x + right
    lpad = (n_fft - win_length) // 2
    w = [0.0] * n_fft
    for n in range(win_length):
        w[lpad + n] = 0.5 - 0.5 * math.cos(2.0 * math.pi * n / win_length)
    frames = 1 + T // hop
    out = np.zeros((n_fft // 2 + 1, frames))
    for t in range(frames):
        for k in range(n_fft // 2 + 1):
            acc = 0j
            for n in range(n_fft):
                acc += xp[t * hop + n] * w[n] * cmath.exp(-2j * math.pi * k * n / n_fft)
            out[k, t] = abs(acc) ** power
    return out


def check_brute_force(o):
    rng = np.random.default_rng(123)
    cases = [
        (8, 2, 8, 9),  # n_fft, hop, win, T
        (8, 3, 8, 11),
        (10, 4, 6, 13),  # non-power-of-two, win < n_fft
        (12, 5, 12, 7),  # T barely above n_fft/2
        (16, 4, 11, 40),  # odd window inside a pow2 frame
    ]
    for n_fft, hop, win, T in cases:
        x = rng.integers(-9, 10, size=T).astype(np.float32)
        for p in (2.0, 1.0):
            ref = brute_power(x, n_fft, hop, win, p)
            got = o.power_spectrogram(x, n_fft, hop, win, p)
            assert got.shape == ref.shape, (got.shape, ref.shape)
            assert np.allclose(got, ref, rtol=1e-10, atol=1e-9), (n_fft, hop, win, T, p)


def brute_power_framed(x, n_fft, hop, win_length, power, center, pad_mode, pad, normalized):
    """Naive STFT power with every framing option spelled out sample by sample."""
    x = [0.0] * pad + [float(v) for v in x] + [0.0] * pad  # torchaudio `pad`: zeros first
    T = len(x)
    c = n_fft // 2 if center else 0

    def sample(i):  # position i of the centre-padded signal
        j = i - c
        if 0 <= j < T:
            return x[j]
        if pad_mode == "constant":
            return 0.0
        if pad_mode == "replicate":
            return x[0] if j < 0 else x[T - 1]
        if pad_mode == "circular":
            return x[j + T] if j < 0 else x[j - T]
        # reflect: the sample as far inside from the edge as j is outside
        return x[-j] if j < 0 else x[(T - 1) - (j - (T - 1))]

    lpad = (n_fft - win_length) // 2
    w = [0.0] * n_fft
    for n in range(win_length):
        w[lpad + n] = 0.5 - 0.5 * math.cos(2.0 * math.pi * n / win_length)
    if normalized in (True, "window"):
        scale = 1.0 / math.sqrt(sum(v * v for v in w))
    elif normalized == "frame_length":
        scale = 1.0 / math.sqrt(win_length)
    else:
        scale = 1.0
    frames = 1 + T // hop if center else 1 + (T - n_fft) // hop
    out = np.zeros((n_fft // 2 + 1, frames))
    for t in range(frames):
        for k in range(n_fft // 2 + 1):
            acc = 0j
            for n in range(n_fft):
                acc += sample(t * hop + n) * w[n] * scale * cmath.exp(-2j * math.pi * k * n / n_fft)
            out[k, t] = abs(acc) ** power
    return out


def check_framing_brute_force(o):
    """Every pad mode, with and without centring, the `pad` zeros and both
    normalisations, against the sample-by-sample brute force."""
    rng = np.random.default_rng(321)
    cases = [  # n_fft, hop, win, T, pad
        (8, 2, 8, 9, 0),
        (8, 3, 6, 13, 2),
        (10, 4, 10, 12, 0),
        (12, 5, 12, 17, 3),
    ]
    for n_fft, hop, win, T, zp in cases:
        x = rng.integers(-9, 10, size=T).astype(np.float32)
        for mode in ("reflect", "constant", "replicate", "circular"):
            for center in (True, False):
                for norm in (False, "window", "frame_length"):
                    ref = brute_power_framed(x, n_fft, hop, win, 2.0, center, mode, zp, norm)
                    got = o.power_spectrogram(x, n_fft, hop, win, 2.0, center, mode, zp, norm)
                    assert got.shape == ref.shape, (mode, center, got.shape, ref.shape)
                    assert np.allclose(got, ref, rtol=1e-10, atol=1e-9 * max(1.0, ref.max())), (
                        n_fft, hop, win, T, zp, mode, center, norm)


# ------------------------------------------------------------ closed forms
def check_impulse(o):
    """x = delta at n0: each frame that holds it has |X[k]| = w[j] for all k."""
    n_fft, hop, T, n0 = 64, 16, 400, 211
    x = np.zeros(T, dtype=np.float32)
    x[n0] = 1.0
    P = o.power_spectrogram(x, n_fft, hop, n_fft, 2.0)  # [n_freqs, frames]
    pad = n_fft // 2
    for t in range(P.shape[1]):
        j = n0 + pad - t * hop
        if 0 <= j < n_fft:
            wj = 0.5 - 0.5 * math.cos(2.0 * math.pi * j / n_fft)
            assert np.allclose(P[:, t], wj * wj, rtol=1e-12, atol=1e-15), t
        else:
            assert np.allclose(P[:, t], 0.0, atol=1e-20), t


def check_parseval(o):
    """|X0|^2 + 2 sum_{0<k<N/2} |Xk|^2 + |X_{N/2}|^2 = N sum y^2 (N even)."""
    rng = np.random.default_rng(7)
    for N in (8, 10, 400, 1024, 2048):
        y = rng.standard_normal((3, N))
        X = o.dft_onesided(y)
        e = np.abs(X) ** 2
        lhs = e[:, 0] + 2.0 * e[:, 1 : N // 2].sum(axis=1) + e[:, N // 2]
        rhs = N * (y * y).sum(axis=1)
        assert np.allclose(lhs, rhs, rtol=1e-12), N


def check_bin_centre_cosine(o):
    """A cosine at bin k0 through the whole chain.

    With a periodic Hann of length N the windowed spectrum of cos(2 pi k0 n/N)
    has |X[k0]| = A N/4 and |X[k0 +- 1]| = A N/8 and nothing else in 0..N/2
    (2 <= k0 <= N/2 - 2), so M[m] = (AN/4)^p F[m,k0] + (AN/8)^p (F[m,k0-1] +
    F[m,k0+1]) for every frame clear of the right edge (phase 0 makes the left
    mirror exact).
    """
    for n_fft, hop, sr, n_mels, k0, A, scale, norm, p in [
        (400, 160, 16000, 80, 37, 0.7, "htk", None, 2.0),
        (1024, 256, 16000, 80, 100, 1.3, "htk", None, 2.0),
        (2048, 512, 22050, 128, 333, 0.25, "slaney", "slaney", 1.0),
    ]:
        T = 8 * n_fft + 3
        n = np.arange(T, dtype=np.float64)
        x = A * np.cos(2.0 * math.pi * k0 * n / n_fft)
        M = o.mel_spectrogram(x, sr, n_fft, hop, n_mels, 0.0, sr / 2.0, p, scale, norm)
        F = o.mel_filterbank(n_fft, sr, n_mels, 0.0, sr / 2.0, scale, norm)
        expect = (A * n_fft / 4) ** p * F[:, k0] + (A * n_fft / 8) ** p * (F[:, k0 - 1] + F[:, k0 + 1])
        pad = n_fft // 2
        clear = [t for t in range(M.shape[1]) if t * hop - pad + n_fft <= T]
        assert len(clear) > 3
        scale_ = max(1.0, float(np.abs(expect).max()))
        for t in clear:
            assert np.allclose(M[:, t], expect, rtol=1e-9, atol=1e-9 * scale_), (n_fft, t)
        # and the cosine lights only the filters whose support holds k0-1..k0+1
        lit = np.nonzero(expect > 0)[0]
        assert lit.size >= 1
        for m in range(n_mels):
            if m not in lit:
                assert np.all(np.abs(M[m, clear]) <= 1e-9 * scale_), m


# ----------------------------------------------------------- filterbank pins
def check_mel_anchors(o):
    with open(os.path.join(GOLDEN, "anchors.json")) as f:
        anchors = json.load(f)
    for scale in ("htk", "slaney"):
        for a in anchors[scale]:
            got = float(o.hz_to_mel(a["hz"], scale))
            if "mel" in a:
                assert abs(got - a["mel"]) <= 1e-9 * max(1.0, a["mel"]), (scale, a, got)
                back = float(o.mel_to_hz(a["mel"], scale))
                assert abs(back - a["hz"]) <= 1e-8 * max(1.0, a["hz"]), (scale, a, back)
            else:
                assert abs(got - a["mel_approx"]) <= a["abs_tol"], (scale, a, got)
    f = np.linspace(0.0, 20000.0, 2001)
    for scale in ("htk", "slaney"):
        assert np.allclose(o.mel_to_hz(o.hz_to_mel(f, scale), scale), f, rtol=1e-12, atol=1e-9)
        # continuity (the Slaney scale joins its two pieces at 1 kHz)
        m = o.hz_to_mel(np.array([999.999999, 1000.0, 1000.000001]), scale)
        assert np.all(np.diff(m) >= 0) and m[2] - m[0] < 1e-5


def check_filterbank_shape(o):
    """Vertices equispaced in mel; support (v_m, v_{m+2}); peaks <= 1;
    adjacent rising + falling edges sum to one between v_1 and v_{n_mels}."""
    for n_fft, sr, n_mels, f_min, f_max, scale in [
        (400, 16000, 80, 0.0, 8000.0, "htk"),
        (400, 16000, 128, 0.0, 8000.0, "htk"),
        (1024, 16000, 80, 0.0, 8000.0, "htk"),
        (2048, 22050, 128, 0.0, 11025.0, "slaney"),
        (512, 16000, 40, 125.0, 7600.0, "slaney"),
    ]:
        v = o.filter_vertices(f_min, f_max, n_mels, scale)
        assert v.shape == (n_mels + 2,)
        assert abs(v[0] - f_min) < 1e-6 and abs(v[-1] - f_max) < 1e-6
        dm = np.diff(o.hz_to_mel(v, scale))
        assert np.allclose(dm, dm[0], rtol=1e-9)
        F = o.mel_filterbank(n_fft, sr, n_mels, f_min, f_max, scale, None)
        fk = np.arange(n_fft // 2 + 1) * sr / n_fft
        assert F.shape == (n_mels, n_fft // 2 + 1)
        assert np.all(F >= 0) and np.all(F <= 1.0 + 1e-12)
        for m in range(n_mels):
            inside = (fk > v[m]) & (fk < v[m + 2])
            assert np.all(F[m, ~inside] == 0.0), m
            # a bin at distance d below the peak has weight 1 - d/(v[m+1]-v[m])
            k = np.nonzero(inside)[0]
            if k.size:
                kk = k[np.argmax(F[m, k])]
                assert abs(fk[kk] - v[m + 1]) <= sr / n_fft + 1e-9
        cover = (fk >= v[1]) & (fk <= v[n_mels])
        assert np.allclose(F[:, cover].sum(axis=0), 1.0, atol=1e-12)
        assert np.all(F[:, ~cover].sum(axis=0) <= 1.0 + 1e-12)


def check_band_limits(o):
    """The filterbank spans exactly the band [f_min, f_max]: its first
    triangle starts at f_min and its last ends at f_max, so on the bin grid
    k sr / n_fft every weight at or below f_min, or at or above f_max, is
    zero, and the bins strictly inside the band carry weight."""
    for n_fft, sr, n_mels, f_min, f_max, scale in [
        (512, 16000, 40, 125.0, 7600.0, "slaney"),
        (1024, 16000, 64, 300.0, 3400.0, "htk"),
        (2048, 44100, 96, 40.0, 15000.0, "slaney"),
    ]:
        F = o.mel_filterbank(n_fft, sr, n_mels, f_min, f_max, scale, None)
        fk = np.arange(n_fft // 2 + 1) * sr / n_fft
        outside = (fk <= f_min) | (fk >= f_max)
        assert np.all(F[:, outside] == 0.0), (n_fft, f_min, f_max)
        inside = ~outside
        assert np.all(F[:, inside].sum(axis=0) > 0.0), (n_fft, f_min, f_max)


def check_shift_and_scale(o):
    """Two invariants of the transform. Shift: advancing the signal by one hop
    moves every frame that reads no padding up by one (frame t + 1 of x is
    frame t of x[hop:]). Homogeneity: scaling the signal by a scales the
    output by a^p, for the power p."""
    rng = np.random.default_rng(17)
    for n_fft, hop, power in [(400, 160, 2.0), (256, 64, 1.0), (512, 200, 0.5)]:
        T = 12 * n_fft + 37
        x = rng.standard_normal((1, T))
        args = (16000, n_fft, hop, 40, 0.0, 8000.0, power, "htk", None)
        full = o.mel_spectrogram(x, *args)[0]
        moved = o.mel_spectrogram(x[:, hop:], *args)[0]
        half = n_fft // 2
        t_lo = -(-half // hop)  # first frame of x[hop:] that starts inside it
        t_hi = (T - hop - half) // hop  # last frame of x[hop:] that ends inside it
        assert t_hi - t_lo > 5
        np.testing.assert_allclose(moved[:, t_lo : t_hi + 1], full[:, t_lo + 1 : t_hi + 2], rtol=1e-9, atol=1e-9)
        a = 3.0
        scaled = o.mel_spectrogram(a * x, *args)[0]
        np.testing.assert_allclose(scaled, a ** power * full, rtol=1e-9, atol=1e-12)


def check_slaney_area(o):
    """With Slaney norm every triangle has unit area (Riemann sum over bins)."""
    sr = 22050
    for n_fft, tol in [(2048, 0.05), (1 << 16, 1e-4)]:
        F = o.mel_filterbank(n_fft, sr, 128, 0.0, 11025.0, "slaney", "slaney")
        area = F.sum(axis=1) * (sr / n_fft)
        assert np.all(np.abs(area - 1.0) <= tol), (n_fft, area.min(), area.max())


# --------------------------------------------------------- conversions, misc
def check_input_conversion(o):
    x = np.array([-32768, -1, 0, 1, 16384, 32767], dtype=np.int16)
    assert np.array_equal(o.to_float64(x), np.array([-1.0, -1 / 32768, 0.0, 1 / 32768, 0.5, 32767 / 32768]))
    h = np.array([0.1, -0.333, 1.0, 6.1e-5], dtype=np.float16)
    assert np.array_equal(o.to_float64(h), h.astype(np.float32).astype(np.float64))


def check_torch_stft(o):
    """Library special case: torch.stft, float64, periodic Hann, centre reflect
    and every other framing torch offers (pad modes, no centring, `pad` zeros
    first as torchaudio applies them, frame-length normalisation rescaled
    from torch's sqrt(n_fft) to the page's sqrt(win_length))."""
    import torch
    import torch.nn.functional as tf

    rng = np.random.default_rng(11)
    for n_fft, hop, win, T in [(400, 160, 400, 3000), (1024, 256, 1024, 5000), (256, 64, 200, 1001)]:
        x = rng.standard_normal(T)
        w = torch.hann_window(win, periodic=True, dtype=torch.float64)
        S = torch.stft(
            torch.from_numpy(x), n_fft, hop, win, window=w, center=True, pad_mode="reflect", return_complex=True
        )
        ref = (S.abs() ** 2).numpy()
        got = o.power_spectrogram(x, n_fft, hop, win, 2.0)
        assert got.shape == ref.shape
        assert np.allclose(got, ref, rtol=1e-9, atol=1e-9 * ref.max())
    for n_fft, hop, win, T, zp in [(400, 160, 400, 1900, 0), (256, 64, 200, 1001, 37), (64, 16, 64, 300, 5)]:
        x = rng.standard_normal(T)
        w = torch.hann_window(win, periodic=True, dtype=torch.float64)
        xt = tf.pad(torch.from_numpy(x)[None], (zp, zp), "constant")[0] if zp else torch.from_numpy(x)
        for mode in ("reflect", "constant", "replicate", "circular"):
            for center in (True, False):
                for normalized in (False, True):
                    S = torch.stft(xt, n_fft, hop, win, window=w, center=center, pad_mode=mode,
                                   normalized=normalized, return_complex=True)
                    # torch.stft's normalized=True divides by sqrt(n_fft), the
                    # page's frame-length normalisation by sqrt(win_length)
                    ref = (S.abs() ** 2).numpy() * (n_fft / win if normalized else 1.0)
                    got = o.power_spectrogram(x, n_fft, hop, win, 2.0, center, mode, zp,
                                              "frame_length" if normalized else False)
                    assert got.shape == ref.shape, (mode, center, got.shape, ref.shape)
                    assert np.allclose(got, ref, rtol=1e-9, atol=1e-9 * ref.max()), (n_fft, mode, center, normalized)


def check_window_normalisation(o):
    """An impulse inside a frame gives |X[k]| = w[j] / sqrt(sum w^2) for every
    k with the window normalisation, and w[j] / sqrt(win_length) with the
    frame-length one (flashmel filters.py make_window)."""
    n_fft, hop, T, n0, win = 64, 16, 400, 211, 50
    x = np.zeros(T)
    x[n0] = 1.0
    lpad = (n_fft - win) // 2
    w = np.zeros(n_fft)
    w[lpad : lpad + win] = [0.5 - 0.5 * math.cos(2.0 * math.pi * n / win) for n in range(win)]
    for normalized, scale in (("window", 1.0 / math.sqrt(float(np.dot(w, w)))), ("frame_length", 1.0 / math.sqrt(win))):
        P = o.power_spectrogram(x, n_fft, hop, win, 1.0, True, "reflect", 0, normalized)
        for t in range(P.shape[1]):
            j = n0 + n_fft // 2 - t * hop
            expect = w[j] * scale if 0 <= j < n_fft else 0.0
            assert np.allclose(P[:, t], expect, rtol=1e-12, atol=1e-15), (normalized, t)


ALL_CHECKS = [
    check_brute_force,
    check_impulse,
    check_parseval,
    check_bin_centre_cosine,
    check_mel_anchors,
    check_filterbank_shape,
    check_slaney_area,
    check_input_conversion,
    check_torch_stft,
    check_framing_brute_force,
    check_window_normalisation,
    check_band_limits,
    check_shift_and_scale,
]
