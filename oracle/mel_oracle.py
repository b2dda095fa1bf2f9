"""Float64 CPU oracle for the batched mel spectrogram.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it. It shares
no code, tables or constants with the CUDA path.

What it computes is the torchaudio-style ``MelSpectrogram`` that the flashmel
0.1.0 page describes (README, sections "Usage" and "How it works"; the host
helpers ``make_window`` and ``pack_fbank`` in ``flashmel/filters.py``):

    centre reflect pad -> frame at hop -> periodic Hann window
    -> n_fft-point real DFT (bins 0..n_fft/2) -> |X|^power
    -> triangular mel filterbank (HTK or Slaney scale, optional Slaney norm)

with the framing options the page lists among the supported torchaudio
arguments (README "Usage": pad, center, pad_mode, normalized; "How it works":
padding and all four pad modes applied as index arithmetic, the normalized
modes folded into the window):

    zero-pad `pad` samples on both sides -> (center) pad n_fft/2 on both
    sides by pad_mode (reflect / constant / replicate / circular) -> frame
    -> window scaled by the normalisation -> DFT -> ...

Every step is the plain definition, in float64, in the page's order. The DFT
is the naive O(N^2) sum written as a matmul against explicit cos/sin
matrices: no FFT, no blocking, no fusion.

Readings where the pages are silent (the mel formulas are not printed: the
page only names torchaudio's ``melscale_fbanks``):
  * bin k sits at frequency k * sr / n_fft (the DFT's own bin spacing);
  * HTK mel: 2595 * log10(1 + f / 700);
  * Slaney mel: linear 3 f / 200 below 1 kHz, logarithmic above with
    27 mels per factor 6.4 (so 1 kHz -> 15, 6.4 kHz -> 42);
  * filter vertices are n_mels + 2 points equally spaced in mel between
    mel(f_min) and mel(f_max); triangles are linear in Hz;
  * Slaney norm scales filter m by 2 / (f[m+2] - f[m]) (unit area);
  * reflect padding mirrors about the edge sample without repeating it;
  * int16 input is scaled by 1/32768; f16 input widens exactly;
  * the pad modes are torch's: constant fills zeros, replicate repeats the
    edge sample, circular wraps around the signal; `pad` zero-pads before the
    centre padding, which then mirrors / repeats / wraps the zero-padded
    signal; without centring, frames start at sample 0 and there are
    1 + floor((T - n_fft) / hop) of them;
  * normalized "window" (or True) divides the spectrum by sqrt(sum w^2),
    "frame_length" by sqrt(win_length) (flashmel README, filters.py
    make_window: the window divided by the square root of its own length;
    equal to torch.stft's sqrt(n_fft) whenever win_length = n_fft).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force, closed forms, Parseval, filterbank invariants).
"""
from __future__ import annotations

import math

import numpy as np

# --------------------------------------------------------------------------
# a1: input conversion (README "Usage": int16 raw PCM scaled by 1/32768)
# --------------------------------------------------------------------------


def to_float64(x: np.ndarray) -> np.ndarray:
    """Widen the stored samples to float64.

    float32 / float16 widen exactly; int16 PCM is scaled by 1/32768
    (flashmel README, "Usage": int16 raw PCM scaled by 1/32768).
    """
    x = np.asarray(x)
    if x.dtype == np.int16:
        return x.astype(np.float64) / 32768.0
    if x.dtype in (np.float32, np.float16, np.float64):
        return x.astype(np.float64)
    raise TypeError(f"unsupported input dtype {x.dtype}")


# --------------------------------------------------------------------------
# a2/a3: centre reflect padding and framing (README "How it works": padding
# and framing applied as index arithmetic; torchaudio defaults center=True,
# pad_mode="reflect")
# --------------------------------------------------------------------------


def reflect_pad(x: np.ndarray, pad: int) -> np.ndarray:
    """Pad the last axis by ``pad`` on each side, mirroring without the edge.

    xp[i] = x[i - pad] inside; x[pad - i] on the left; x[2(T-1) - (i - pad)]
    on the right. Requires T > pad (a mirror cannot reach further).
    """
    T = x.shape[-1]
    if pad >= T:
        raise ValueError(f"reflect padding needs T > pad (T={T}, pad={pad})")
    left = x[..., 1 : pad + 1][..., ::-1]
    right = x[..., T - 1 - pad : T - 1][..., ::-1]
    return np.concatenate([left, x, right], axis=-1)


PAD_MODES = ("reflect", "constant", "replicate", "circular")


def centre_pad(x: np.ndarray, pad: int, mode: str) -> np.ndarray:
    """Pad the last axis by ``pad`` on each side by ``mode``.

    Position i of the result holds x[i - pad] inside; outside, with
    j = i - pad < 0 or j >= T:
      reflect   : x[-j] / x[2(T-1) - j]   (mirror without the edge; T > pad)
      replicate : x[0] / x[T-1]
      circular  : x[j mod T]               (T >= pad)
      constant  : 0
    """
    if mode == "reflect":
        return reflect_pad(x, pad)
    T = x.shape[-1]
    j = np.arange(-pad, T + pad)
    if mode == "replicate":
        return x[..., np.clip(j, 0, T - 1)]
    if mode == "circular":
        if pad > T:
            raise ValueError(f"circular padding needs T >= pad (T={T}, pad={pad})")
        return x[..., j % T]
    if mode == "constant":
        out = np.zeros(x.shape[:-1] + (T + 2 * pad,), dtype=x.dtype)
        out[..., pad : pad + T] = x
        return out
    raise ValueError(mode)


def zero_pad(x: np.ndarray, pad: int) -> np.ndarray:
    """torchaudio's ``pad`` argument: ``pad`` zeros on each side of the signal."""
    if pad == 0:
        return x
    return centre_pad(x, pad, "constant")


def n_frames(T: int, hop: int) -> int:
    """Frame count with centre padding: 1 + floor(T / hop)."""
    return 1 + T // hop


def n_frames_uncentred(T: int, n_fft: int, hop: int) -> int:
    """Frame count without centre padding: 1 + floor((T - n_fft) / hop)."""
    if T < n_fft:
        raise ValueError(f"without centring the signal must hold one frame (T={T}, n_fft={n_fft})")
    return 1 + (T - n_fft) // hop


def frame(xp: np.ndarray, n_fft: int, hop: int, count: int) -> np.ndarray:
    """Frame t = xp[t*hop : t*hop + n_fft], t = 0..count-1 -> [..., count, n_fft]."""
    idx = np.arange(count)[:, None] * hop + np.arange(n_fft)[None, :]
    return xp[..., idx]


# --------------------------------------------------------------------------
# a4: periodic Hann, zero-padded and centred to n_fft (filters.py make_window)
# --------------------------------------------------------------------------


def hann_periodic(win_length: int, n_fft: int) -> np.ndarray:
    """w[n] = 0.5 - 0.5 cos(2 pi n / win_length), centred in n_fft zeros.

    Periodic Hann (denominator win_length, not win_length - 1) as in
    filters.py ``make_window``; left zero pad = (n_fft - win_length) // 2.
    """
    if win_length > n_fft:
        raise ValueError("win_length must not exceed n_fft")
    n = np.arange(win_length, dtype=np.float64)
    w = 0.5 - 0.5 * np.cos(2.0 * math.pi * n / win_length)
    out = np.zeros(n_fft, dtype=np.float64)
    left = (n_fft - win_length) // 2
    out[left : left + win_length] = w
    return out


# --------------------------------------------------------------------------
# a5/a6: naive real-input DFT and |X|^power (README: R2C FFT, |X|^power)
# --------------------------------------------------------------------------


def dft_matrices(n_fft: int) -> tuple[np.ndarray, np.ndarray]:
    """cos / sin matrices [n_fft, n_fft//2 + 1] of 2 pi k n / n_fft."""
    n = np.arange(n_fft, dtype=np.float64)[:, None]
    k = np.arange(n_fft // 2 + 1, dtype=np.float64)[None, :]
    # reduce k*n mod N in integers first so the angle is exact for large N
    kn = (np.arange(n_fft)[:, None] * np.arange(n_fft // 2 + 1)[None, :]) % n_fft
    ang = 2.0 * math.pi * kn.astype(np.float64) / n_fft
    del n, k
    return np.cos(ang), np.sin(ang)


def dft_onesided(y: np.ndarray) -> np.ndarray:
    """X[k] = sum_n y[n] (cos(2 pi k n/N) - i sin(2 pi k n/N)), k = 0..N/2."""
    N = y.shape[-1]
    C, S = dft_matrices(N)
    return y @ C - 1j * (y @ S)


def spectral_power(X: np.ndarray, power: float) -> np.ndarray:
    """|X|^power = (Re^2 + Im^2)^(power/2)."""
    mag2 = X.real * X.real + X.imag * X.imag
    if power == 2.0:
        return mag2
    if power == 1.0:
        return np.sqrt(mag2)
    return mag2 ** (power / 2.0)


def window_norm(w: np.ndarray, win_length: int, normalized) -> float:
    """Scale folded into the window (filters.py make_window): 1,
    1/sqrt(sum w^2) ("window" or True), or 1/sqrt(win_length) ("frame_length")."""
    if normalized in (False, None, "none"):
        return 1.0
    if normalized in (True, "window"):
        return 1.0 / math.sqrt(float(np.sum(w * w)))
    if normalized == "frame_length":
        return 1.0 / math.sqrt(win_length)
    raise ValueError(normalized)


def power_spectrogram(
    x: np.ndarray,
    n_fft: int,
    hop: int,
    win_length: int | None = None,
    power: float = 2.0,
    center: bool = True,
    pad_mode: str = "reflect",
    pad: int = 0,
    normalized=False,
) -> np.ndarray:
    """Steps a1-a6 for input [..., T] -> [..., n_fft//2 + 1, n_frames]."""
    win_length = n_fft if win_length is None else win_length
    xd = zero_pad(to_float64(x), pad)
    T = xd.shape[-1]
    if center:
        xp = centre_pad(xd, n_fft // 2, pad_mode)
        count = n_frames(T, hop)
    else:
        xp = xd
        count = n_frames_uncentred(T, n_fft, hop)
    frames = frame(xp, n_fft, hop, count)
    w = hann_periodic(win_length, n_fft)
    y = frames * (w * window_norm(w, win_length, normalized))
    P = spectral_power(dft_onesided(y), power)
    return np.swapaxes(P, -1, -2)


# --------------------------------------------------------------------------
# a7: triangular mel filterbank (filters.py pack_fbank -> melscale_fbanks)
# --------------------------------------------------------------------------

_SLANEY_F_SP = 200.0 / 3.0  # Hz per mel on the linear part
_SLANEY_BREAK_HZ = 1000.0
_SLANEY_BREAK_MEL = _SLANEY_BREAK_HZ / _SLANEY_F_SP  # = 15
_SLANEY_LOGSTEP = math.log(6.4) / 27.0  # 27 mels per factor 6.4


def hz_to_mel(f, scale: str):
    """HTK: 2595 log10(1 + f/700). Slaney: f/(200/3) below 1 kHz, log above."""
    f = np.asarray(f, dtype=np.float64)
    if scale == "htk":
        return 2595.0 * np.log10(1.0 + f / 700.0)
    if scale == "slaney":
        lin = f / _SLANEY_F_SP
        with np.errstate(divide="ignore"):
            log = _SLANEY_BREAK_MEL + np.log(np.maximum(f, 1e-300) / _SLANEY_BREAK_HZ) / _SLANEY_LOGSTEP
        return np.where(f >= _SLANEY_BREAK_HZ, log, lin)
    raise ValueError(scale)


def mel_to_hz(m, scale: str):
    """Inverse of :func:`hz_to_mel`."""
    m = np.asarray(m, dtype=np.float64)
    if scale == "htk":
        return 700.0 * (10.0 ** (m / 2595.0) - 1.0)
    if scale == "slaney":
        lin = _SLANEY_F_SP * m
        log = _SLANEY_BREAK_HZ * np.exp(_SLANEY_LOGSTEP * (m - _SLANEY_BREAK_MEL))
        return np.where(m >= _SLANEY_BREAK_MEL, log, lin)
    raise ValueError(scale)


def filter_vertices(f_min: float, f_max: float, n_mels: int, scale: str) -> np.ndarray:
    """n_mels + 2 vertex frequencies, equally spaced in mel."""
    m = np.linspace(hz_to_mel(f_min, scale), hz_to_mel(f_max, scale), n_mels + 2)
    return mel_to_hz(m, scale)


def bin_frequencies(n_fft: int, sr: float) -> np.ndarray:
    """Frequency of one-sided DFT bin k: k * sr / n_fft."""
    return np.arange(n_fft // 2 + 1, dtype=np.float64) * (float(sr) / n_fft)


def mel_filterbank(
    n_fft: int, sr: float, n_mels: int, f_min: float, f_max: float, scale: str = "htk", norm: str | None = None
) -> np.ndarray:
    """Dense filterbank F [n_mels, n_fft//2 + 1].

    F[m, k] = max(0, min((f_k - v_m) / (v_{m+1} - v_m), (v_{m+2} - f_k) / (v_{m+2} - v_{m+1})))
    and, with Slaney norm, row m is scaled by 2 / (v_{m+2} - v_m).
    """
    if f_max is None or f_max <= 0:
        f_max = sr / 2.0
    fk = bin_frequencies(n_fft, sr)[None, :]
    v = filter_vertices(f_min, f_max, n_mels, scale)
    lo, mid, hi = v[:-2, None], v[1:-1, None], v[2:, None]
    rising = (fk - lo) / (mid - lo)
    falling = (hi - fk) / (hi - mid)
    F = np.maximum(0.0, np.minimum(rising, falling))
    if norm == "slaney":
        F = F * (2.0 / (v[2:] - v[:-2]))[:, None]
    elif norm not in (None, "none"):
        raise ValueError(norm)
    return F


# --------------------------------------------------------------------------
# whole path
# --------------------------------------------------------------------------


def mel_spectrogram(
    x: np.ndarray,
    sr: int,
    n_fft: int,
    hop: int,
    n_mels: int,
    f_min: float = 0.0,
    f_max: float | None = None,
    power: float = 2.0,
    scale: str = "htk",
    norm: str | None = None,
    win_length: int | None = None,
    center: bool = True,
    pad_mode: str = "reflect",
    pad: int = 0,
    normalized=False,
) -> np.ndarray:
    """Input [..., T] (f32 / int16 / f16) -> float64 [..., n_mels, n_frames]."""
    P = power_spectrogram(x, n_fft, hop, win_length, power, center, pad_mode, pad, normalized)
    F = mel_filterbank(n_fft, sr, n_mels, f_min, f_max, scale, norm)
    return np.einsum("mk,...kt->...mt", F, P)
