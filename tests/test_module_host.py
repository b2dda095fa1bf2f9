"""Host-side logic of the torchaudio-style module, without a GPU.

MelSpectrogram works out its output shape on the host, before it makes a
plan. Its frame count must agree with the float64 oracle's framing for every
combination of centring, zero padding and pad mode; and it refuses what the
path cannot compute (onesided=False, an output dtype other than f32 / f16,
a CPU tensor) before any CUDA call.
"""
from __future__ import annotations


import numpy as np
import pytest

import oracle.mel_oracle as o
from mel_spectrogram_gb300 import MelSpectrogram


def shortest(n_fft, center, pad_mode, pad):
    """The shortest signal the framing accepts (T' = T + 2 pad): uncentred
    T' >= n_fft, reflect T' > n_fft / 2, circular T' >= n_fft / 2, else 1."""
    if not center:
        return max(1, n_fft - 2 * pad)
    if pad_mode == "reflect":
        return max(1, n_fft // 2 + 1 - 2 * pad)
    if pad_mode == "circular":
        return max(1, n_fft // 2 - 2 * pad)
    return 1


def oracle_frame_count(T, n_fft, hop, center, pad_mode, pad):
    x = np.random.default_rng(T).standard_normal((1, T))
    return o.power_spectrogram(x, n_fft, hop, center=center, pad_mode=pad_mode, pad=pad).shape[-1]


@pytest.mark.parametrize("n_fft,hop", [(400, 160), (64, 16), (1024, 256), (256, 100)])
@pytest.mark.parametrize("center,pad_mode,pad", [(True, "reflect", 0), (True, "constant", 3), (True, "circular", 0),
                                                 (True, "replicate", 7), (False, "reflect", 0), (False, "reflect", 5)])
def test_frame_count_matches_oracle(n_fft, hop, center, pad_mode, pad):
    mel = MelSpectrogram(sample_rate=16000, n_fft=n_fft, hop_length=hop, n_mels=40, center=center,
                         pad_mode=pad_mode, pad=pad)
    lo = shortest(n_fft, center, pad_mode, pad)
    for T in sorted({lo, lo + 1, lo + hop - 1, 3 * hop + 7, 5 * n_fft + 3}):
        if T < lo:
            continue
        assert mel.n_frames(T) == oracle_frame_count(T, n_fft, hop, center, pad_mode, pad), T


def test_uncentred_too_short_has_no_frame():
    mel = MelSpectrogram(sample_rate=16000, n_fft=400, hop_length=160, center=False)
    assert mel.n_frames(399) == -1
    assert mel.n_frames(400) == 1


def test_refusals_before_any_cuda_call():
    import torch

    with pytest.raises(ValueError):
        MelSpectrogram(onesided=False)
    with pytest.raises(ValueError):
        MelSpectrogram(dtype=torch.float64)
    mel = MelSpectrogram(sample_rate=16000, n_fft=400, hop_length=160)
    with pytest.raises(ValueError):
        mel(torch.zeros(2, 1000))  # a CPU tensor
    assert mel._plans == {}  # nothing was planned


@pytest.mark.parametrize("win_length,hop_length", [(None, None), (300, None), (None, 100)])
def test_defaults_follow_torchaudio(win_length, hop_length):
    mel = MelSpectrogram(sample_rate=22050, n_fft=512, win_length=win_length, hop_length=hop_length)
    win = 512 if win_length is None else win_length
    assert mel.win_length == win
    assert mel.hop_length == (win // 2 if hop_length is None else hop_length)
    assert mel.f_max == 22050 / 2 and mel.n_mels == 128 and mel.power == 2.0


def test_device_input_generator_recipes():
    """make_input_device (the generator of the batches past 2^31 samples)
    follows the recipes' dtype and range, is seeded, and refuses the others;
    on the CPU here, torch's generator being the same code on any device."""
    import dataclasses

    import torch

    from mel_spectrogram_gb300.workloads import WORKLOADS, make_input_device

    w = WORKLOADS["int16"].resized(B=2, T=50000)
    a, b = make_input_device(w, "cpu"), make_input_device(w, "cpu")
    assert a.dtype == torch.int16 and tuple(a.shape) == (2, 50000)
    assert torch.equal(a, b)  # seeded
    assert int(a.min()) < -30000 and int(a.max()) > 30000  # the full int16 range
    assert not torch.equal(a, make_input_device(w, "cpu", seed=99))
    s = make_input_device(WORKLOADS["speech"].resized(B=1, T=100000), "cpu")
    assert s.dtype == torch.float32 and abs(float(s.mean())) < 0.02 and abs(float(s.std()) - 1.0) < 0.02
    with pytest.raises(ValueError):
        make_input_device(dataclasses.replace(w, recipe="music16"), "cpu")
