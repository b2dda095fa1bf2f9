"""Seeded random configurations through the C ABI against the float64 oracle.

Each case draws an n_fft (400 or a power of two from 64 to 16384), a hop
(short, n_fft/4, n_fft/2, odd, or longer than the frame), mel count and
band, scale and norm, power, input and output dtype, and the framing options
(center, pad_mode, pad, normalized) of fm_plan_create_ex, so that every
kernel build a plan can choose (hop-specialised, any-hop, fewer tile groups
for long hops, one frame per thread, odd hops, large transforms) meets
combinations the targeted tests do not list. Every output element is
compared; f16 output may saturate to +inf where the oracle leaves the f16
range (flashmel README "Development")."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest

import oracle.mel_oracle as o
from mel_spectrogram_gb300 import _binding as fb
from mel_spectrogram_gb300.workloads import Workload, make_input
from tests.gpu_util import check_close, check_close_saturating, torch_dtype

pytestmark = pytest.mark.gpu

N_CASES = 96
SIZES = [64, 128, 256, 400, 512, 1024, 2048, 4096, 8192, 16384]
MODES = ["reflect", "constant", "replicate", "circular"]
RECIPE = {"f32": "normal", "i16": "pcm16", "f16": "music16"}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mel_spectrogram_gb300.build import build

    build()


def draw(i: int) -> dict:
    rng = np.random.default_rng(1000 + i)
    n_fft = int(SIZES[i % len(SIZES)])
    kind = int(rng.integers(0, 5))
    hop = [max(1, n_fft // 4), max(1, n_fft // 2), int(rng.integers(1, 64)) | 1,
           int(rng.integers(n_fft // 8 + 1, n_fft + n_fft // 2)), n_fft // 4 + 1][kind]
    sr = int(rng.choice([8000, 16000, 22050, 44100]))
    n_bins = n_fft // 2 + 1
    n_mels = int(min(256, max(1, rng.integers(1, min(n_bins, 160) + 1))))
    f_max = float(sr / 2 if rng.random() < 0.5 else rng.uniform(0.3, 1.0) * sr / 2)
    f_min = float(0.0 if rng.random() < 0.5 else rng.uniform(0.0, 0.2) * f_max)
    center = bool(rng.random() < 0.75)
    # frames the float64 oracle can afford: it computes an n_fft x n_fft DFT per frame
    frames = int(rng.integers(2, 40 if n_fft <= 2048 else 6))
    T = int(n_fft + hop * frames + rng.integers(0, hop + 1))
    return dict(
        n_fft=n_fft, hop=hop, sr=sr, n_mels=n_mels, f_min=f_min, f_max=f_max,
        win_length=int(n_fft if rng.random() < 0.7 else rng.integers(n_fft // 2, n_fft + 1)),
        power=float(rng.choice([1.0, 2.0, 0.5, 3.0])),
        mel_scale=str(rng.choice(["htk", "slaney"])), norm=None if rng.random() < 0.6 else "slaney",
        in_dtype=str(rng.choice(["f32", "i16", "f16"])), out_dtype=str(rng.choice(["f32", "f32", "f16"])),
        center=center, pad_mode=str(rng.choice(MODES)), pad=int(rng.choice([0, 0, 0, 3, 64])),
        normalized=[False, "window", "frame_length"][int(rng.integers(0, 3))], T=T,
        B=int(rng.integers(1, 4)), seed=2000 + i)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_configuration(i):
    import torch

    c = draw(i)
    w = Workload(name="random", B=c["B"], T=c["T"], in_dtype=c["in_dtype"], out_dtype=c["out_dtype"], sr=c["sr"],
                 n_fft=c["n_fft"], hop=c["hop"], win_length=c["win_length"], n_mels=c["n_mels"], f_min=c["f_min"],
                 f_max=c["f_max"], power=c["power"], mel_scale=c["mel_scale"], norm=c["norm"],
                 recipe=RECIPE[c["in_dtype"]], seed=c["seed"])
    x = make_input(w)
    try:
        plan = fb.fm_plan_create_ex(w.sr, w.n_fft, w.hop, w.win_length, w.n_mels, w.f_min, w.f_max, w.power,
                                    w.mel_scale, w.norm, w.in_dtype, w.out_dtype, c["center"], c["pad_mode"],
                                    c["pad"], c["normalized"])
    except fb.FmError as e:
        if e.status == fb.FM_ERR_UNSUPPORTED:
            pytest.skip(f"no kernel fits this hop: {c}")
        raise
    try:
        nf = fb.fm_n_frames(plan, w.T)
        assert nf >= 1, c
        xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
        out = torch.full((w.B, w.n_mels, nf), float("nan"), dtype=torch_dtype(w.out_dtype), device="cuda")
        fb.fm_mel_forward(plan, xd.data_ptr(), w.B, w.T, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert fb.fm_plan_poll_error(plan) == fb.FM_OK
        got = out.double().cpu().numpy()
    finally:
        fb.fm_plan_destroy(plan)
    ref = o.mel_spectrogram(x, w.sr, w.n_fft, w.hop, w.n_mels, w.f_min, w.f_max, w.power, w.mel_scale, w.norm,
                            w.win_length, c["center"], c["pad_mode"], c["pad"], c["normalized"])
    if w.out_dtype == "f16":
        check_close_saturating(got, ref, str(c))
    else:
        check_close(got, ref, "f32", str(c))


def test_cases_reach_every_kernel_kind():
    """The draws cover every n_fft and both odd and even hops (so the odd-hop,
    packed, one-frame and large-transform kernels all run)."""
    cases = [draw(i) for i in range(N_CASES)]
    assert {c["n_fft"] for c in cases} == set(SIZES)
    assert any(c["hop"] % 2 for c in cases) and any(c["hop"] % 2 == 0 for c in cases)
    assert any(c["hop"] > c["n_fft"] for c in cases)
    assert dataclasses.is_dataclass(Workload)
