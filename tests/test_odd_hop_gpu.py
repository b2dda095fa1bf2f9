"""Odd hops (torchaudio accepts any hop, e.g. 441 = 10 ms at 44.1 kHz): every
FFT size against the float64 oracle, with int16 / f16 input, the pad modes,
no centring and unaligned input rows.

An odd hop cannot keep sample pairs aligned in rows of one hop, so these
plans run a build of the one-frame-per-thread kernel that stages each tile as
one contiguous run of samples and reads every sample pair as two samples."""
from __future__ import annotations

import numpy as np
import pytest

from mel_spectrogram_gb300 import _binding as fb
from mel_spectrogram_gb300.workloads import Workload, make_input
from tests.gpu_util import check_close, oracle_for, run_gpu, torch_dtype

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mel_spectrogram_gb300.build import build

    build()


def W(**kw) -> Workload:
    base = dict(name="odd", B=2, T=6001, in_dtype="f32", out_dtype="f32", sr=16000, n_fft=400, hop=441,
                win_length=None, n_mels=64, f_min=0.0, f_max=0.0, power=2.0, mel_scale="htk", norm=None,
                recipe="normal", seed=441)
    base.update(kw)
    if base["win_length"] is None:
        base["win_length"] = base["n_fft"]
    if not base["f_max"]:
        base["f_max"] = base["sr"] / 2
    return Workload(**base)


# (n_fft, hop, T): several tiles and a ragged last tile for every size;
# hop 1 and 3, hops above n_fft, 441 and 221 (10 / 5 ms at 44.1 kHz)
CASES = [
    (64, 1, 300), (64, 17, 3001), (128, 33, 4001), (256, 65, 9001), (256, 301, 12001),
    (400, 441, 30001), (400, 161, 12345), (400, 3, 700), (512, 129, 20001), (1024, 441, 44101),
    (1024, 221, 20001), (2048, 441, 44100), (2048, 511, 30001), (4096, 1023, 40001),
]


@pytest.mark.parametrize("n_fft,hop,T", CASES, ids=lambda v: str(v))
def test_odd_hop_each_size(n_fft, hop, T):
    w = W(n_fft=n_fft, hop=hop, T=T, sr=44100 if hop in (441, 221) else 16000)
    x = make_input(w)
    check_close(run_gpu(w, x), oracle_for(w, x), "f32", f"n_fft={n_fft} hop={hop}")


@pytest.mark.parametrize("in_dtype,recipe,out_dtype", [("i16", "pcm16", "f32"), ("f16", "music16", "f16")])
@pytest.mark.parametrize("n_fft,hop", [(400, 441), (1024, 221), (2048, 441)])
def test_odd_hop_16bit_input(n_fft, hop, in_dtype, recipe, out_dtype):
    w = W(n_fft=n_fft, hop=hop, T=44101, sr=44100, in_dtype=in_dtype, recipe=recipe, out_dtype=out_dtype,
          mel_scale="slaney", norm="slaney")
    x = make_input(w)
    check_close(run_gpu(w, x), oracle_for(w, x), out_dtype, f"{in_dtype} n_fft={n_fft} hop={hop}")


@pytest.mark.parametrize("pad_mode", ["reflect", "constant", "replicate", "circular"])
@pytest.mark.parametrize("n_fft,hop", [(400, 441), (1024, 221)])
def test_odd_hop_framing(n_fft, hop, pad_mode):
    import torch

    import oracle.mel_oracle as o

    w = W(n_fft=n_fft, hop=hop, T=9001)
    x = make_input(w)
    for center, pad in ((True, 0), (True, 7), (False, 0)):
        plan = fb.fm_plan_create_ex(w.sr, n_fft, hop, n_fft, w.n_mels, w.f_min, w.f_max, w.power, w.mel_scale,
                                    w.norm, w.in_dtype, w.out_dtype, center, pad_mode, pad, False)
        try:
            nf = fb.fm_n_frames(plan, w.T)
            xd = torch.from_numpy(x).cuda()
            out = torch.full((w.B, w.n_mels, nf), float("nan"), device="cuda")
            fb.fm_mel_forward(plan, xd.data_ptr(), w.B, w.T, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            assert fb.fm_plan_poll_error(plan) == fb.FM_OK
        finally:
            fb.fm_plan_destroy(plan)
        ref = o.mel_spectrogram(x, w.sr, n_fft, hop, w.n_mels, w.f_min, w.f_max, w.power, w.mel_scale, w.norm,
                                n_fft, center=center, pad_mode=pad_mode, pad=pad)
        check_close(out.double().cpu().numpy(), ref, "f32", f"{pad_mode} center={center} pad={pad}")


@pytest.mark.parametrize("in_dtype,recipe", [("f32", "normal"), ("i16", "pcm16"), ("f16", "music16")])
def test_odd_hop_unaligned_rows(in_dtype, recipe):
    """Rows starting one element off every vector boundary take the element path."""
    import torch

    w = W(n_fft=1024, hop=441, T=20001, in_dtype=in_dtype, recipe=recipe)
    x = make_input(w)
    plan = fb.fm_plan_create(w.sr, w.n_fft, w.hop, w.win_length, w.n_mels, w.f_min, w.f_max, w.power, w.mel_scale,
                             w.norm, w.in_dtype, w.out_dtype)
    try:
        flat = torch.zeros(w.B * w.T + 1, dtype=torch_dtype(in_dtype), device="cuda")
        flat[1:] = torch.from_numpy(x.reshape(-1)).cuda()
        nf = fb.fm_n_frames(plan, w.T)
        out = torch.full((w.B, w.n_mels, nf), float("nan"), device="cuda")
        fb.fm_mel_forward(plan, flat[1:].data_ptr(), w.B, w.T, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
    finally:
        fb.fm_plan_destroy(plan)
    check_close(out.double().cpu().numpy(), oracle_for(w, x), "f32", f"unaligned {in_dtype}")
