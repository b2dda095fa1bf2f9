"""Batches past 2^31 samples and 2^31 output elements, on every kernel family.

Two signals of T = 2^31 + 800 or 2^31 + 777 int16 samples (8.6 GB): sample
offsets pass 2^32 in the second signal, output offsets pass 2^31 in the
second signal's upper mels, and T = 2^31 + 777 makes the second signal start
off the 16-byte grid (no tensor-map or bulk copies for it). The output is
filled with NaN first and must come back finite everywhere (every element
written); sampled frames -- both edges, the frames around sample 2^31, and a
seeded random interior block -- are compared with the float64 oracle on the
slice of the signal that those frames read.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle.mel_oracle as o
from mel_spectrogram_gb300 import _binding as fb
from mel_spectrogram_gb300.workloads import Workload, make_input_device
from tests.gpu_util import check_close, torch_dtype

pytestmark = pytest.mark.gpu

BIG = 1 << 31


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mel_spectrogram_gb300.build import build

    build()


def W(n_fft, hop, T, out_dtype, n_mels=128):
    return Workload("max", 2, T, "i16", out_dtype, 16000, n_fft, hop, n_fft, n_mels, 0.0, 8000.0, 2.0, "htk", None,
                    "pcm16", 11)


def ref_block(w: Workload, row, t0: int, t1: int, n_frames: int) -> np.ndarray:
    """Oracle frames [t0, t1) of one centred (reflect-padded) device signal
    `row`, computed on the part of the signal those frames read."""
    half, hop, T = w.n_fft // 2, w.hop, w.T
    args = (w.sr, w.n_fft, hop, w.n_mels, w.f_min, w.f_max, w.power, w.mel_scale, w.norm, w.win_length)
    if t0 * hop - half >= 0 and (t1 - 1) * hop + half <= T:
        # interior: the frames read x[t0 hop - half, (t1 - 1) hop + half), no padding
        seg = row[t0 * hop - half : (t1 - 1) * hop + half].cpu().numpy()
        return o.mel_spectrogram(seg[None], *args, center=False)[0]
    if t0 * hop - half < 0:
        # left edge: a centred prefix reflects the same samples into its first frames
        assert t1 * hop + w.n_fft < T
        seg = row[: t1 * hop + w.n_fft].cpu().numpy()
        return o.mel_spectrogram(seg[None], *args)[0][:, t0:t1]
    # right edge: a centred suffix starting on a frame boundary, early enough
    # that its own left padding reaches none of the compared frames
    k0 = t0 - (half + hop - 1) // hop - 1
    seg = row[k0 * hop :].cpu().numpy()
    sub = o.mel_spectrogram(seg[None], *args)[0]
    assert sub.shape[1] == n_frames - k0
    return sub[:, t0 - k0 : t1 - k0]


# every case passes 2^32 in sample offsets; all but the last also 2^31 in output offsets
CASES = [
    dict(n_fft=400, hop=160, T=BIG + 800, out_dtype="f16"),   # packed kernel, tensor-map copies in both signals
    dict(n_fft=400, hop=160, T=BIG + 777, out_dtype="f32"),   # packed kernel, element copies for signal 1
    dict(n_fft=1024, hop=256, T=BIG + 777, out_dtype="f16"),  # one frame per thread group
    dict(n_fft=4096, hop=1024, T=BIG + 777, out_dtype="f16", n_mels=96),  # shared-memory passes
]


@pytest.mark.parametrize("kw", CASES, ids=lambda k: f"n{k['n_fft']}-T{k['T'] - BIG}-{k['out_dtype']}")
def test_beyond_2_to_the_31(kw):
    import torch

    w = W(**kw)
    free, _ = torch.cuda.mem_get_info()
    nf_est = 1 + w.T // w.hop
    need = w.B * w.T * 2 + w.B * w.n_mels * nf_est * (4 if w.out_dtype == "f32" else 2)
    if free < need + (2 << 30):
        pytest.skip(f"needs {need / 1e9:.1f} GB of device memory, {free / 1e9:.1f} GB free")
    plan = fb.fm_plan_create(w.sr, w.n_fft, w.hop, w.win_length, w.n_mels, w.f_min, w.f_max, w.power,
                             w.mel_scale, w.norm, w.in_dtype, w.out_dtype)
    try:
        nf = fb.fm_n_frames(plan, w.T)
        assert nf == nf_est
        x = make_input_device(w, "cuda")
        out = torch.full((w.B, w.n_mels, nf), float("nan"), dtype=torch_dtype(w.out_dtype), device="cuda")
        assert x.numel() > 2 * BIG and (out.numel() > BIG or w.n_fft == 4096)
        s = torch.cuda.current_stream()
        fb.fm_mel_forward(plan, x.data_ptr(), w.B, w.T, out.data_ptr(), s.cuda_stream)
        s.synchronize()
        assert fb.fm_plan_poll_error(plan) == fb.FM_OK
        assert bool(torch.isfinite(out).all()), "an output element was not written"
        rng = np.random.default_rng(5)
        tc = BIG // w.hop
        blocks = [(0, 8), (tc - 4, tc + 4), (nf - 8, nf)]
        r = int(rng.integers(8, nf - 48))
        blocks.append((r, r + 40))
        for b in range(w.B):
            for t0, t1 in blocks:
                got = out[b, :, t0:t1].double().cpu().numpy()
                check_close(got, ref_block(w, x[b], t0, t1, nf), w.out_dtype, f"{kw} b={b} frames [{t0}, {t1})")
        del x, out
    finally:
        fb.fm_plan_destroy(plan)
        torch.cuda.empty_cache()
