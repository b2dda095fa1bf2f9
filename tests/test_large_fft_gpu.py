"""The large transforms (n_fft 4096, 8192, 16384: README "Usage", "400 or a
power of 2 in [64, 16384]") on the CUDA path against the float64 oracle,
element by element through the C ABI: the shared-memory kernel's three
autosorting passes, its split and its CSR projection, over tiles with a
ragged tail, every pad mode with and without centring, 16-bit inputs, f16
output and the Slaney scale with its norm."""
from __future__ import annotations

import numpy as np
import pytest

import oracle.mel_oracle as o
from mel_spectrogram_gb300 import _binding as fb
from mel_spectrogram_gb300.workloads import Workload, make_input
from tests.gpu_util import check_close, torch_dtype

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mel_spectrogram_gb300.build import build

    build()


def W(**kw) -> Workload:
    base = dict(name="large", B=2, T=40000, in_dtype="f32", out_dtype="f32", sr=44100, n_fft=4096, hop=1024,
                n_mels=128, f_min=0.0, f_max=22050.0, power=2.0, mel_scale="htk", norm=None, recipe="normal", seed=5)
    base.update(kw)
    base.setdefault("win_length", base["n_fft"])
    if "win_length" not in kw:
        base["win_length"] = base["n_fft"]
    return Workload(**base)


def run(w: Workload, x: np.ndarray, center=True, pad_mode="reflect", pad=0, normalized=False) -> np.ndarray:
    import torch

    plan = fb.fm_plan_create_ex(w.sr, w.n_fft, w.hop, w.win_length, w.n_mels, w.f_min, w.f_max, w.power,
                                w.mel_scale, w.norm, w.in_dtype, w.out_dtype, center, pad_mode, pad, normalized)
    try:
        B, T = x.shape
        nf = fb.fm_n_frames(plan, T)
        xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
        out = torch.full((B, w.n_mels, nf), float("nan"), dtype=torch_dtype(w.out_dtype), device="cuda")
        fb.fm_mel_forward(plan, xd.data_ptr(), B, T, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert fb.fm_plan_poll_error(plan) == fb.FM_OK
        return out.double().cpu().numpy()
    finally:
        fb.fm_plan_destroy(plan)


def ref(w, x, center=True, pad_mode="reflect", pad=0, normalized=False):
    return o.mel_spectrogram(x, w.sr, w.n_fft, w.hop, w.n_mels, w.f_min, w.f_max, w.power, w.mel_scale, w.norm,
                             w.win_length, center, pad_mode, pad, normalized)


@pytest.mark.parametrize("kw", [
    dict(n_fft=4096, hop=1024, T=40001),
    dict(n_fft=4096, hop=512, T=20000, power=1.0, mel_scale="slaney", norm="slaney", out_dtype="f16"),
    dict(n_fft=8192, hop=2048, T=60003, n_mels=256),
    dict(n_fft=8192, hop=1000, T=30000, win_length=6000, power=0.5),
    dict(n_fft=16384, hop=4096, T=90001, n_mels=256),
    dict(n_fft=16384, hop=2048, T=40000, mel_scale="slaney", norm="slaney", power=1.0),
], ids=lambda k: f"n{k['n_fft']}h{k['hop']}")
def test_large_transforms_match_oracle(kw):
    w = W(**kw)
    x = make_input(w)
    check_close(run(w, x), ref(w, x), w.out_dtype, str(kw))


@pytest.mark.parametrize("n_fft", [4096, 16384])
@pytest.mark.parametrize("pad_mode", ["reflect", "constant", "replicate", "circular"])
def test_large_transform_framings(n_fft, pad_mode):
    w = W(n_fft=n_fft, hop=n_fft // 4, T=3 * n_fft + 5, n_mels=64)
    x = make_input(w)
    for center, pad in ((True, 0), (False, 0), (True, 77)):
        check_close(run(w, x, center, pad_mode, pad), ref(w, x, center, pad_mode, pad), "f32",
                    f"n_fft={n_fft} {pad_mode} center={center} pad={pad}")


@pytest.mark.parametrize("in_dtype,recipe", [("i16", "pcm16"), ("f16", "music16")])
def test_large_transform_sixteen_bit_inputs(in_dtype, recipe):
    w = W(n_fft=8192, hop=2048, T=50001, in_dtype=in_dtype, recipe=recipe)
    x = make_input(w)
    check_close(run(w, x), ref(w, x), "f32", in_dtype)


def test_large_transform_shortest_signal():
    for n_fft in (4096, 8192, 16384):
        w = W(n_fft=n_fft, hop=n_fft // 4, T=n_fft // 2 + 1, n_mels=64)
        x = make_input(w)
        check_close(run(w, x), ref(w, x), "f32", f"n_fft={n_fft} T={w.T}")
