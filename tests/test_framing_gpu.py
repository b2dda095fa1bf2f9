"""The torchaudio framing options on the CUDA path against the float64 oracle.

flashmel README "Usage" lists pad, center, pad_mode and normalized among the
supported MelSpectrogram arguments; "How it works" applies the padding (all
four pad modes) as index arithmetic and folds the normalisation into the
window. Every output element is compared, through the C ABI
(fm_plan_create_ex), for both kernels (the packed one at n_fft 400 / 256,
with and without the compile-time hop, and the one-frame-per-thread one at
1024 / 2048), on signals that put every tile edge, the shortest legal
lengths and the zero padding in play.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle.mel_oracle as o
from mel_spectrogram_gb300 import _binding as fb
from mel_spectrogram_gb300.workloads import Workload, make_input
from tests.gpu_util import check_close, torch_dtype

pytestmark = pytest.mark.gpu

MODES = ["reflect", "constant", "replicate", "circular"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mel_spectrogram_gb300.build import build

    build()


def W(**kw) -> Workload:
    base = dict(name="framing", B=2, T=5000, in_dtype="f32", out_dtype="f32", sr=16000, n_fft=400, hop=160,
                win_length=400, n_mels=80, f_min=0.0, f_max=8000.0, power=2.0, mel_scale="htk", norm=None,
                recipe="normal", seed=7)
    base.update(kw)
    if "win_length" not in kw:
        base["win_length"] = base["n_fft"]
    return Workload(**base)


def run(w: Workload, x: np.ndarray, center, pad_mode, pad, normalized) -> np.ndarray:
    import torch

    plan = fb.fm_plan_create_ex(w.sr, w.n_fft, w.hop, w.win_length, w.n_mels, w.f_min, w.f_max, w.power,
                                w.mel_scale, w.norm, w.in_dtype, w.out_dtype, center, pad_mode, pad, normalized)
    try:
        B, T = x.shape
        nf = fb.fm_n_frames(plan, T)
        assert nf >= 1
        xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
        out = torch.full((B, w.n_mels, nf), float("nan"), dtype=torch_dtype(w.out_dtype), device="cuda")
        fb.fm_mel_forward(plan, xd.data_ptr(), B, T, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert fb.fm_plan_poll_error(plan) == fb.FM_OK
        return out.double().cpu().numpy()
    finally:
        fb.fm_plan_destroy(plan)


def ref(w: Workload, x: np.ndarray, center, pad_mode, pad, normalized) -> np.ndarray:
    return o.mel_spectrogram(x, w.sr, w.n_fft, w.hop, w.n_mels, w.f_min, w.f_max, w.power, w.mel_scale, w.norm,
                             w.win_length, center, pad_mode, pad, normalized)


KERNELS = [
    dict(n_fft=400, hop=160, T=7003),                # packed, compile-time hop, tensor-map copies
    dict(n_fft=400, hop=100, T=5001, n_mels=64),     # packed, any hop
    dict(n_fft=256, hop=64, T=3001, n_mels=40),      # packed, other split
    dict(n_fft=1024, hop=256, T=9001),               # one frame per thread
    dict(n_fft=2048, hop=512, T=12001, n_mels=128, out_dtype="f16", mel_scale="slaney", norm="slaney"),
]


@pytest.mark.parametrize("kw", KERNELS, ids=lambda k: f"n{k['n_fft']}h{k['hop']}")
@pytest.mark.parametrize("pad_mode", MODES)
@pytest.mark.parametrize("center", [True, False])
def test_pad_modes_and_centring(kw, pad_mode, center):
    w = W(**kw)
    x = make_input(w)
    check_close(run(w, x, center, pad_mode, 0, False), ref(w, x, center, pad_mode, 0, False), w.out_dtype,
                f"{kw} {pad_mode} center={center}")


@pytest.mark.parametrize("kw", KERNELS[:1] + KERNELS[3:4], ids=lambda k: f"n{k['n_fft']}h{k['hop']}")
@pytest.mark.parametrize("pad_mode", MODES)
@pytest.mark.parametrize("pad", [1, 37, 400])
def test_zero_padding_before_centring(kw, pad_mode, pad):
    w = W(**kw)
    x = make_input(w)
    for center in (True, False):
        check_close(run(w, x, center, pad_mode, pad, False), ref(w, x, center, pad_mode, pad, False), w.out_dtype,
                    f"{kw} {pad_mode} pad={pad} center={center}")


@pytest.mark.parametrize("normalized", [True, "window", "frame_length"])
@pytest.mark.parametrize("kw", [KERNELS[0], KERNELS[3], dict(n_fft=400, hop=160, T=4000, win_length=300)],
                         ids=lambda k: f"n{k['n_fft']}w{k.get('win_length', k['n_fft'])}")
def test_normalisation(kw, normalized):
    w = W(**kw)
    x = make_input(w)
    for power in (2.0, 1.0):
        w2 = W(**{**kw, "power": power})
        check_close(run(w2, x, True, "reflect", 0, normalized), ref(w2, x, True, "reflect", 0, normalized), "f32",
                    f"{kw} normalized={normalized} power={power}")


def shortest(n_fft, center, pad_mode, pad):
    """The shortest T the framing accepts."""
    if not center:
        return max(1, n_fft - 2 * pad)
    if pad_mode == "reflect":
        return max(1, n_fft // 2 + 1 - 2 * pad)
    if pad_mode == "circular":
        return max(1, n_fft // 2 - 2 * pad)
    return 1


@pytest.mark.parametrize("n_fft,hop", [(400, 160), (256, 64), (1024, 256)])
@pytest.mark.parametrize("pad_mode", MODES)
@pytest.mark.parametrize("center,pad", [(True, 0), (False, 0), (True, 5)])
def test_shortest_signals(n_fft, hop, pad_mode, center, pad):
    T = shortest(n_fft, center, pad_mode, pad)
    w = W(n_fft=n_fft, hop=hop, win_length=n_fft, T=T, n_mels=40)
    x = make_input(w)
    for Tx in (T, T + 1, T + hop + 3):
        xs = np.ascontiguousarray(make_input(w.resized(T=Tx)))
        check_close(run(w, xs, center, pad_mode, pad, False), ref(w, xs, center, pad_mode, pad, False), "f32",
                    f"n_fft={n_fft} {pad_mode} center={center} pad={pad} T={Tx}")
    del x


@pytest.mark.parametrize("n_fft,hop", [(400, 160), (1024, 256)])
@pytest.mark.parametrize("pad_mode", MODES)
def test_too_short_is_rejected(n_fft, hop, pad_mode):
    import torch

    for center, pad in ((True, 0), (False, 0), (False, 3)):
        T = shortest(n_fft, center, pad_mode, pad) - 1
        if T < 1:
            continue
        plan = fb.fm_plan_create_ex(16000, n_fft, hop, n_fft, 40, 0.0, 8000.0, 2.0, "htk", None, "f32", "f32",
                                    center, pad_mode, pad, False)
        try:
            assert fb.fm_n_frames(plan, T) == -1
            x = torch.zeros((1, max(T, 1)), device="cuda")
            out = torch.zeros(16, device="cuda")
            with pytest.raises(fb.FmError):
                fb.fm_mel_forward(plan, x.data_ptr(), 1, T, out.data_ptr())
        finally:
            fb.fm_plan_destroy(plan)


@pytest.mark.parametrize("in_dtype", ["i16", "f16"])
@pytest.mark.parametrize("pad_mode", MODES)
def test_sixteen_bit_inputs(in_dtype, pad_mode):
    recipe = "pcm16" if in_dtype == "i16" else "music16"
    for kw in (KERNELS[0], KERNELS[3]):
        w = W(**{**kw, "in_dtype": in_dtype, "recipe": recipe, "T": kw["T"] - 2})
        x = make_input(w)
        for center, pad in ((True, 0), (False, 11)):
            check_close(run(w, x, center, pad_mode, pad, False), ref(w, x, center, pad_mode, pad, False), "f32",
                        f"{in_dtype} {kw} {pad_mode} center={center}")


def test_transform_framing_matches_oracle():
    import torch

    from mel_spectrogram_gb300 import MelSpectrogram

    w = W(T=6000)
    x = make_input(w)
    mel = MelSpectrogram(sample_rate=16000, n_fft=400, hop_length=160, n_mels=80, f_max=8000.0, pad=13,
                         center=False, pad_mode="replicate", normalized=True)
    try:
        got = mel(torch.from_numpy(x).cuda()).double().cpu().numpy()
    finally:
        mel.close()
    check_close(got, ref(w, x, False, "replicate", 13, True), "f32", "MelSpectrogram framing")
