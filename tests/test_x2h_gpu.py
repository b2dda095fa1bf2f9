"""The lane-pair variant of the two-frame packed kernel at n_fft 400, hop 160
(each pass-1 20-point DFT as two 10-point halves on lanes g and g + 16 joined
by a radix-2 step over shuffles, each pass-2 pair split the same way: half
the registers a thread, twice the warps), selected with
FM_MEL_N400_KERNEL=x2h at plan creation: every element against the float64
oracle, like the default kernel it is measured against."""
from __future__ import annotations

import pytest

from mel_spectrogram_gb300 import _binding as fb
from mel_spectrogram_gb300.workloads import WORKLOADS, Workload, make_input
from tests.gpu_util import check_close, oracle_for, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mel_spectrogram_gb300.build import build

    build()


@pytest.fixture
def x2h(monkeypatch):
    monkeypatch.setenv("FM_MEL_N400_KERNEL", "x2h")


def W(**kw) -> Workload:
    base = dict(name="x2h", B=3, T=16001, in_dtype="f32", out_dtype="f32", sr=16000, n_fft=400, hop=160,
                win_length=400, n_mels=128, f_min=0.0, f_max=8000.0, power=2.0, mel_scale="htk", norm=None,
                recipe="normal", seed=14)
    base.update(kw)
    return Workload(**base)


def test_switch_selects_the_lane_pair_kernel(x2h):
    w = W()
    plan = fb.fm_plan_create(w.sr, w.n_fft, w.hop, w.win_length, w.n_mels, w.f_min, w.f_max, w.power, w.mel_scale,
                             w.norm, w.in_dtype, w.out_dtype)
    try:
        info = fb.fm_plan_get_info(plan)
    finally:
        fb.fm_plan_destroy(plan)
    assert info["threads_per_block"] == 992 and info["frames_per_tile"] == 32, info


CASES = [
    dict(),
    dict(T=201, B=2),  # the shortest signal reflect padding allows
    dict(T=7003, power=1.0, mel_scale="slaney", norm="slaney"),
    dict(T=9000, n_mels=64, power=0.5, out_dtype="f16"),
    dict(win_length=300, T=5000),
    dict(in_dtype="i16", recipe="pcm16", T=20000, B=4),
    dict(in_dtype="f16", recipe="music16", T=12345),
]


@pytest.mark.parametrize("kw", CASES, ids=lambda k: "-".join(f"{a}{b}" for a, b in k.items() if a != "recipe") or "speech")
def test_lane_pair_kernel_matches_oracle(x2h, kw):
    w = W(**kw)
    x = make_input(w)
    check_close(run_gpu(w, x), oracle_for(w, x), w.out_dtype, str(kw))


def test_lane_pair_kernel_full_speech_batch(x2h):
    """The bench's speech batch (B = 8 x 480000), signals 0 and 7 in full."""
    w = WORKLOADS["speech"]
    x = make_input(w)
    got = run_gpu(w, x)
    for b in (0, 7):
        check_close(got[b:b + 1], oracle_for(w, x[b:b + 1]), "f32", f"signal {b}")
