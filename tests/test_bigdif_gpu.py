"""The decimation-in-frequency build of the large-transform kernel (n_fft
4096, 8192, 16384 as 16 x M/16: the first 16-point DFTs fused with the load,
then each warp's sub-frames in shared memory with warp barriers only), the
default at 8192 and 16384 and selected at 4096 with FM_MEL_BIG_KERNEL=dif:
every element against the float64 oracle, over ragged tails, odd and long
hops, every pad mode, 16-bit inputs, f16 output and the three |X|^p modes,
under both of its mel mappings (a lane per filter and frame, or a warp per
filter with the lanes over its taps; FM_MEL_BIG_MEL forces one). The
three-pass build it replaced at 8192 and 16384 stays reachable with
FM_MEL_BIG_KERNEL=passes and is checked the same way."""
from __future__ import annotations

import pytest

from mel_spectrogram_gb300 import _binding as fb
from mel_spectrogram_gb300.workloads import WORKLOADS, Workload, make_input
from tests.gpu_util import check_close, check_close_saturating
from tests.test_large_fft_gpu import W, ref, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mel_spectrogram_gb300.build import build

    build()


@pytest.fixture(params=["taps", "lanes"])
def dif(request, monkeypatch):
    monkeypatch.setenv("FM_MEL_BIG_KERNEL", "dif")
    monkeypatch.setenv("FM_MEL_BIG_MEL", request.param)


def info_for(w: Workload) -> dict:
    plan = fb.fm_plan_create(w.sr, w.n_fft, w.hop, w.win_length, w.n_mels, w.f_min, w.f_max, w.power, w.mel_scale,
                             w.norm, w.in_dtype, w.out_dtype)
    try:
        return fb.fm_plan_get_info(plan)
    finally:
        fb.fm_plan_destroy(plan)


@pytest.mark.parametrize("n_fft", [8192, 16384])
def test_default_is_the_dif_build(monkeypatch, n_fft):
    """One group of 512 threads on tiles of 32768 / n_fft frames, and a plan
    that differs from the three-pass build's (two groups of 2-frame tiles at
    8192; a transform buffer of 16 padded sub-frames a frame at 16384)."""
    w = W(n_fft=n_fft, hop=n_fft // 4)
    monkeypatch.delenv("FM_MEL_BIG_KERNEL", raising=False)
    info = info_for(w)
    assert info["threads_per_block"] == 512 and info["frames_per_tile"] == 32768 // n_fft, info
    monkeypatch.setenv("FM_MEL_BIG_KERNEL", "passes")
    passes = info_for(w)
    assert passes != info, (passes, info)
    monkeypatch.setenv("FM_MEL_BIG_KERNEL", "dif")
    assert info_for(w) == info


def test_switch_selects_dif_at_4096(monkeypatch):
    w = W(n_fft=4096, hop=1024)
    monkeypatch.delenv("FM_MEL_BIG_KERNEL", raising=False)
    default = info_for(w)
    monkeypatch.setenv("FM_MEL_BIG_KERNEL", "dif")
    info = info_for(w)
    assert info["threads_per_block"] == 512 and info["frames_per_tile"] == 8, info
    assert default["frames_per_tile"] == 4, default  # the three-pass build: two groups of 4-frame tiles


CASES = [
    dict(n_fft=4096, hop=1024, T=40001),
    dict(n_fft=4096, hop=441, T=20000, power=1.0, mel_scale="slaney", norm="slaney", out_dtype="f16"),
    dict(n_fft=8192, hop=2048, T=60003, n_mels=256),
    dict(n_fft=8192, hop=1001, T=30000, win_length=6000, power=0.5),
    dict(n_fft=16384, hop=4096, T=90001, n_mels=256),
    dict(n_fft=16384, hop=2048, T=40000, mel_scale="slaney", norm="slaney", power=1.0),
    dict(n_fft=16384, hop=5000, T=70000, in_dtype="i16", recipe="pcm16", power=3.0),
    dict(n_fft=16384, hop=16000, T=16385, in_dtype="f16", recipe="music16", B=3),
    dict(n_fft=16384, hop=4096, T=50000, n_mels=7, f_min=300.0, f_max=900.0),
    dict(n_fft=8192, hop=8191, T=8193, n_mels=40, out_dtype="f16"),
    dict(n_fft=8192, hop=512, T=20000, n_mels=1),
]


def ids(k: dict) -> str:
    return f"n{k['n_fft']}h{k['hop']}T{k['T']}m{k.get('n_mels', 128)}"


def check(w: Workload, got, want, what: str) -> None:
    if w.out_dtype == "f16":  # |X|^2 of unit-variance noise leaves the f16 range at n_fft 8192
        check_close_saturating(got, want, what)
    else:
        check_close(got, want, w.out_dtype, what)


@pytest.mark.parametrize("kw", CASES, ids=ids)
def test_dif_build_matches_oracle(dif, kw):
    w = W(**kw)
    x = make_input(w)
    check(w, run(w, x), ref(w, x), str(kw))


@pytest.mark.parametrize("n_fft", [4096, 16384])
@pytest.mark.parametrize("pad_mode", ["reflect", "constant", "replicate", "circular"])
def test_dif_build_framings(dif, n_fft, pad_mode):
    w = W(n_fft=n_fft, hop=n_fft // 4, T=3 * n_fft + 5, n_mels=64)
    x = make_input(w)
    for center, pad in ((True, 0), (False, 0), (True, 77)):
        check_close(run(w, x, center, pad_mode, pad), ref(w, x, center, pad_mode, pad), "f32",
                    f"{n_fft} {pad_mode} center={center} pad={pad}")


def test_dif_build_huge_workload_sampled(dif):
    """The bench's huge batch (16 x 30 s at 44.1 kHz, n_fft 16384, hop 4096,
    256 mels): signals 0 and 15 in full against the oracle."""
    from tests.gpu_util import oracle_for, run_gpu

    w = WORKLOADS["huge"]
    x = make_input(w)
    got = run_gpu(w, x)
    check_close(got[[0, 15]], oracle_for(w, x[[0, 15]]), "f32", "signals 0 and 15")


@pytest.mark.parametrize("kw", [c for c in CASES if c["n_fft"] != 4096], ids=ids)
def test_three_pass_build_matches_oracle(monkeypatch, kw):
    monkeypatch.setenv("FM_MEL_BIG_KERNEL", "passes")
    w = W(**kw)
    x = make_input(w)
    check(w, run(w, x), ref(w, x), str(kw))
