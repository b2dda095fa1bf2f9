"""The index-checked debug build (libfm_mel_check.so, compiled with
-DFM_BOUNDS_CHECK): every guarded shared- and global-memory access of every
kernel family tests its index against the buffer it touches, records
FM_ERR_BOUNDS in the plan's error word on a miss and skips the access (it
never traps). Small and ragged cases of each family run through it: no check
may fire (fm_plan_poll_error == FM_OK) and the output must match the float64
oracle, as in the release build.

This stands in for compute-sanitizer, which is closed on this machine."""
from __future__ import annotations

import numpy as np
import pytest

from mel_spectrogram_gb300 import _binding as fb
from mel_spectrogram_gb300.workloads import Workload, make_input
from tests.gpu_util import check_close, oracle_for, torch_dtype

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _check_build():
    from mel_spectrogram_gb300.build import build

    return build(check=True)


def W(**kw) -> Workload:
    base = dict(name="check", B=2, T=6001, in_dtype="f32", out_dtype="f32", sr=16000, n_fft=400, hop=160,
                win_length=None, n_mels=64, f_min=0.0, f_max=8000.0, power=2.0, mel_scale="htk", norm=None,
                recipe="normal", seed=7)
    base.update(kw)
    if base["win_length"] is None:
        base["win_length"] = base["n_fft"]
    return Workload(**base)


def run_checked(w: Workload, x: np.ndarray, center=True, pad_mode="reflect", pad=0) -> np.ndarray:
    """One launch through the debug build; asserts that no index check fired."""
    import torch

    with fb.library(fb.CHECK_LIB_PATH):
        plan = fb.fm_plan_create_ex(w.sr, w.n_fft, w.hop, w.win_length, w.n_mels, w.f_min, w.f_max, w.power,
                                    w.mel_scale, w.norm, w.in_dtype, w.out_dtype, center, pad_mode, pad, False)
        try:
            xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
            nf = fb.fm_n_frames(plan, w.T)
            out = torch.full((w.B, w.n_mels, nf), float("nan"), dtype=torch_dtype(w.out_dtype), device="cuda")
            fb.fm_mel_forward(plan, xd.data_ptr(), w.B, w.T, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            st = fb.fm_plan_poll_error(plan)
        finally:
            fb.fm_plan_destroy(plan)
    assert st == fb.FM_OK, f"debug build reported {fb.status_string(st)}"
    return out.double().cpu().numpy()


CASES = [
    # two-frame kernel: the hop-160 build, any even hop, 256 and 64; the Q = P
    # split at 128 (one group per CTA) and 512 (two groups)
    dict(n_fft=400, hop=160, T=16000, n_mels=128, B=3),
    dict(n_fft=400, hop=160, T=201),  # the shortest signal reflect padding allows
    dict(n_fft=400, hop=160, T=200037, B=4, n_mels=128),  # signals' first / last tiles swapped into spare slots
    dict(n_fft=400, hop=100, T=5001, in_dtype="i16", recipe="pcm16"),
    dict(n_fft=256, hop=64, T=6001, mel_scale="slaney", norm="slaney"),
    dict(n_fft=64, hop=16, T=3001, n_mels=40),
    dict(n_fft=128, hop=32, T=4001),
    dict(n_fft=512, hop=128, T=9001, n_mels=128),
    dict(n_fft=512, hop=64, T=20001, n_mels=128, B=3, power=1.0, out_dtype="f16"),
    # long even hops: the packed kernel with two groups (400) and one (256),
    # and the one-frame kernel past that (512)
    dict(n_fft=400, hop=200, T=12001, n_mels=128),
    dict(n_fft=256, hop=700, T=30001),
    dict(n_fft=512, hop=1400, T=60001),
    # the large-transform kernel at hops too long for the one-frame kernel
    dict(n_fft=2048, hop=1024, T=30001, n_mels=128),
    dict(n_fft=1024, hop=2600, T=40001, in_dtype="i16", recipe="pcm16"),
    # one frame per thread: 1024, 2048
    dict(n_fft=1024, hop=256, T=9001, in_dtype="f16", recipe="music16"),
    dict(n_fft=2048, hop=512, T=12345, out_dtype="f16", power=1.0),
    # odd hops (contiguous staging)
    dict(n_fft=400, hop=441, T=30001, sr=44100, f_max=22050.0),
    dict(n_fft=1024, hop=221, T=20001, in_dtype="i16", recipe="pcm16"),
    # shared-memory passes: a staged span and one too large to stage
    dict(n_fft=4096, hop=1024, T=40001),
    dict(n_fft=16384, hop=4096, T=50001, sr=44100, f_max=22050.0, n_mels=128),
    dict(n_fft=8192, hop=8000, T=40001),
]


@pytest.mark.parametrize("kw", CASES, ids=lambda k: "-".join(f"{a}{b}" for a, b in k.items() if a != "recipe"))
def test_debug_build_checks_pass(kw):
    w = W(**kw)
    x = make_input(w)
    check_close(run_checked(w, x), oracle_for(w, x), w.out_dtype, str(kw))


@pytest.mark.parametrize("pad_mode", ["constant", "replicate", "circular"])
@pytest.mark.parametrize("n_fft,hop", [(400, 100), (1024, 256), (4096, 1024)])
def test_debug_build_framing(n_fft, hop, pad_mode):
    import oracle.mel_oracle as o

    w = W(n_fft=n_fft, hop=hop, T=3 * n_fft + 17)
    x = make_input(w)
    for center, pad in ((True, 5), (False, 0)):
        ref = o.mel_spectrogram(x, w.sr, n_fft, hop, w.n_mels, w.f_min, w.f_max, w.power, w.mel_scale, w.norm,
                                n_fft, center=center, pad_mode=pad_mode, pad=pad)
        check_close(run_checked(w, x, center, pad_mode, pad), ref, "f32", f"{pad_mode} center={center} pad={pad}")
