"""Even hops on both sides of the packed kernel's shared-memory limits.

The packed two-frame kernel (n_fft 64 to 512) keeps one exchange buffer and
one staged tile per tile group. Once a long hop's staged tile no longer fits
three groups (n_fft 256, 400) or two (512), the plan takes a build with fewer
groups per CTA, and past that (512) the one-frame kernel; torchaudio's
default hop at n_fft 400 (win_length // 2 = 200) is such a hop. At n_fft
1024 and 2048 the one-frame kernel's staged tile stops fitting at long hops
(2048 from ~810 on, half-overlap hop 1024 among them) and the
large-transform kernel, which reads frames straight from the signal, takes
them. At n_fft 64
and 128 the packed kernel runs one group per CTA and takes every hop listed.
Every case checks every output element against the float64 oracle, and the
sizes with longer-hop builds are shown to run more than one over their hop
lists (their CTA or tile sizes differ)."""
from __future__ import annotations

import dataclasses

import pytest

from mel_spectrogram_gb300 import _binding as fb
from mel_spectrogram_gb300.workloads import Workload, make_input
from tests.gpu_util import check_close, oracle_for, plan_for, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mel_spectrogram_gb300.build import build

    build()


# per size: short hops, n_fft/4, n_fft/2, n_fft, and long hops (past the
# three-group packed kernel's staging room at 256-512; on the one-group
# packed kernel at 64 and 128)
HOPS = {
    64: [2, 16, 32, 64, 600, 1200],
    128: [2, 32, 64, 128, 500, 1200],
    256: [2, 64, 128, 256, 500, 700],
    400: [2, 100, 160, 200, 400, 600],
    512: [2, 128, 256, 512, 1200, 1400],
    1024: [2, 256, 512, 2600],
    2048: [2, 512, 1024, 2048, 2999],
}
CASES = [(n, h) for n, hops in HOPS.items() for h in hops]


def W(n_fft: int, hop: int) -> Workload:
    return Workload(name="choice", B=2, T=40 * hop + n_fft + 123, in_dtype="f32", out_dtype="f32", sr=16000,
                    n_fft=n_fft, hop=hop, win_length=n_fft, n_mels=40 if n_fft < 256 else 64, f_min=0.0,
                    f_max=8000.0, power=2.0, mel_scale="htk", norm=None, recipe="normal", seed=n_fft + hop)


@pytest.mark.parametrize("n_fft,hop", CASES, ids=lambda v: str(v))
def test_even_hop_each_kernel(n_fft, hop):
    w = W(n_fft, hop)
    x = make_input(w)
    check_close(run_gpu(w, x), oracle_for(w, x), "f32", f"n_fft={n_fft} hop={hop}")


@pytest.mark.parametrize("n_fft", [256, 400, 512, 1024, 2048])
def test_long_hop_builds_chosen(n_fft):
    shapes = {}
    for hop in HOPS[n_fft]:
        plan = plan_for(W(n_fft, hop))
        try:
            info = fb.fm_plan_get_info(plan)
            shapes[hop] = (info["threads_per_block"], info["frames_per_tile"])
        finally:
            fb.fm_plan_destroy(plan)
    # the shortest hop runs the full packed kernel, the longest a build for long hops
    assert shapes[HOPS[n_fft][0]] != shapes[HOPS[n_fft][-1]], shapes


# the packed kernel's Q = P split (128, 512), its hop-specialised builds
# (128 / 32, 256 / 64, 400 / 100, 512 / 128, 400 / 200 with two groups) and
# an any-hop build (400 / 120) under every power mode, 16-bit input and f16
# output
MODES = [dict(power=1.0), dict(power=0.5, out_dtype="f16"), dict(power=2.0, in_dtype="i16", recipe="pcm16"),
         dict(power=3.0, in_dtype="f16", recipe="music16")]


@pytest.mark.parametrize("mode", MODES, ids=lambda m: "-".join(f"{a}{b}" for a, b in m.items() if a != "recipe"))
@pytest.mark.parametrize("n_fft,hop", [(128, 32), (256, 64), (400, 100), (512, 128), (400, 200), (400, 120)],
                         ids=lambda v: str(v))
def test_power_modes_and_dtypes(n_fft, hop, mode):
    w = dataclasses.replace(W(n_fft, hop), **mode)
    x = make_input(w)
    check_close(run_gpu(w, x), oracle_for(w, x), w.out_dtype, f"n_fft={n_fft} hop={hop} {mode}")
