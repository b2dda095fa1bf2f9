"""CUDA path against the float64 oracle, element by element, through the C ABI.

Sizes are cut so the oracle finishes in seconds while still spanning several
tiles and a ragged last tile; the full-size workloads (the launch the bench
times) are checked on whole sampled signals.
"""
from __future__ import annotations

import numpy as np
import pytest

from mel_spectrogram_gb300.workloads import ORDER, WORKLOADS, make_input
from tests.gpu_util import check_close, oracle_for, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mel_spectrogram_gb300.build import build

    build()


# reduced (B, T) per workload: several tiles, ragged tail, odd sample counts
REDUCED = {
    "tiny": (1, 16000),
    "speech": (2, 48000 + 37),
    "int16": (3, 20011),
    "pow2": (4, 32768),
    "music": (2, 44100 + 123),
}


@pytest.mark.parametrize("name", ORDER)
def test_workload_parity_reduced(name):
    w = WORKLOADS[name].resized(*REDUCED[name])
    x = make_input(w)
    check_close(run_gpu(w, x), oracle_for(w, x), w.out_dtype, name)


@pytest.mark.parametrize("name", ["speech", "int16", "pow2", "music"])
def test_workload_parity_full_size_sampled_rows(name):
    """Full B x T launch (the bench's configuration); whole signals sampled."""
    w = WORKLOADS[name]
    x = make_input(w)
    got = run_gpu(w, x)
    for b in sorted({0, w.B // 2 + 1, w.B - 1}):
        ref = oracle_for(w.resized(B=1), x[b : b + 1])
        check_close(got[b : b + 1], ref, w.out_dtype, f"{name}[b={b}]")
