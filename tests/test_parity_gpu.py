"""CUDA path against the float64 oracle, element by element, through the C ABI.

Sizes are cut so the oracle finishes in seconds while still spanning several
tiles and a ragged last tile; the full-size workloads (the launch the bench
times) are checked on whole sampled signals.
"""
from __future__ import annotations

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


@pytest.mark.parametrize("B,in_dtype,recipe", [(4, "f32", "normal"), (5, "i16", "pcm16")])
def test_edge_tiles_moved_to_spare_slots(B, in_dtype, recipe):
    """Batches large enough that the packed kernel runs every signal's first
    and last tile in the third tile group's first slots (more than three tile
    rounds of 152 CTAs), compared element by element with the oracle."""
    import dataclasses

    w = dataclasses.replace(WORKLOADS["speech"].resized(B=B, T=480000 + 37), in_dtype=in_dtype, recipe=recipe)
    tiles = B * -(-(1 + w.T // w.hop) // 32)
    assert tiles >= 2 * 152 + 2 * B  # room for the swap on a 152-SM part
    x = make_input(w)
    check_close(run_gpu(w, x), oracle_for(w, x), w.out_dtype, f"B={B} {in_dtype}")
