"""fm_mel_forward_host_noalloc against fm_mel_forward_host, through the C ABI.

The no-allocation entry point serves callers that hold audio in host memory
but cannot allocate device memory when they want a spectrogram (a real-time
audio callback, or a process whose device memory belongs to another
allocator): it stages input and output in the library's static device array
instead of caller buffers. Its results must equal those of the host-buffer
entry point with caller-supplied device buffers, on consecutive calls that
reuse the shared array. This file is named to run after every other test.
"""
from __future__ import annotations

import numpy as np
import pytest

from mel_spectrogram_gb300 import _binding as fb
from mel_spectrogram_gb300.workloads import WORKLOADS, make_input
from tests.gpu_util import check_close, plan_for, torch_dtype

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mel_spectrogram_gb300.build import build

    build()


def _host(x: np.ndarray):
    import torch

    return torch.from_numpy(np.ascontiguousarray(x)).pin_memory()


def _both(w, plan, x: np.ndarray):
    """(caller-scratch result, no-alloc result) for one input, as float64."""
    import torch

    B, T = x.shape
    nf = fb.fm_n_frames(plan, T)
    s = torch.cuda.current_stream()
    h_in = _host(x)
    h_ref = torch.full((B, w.n_mels, nf), float("nan"), dtype=torch_dtype(w.out_dtype)).pin_memory()
    h_got = torch.full((B, w.n_mels, nf), float("nan"), dtype=torch_dtype(w.out_dtype)).pin_memory()
    d_in = torch.empty((B, T), dtype=torch_dtype(w.in_dtype), device="cuda")
    d_out = torch.empty((B, w.n_mels, nf), dtype=torch_dtype(w.out_dtype), device="cuda")
    fb.fm_mel_forward_host(plan, h_in.data_ptr(), B, T, h_ref.data_ptr(), d_in.data_ptr(), d_out.data_ptr(),
                           s.cuda_stream)
    fb.fm_mel_forward_host_noalloc(plan, h_in.data_ptr(), B, T, h_got.data_ptr(), s.cuda_stream)
    s.synchronize()
    assert fb.fm_plan_poll_error(plan) == fb.FM_OK
    return h_ref.double().numpy(), h_got.double().numpy()


@pytest.mark.parametrize("name,B,T", [("speech", 2, 48000 + 37), ("int16", 3, 20011), ("music", 1, 44100 + 123),
                                      ("speech", 8, 480000)])
def test_noalloc_matches_caller_scratch_on_consecutive_calls(name, B, T):
    w = WORKLOADS[name].resized(B=B, T=T)
    plan = plan_for(w)
    try:
        for seed in (101, 202):  # two calls in a row on the shared array, different inputs
            x = make_input(w, seed=seed)
            ref, got = _both(w, plan, x)
            check_close(got, ref, w.out_dtype, f"{name} B={B} T={T} seed={seed}")
    finally:
        fb.fm_plan_destroy(plan)


def test_noalloc_rejects_calls_beyond_the_staging_array():
    w = WORKLOADS["speech"]
    plan = plan_for(w)
    try:
        B, T = 10, 480000  # 19.2 MB in + 15.4 MB out > 32 MiB: rejected before any copy
        in_b = -(-B * T * 4 // 256) * 256
        assert in_b + B * w.n_mels * (1 + T // w.hop) * 4 > fb.FM_NOALLOC_MAX_BYTES
        h = np.zeros(1, np.float32)
        st = fb.lib().fm_mel_forward_host_noalloc(plan, h.ctypes.data, B, T, h.ctypes.data, None)
        assert st == fb.FM_ERR_INVALID_ARG
        with pytest.raises(fb.FmError, match="staging array"):
            fb.fm_mel_forward_host_noalloc(plan, h.ctypes.data, B, T, h.ctypes.data)
    finally:
        fb.fm_plan_destroy(plan)
