"""Edge cases of the CUDA path: degenerate sizes, other FFT sizes and
parameters, every element written, exact dtype conversions, alignment,
streams, host-buffer entry point."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest

from mel_spectrogram_gb300 import _binding as fb
from mel_spectrogram_gb300.workloads import WORKLOADS, Workload, make_input
from tests.gpu_util import check_close, check_close_saturating, oracle_for, plan_for, run_gpu, torch_dtype

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mel_spectrogram_gb300.build import build

    build()


def W(**kw) -> Workload:
    base = dict(name="edge", B=2, T=5000, in_dtype="f32", out_dtype="f32", sr=16000, n_fft=400, hop=160,
                win_length=400, n_mels=80, f_min=0.0, f_max=8000.0, power=2.0, mel_scale="htk", norm=None,
                recipe="normal", seed=99)
    base.update(kw)
    return Workload(**base)


@pytest.mark.parametrize("T", [201, 202, 250, 359, 400, 401, 5119])
def test_short_and_ragged_signals_400(T):
    w = W(T=T)
    x = make_input(w)
    check_close(run_gpu(w, x), oracle_for(w, x), "f32", f"T={T}")


@pytest.mark.parametrize("n_fft", [64, 128, 256, 512, 1024, 2048])
def test_minimum_length_each_size(n_fft):
    w = W(n_fft=n_fft, win_length=n_fft, hop=n_fft // 4, T=n_fft // 2 + 1, n_mels=32)
    x = make_input(w)
    check_close(run_gpu(w, x), oracle_for(w, x), "f32", f"n_fft={n_fft}")


SIZES = [
    dict(n_fft=64, hop=16, n_mels=40, T=3000),
    dict(n_fft=128, hop=32, n_mels=64, T=4000, f_min=60.0),
    dict(n_fft=256, hop=64, n_mels=128, T=6000, mel_scale="slaney"),
    dict(n_fft=512, hop=128, n_mels=256, T=9000, norm="slaney"),
    dict(n_fft=1024, hop=256, n_mels=80, T=9001, power=1.0),
    dict(n_fft=2048, hop=512, n_mels=128, T=12345, power=0.5, out_dtype="f16"),
    dict(n_fft=400, hop=100, n_mels=1, T=4000, f_min=300.0, f_max=3400.0),
    dict(n_fft=400, hop=2, n_mels=40, T=600),
    dict(n_fft=256, hop=300, n_mels=20, T=5000),  # hop > n_fft: samples skipped
    dict(n_fft=1024, hop=160, n_mels=128, T=7000, power=3.0, mel_scale="slaney", norm="slaney"),
]


@pytest.mark.parametrize("kw", SIZES, ids=lambda k: "-".join(f"{a}{b}" for a, b in k.items()))
def test_other_sizes_and_parameters(kw):
    kw = dict(kw)
    kw.setdefault("win_length", kw["n_fft"])
    w = W(**kw)
    x = make_input(w)
    check_close(run_gpu(w, x), oracle_for(w, x), w.out_dtype, str(kw))


@pytest.mark.parametrize("n_fft,win", [(400, 320), (1024, 600), (2048, 1999), (64, 17)])
def test_window_shorter_than_frame(n_fft, win):
    w = W(n_fft=n_fft, win_length=win, hop=n_fft // 4, T=4 * n_fft + 7, n_mels=40)
    x = make_input(w)
    check_close(run_gpu(w, x), oracle_for(w, x), "f32", f"win={win}")


def test_empty_filters_are_exact_zeros():
    w = W(n_mels=128, T=16000)
    x = make_input(w)
    got = run_gpu(w, x)
    _, ln, _, _ = fb.fm_mel_filterbank_csr(16000, 400, 128, 0.0, 8000.0, "htk", None)
    empty = np.nonzero(ln == 0)[0]
    assert empty.size > 0
    assert np.all(got[:, empty, :] == 0.0)


def test_batch_zero_is_a_no_op_and_short_signal_is_rejected():
    import torch

    w = W()
    plan = plan_for(w)
    try:
        out = torch.full((4,), 7.0, device="cuda")
        fb.fm_mel_forward(plan, 0, 0, 5000, 0, 0)
        torch.cuda.synchronize()
        assert torch.all(out == 7.0)
        x = torch.zeros((1, 200), device="cuda")
        with pytest.raises(fb.FmError) as e:
            fb.fm_mel_forward(plan, x.data_ptr(), 1, 200, out.data_ptr(), 0)
        assert e.value.status == fb.FM_ERR_INVALID_ARG
        with pytest.raises(fb.FmError):
            fb.fm_mel_forward(plan, x.data_ptr(), -1, 300, out.data_ptr(), 0)
        assert fb.fm_plan_poll_error(plan) == fb.FM_OK
    finally:
        fb.fm_plan_destroy(plan)


def test_every_element_written_and_redzone_untouched():
    import torch

    w = W(B=3, T=7777, n_mels=96)
    x = torch.from_numpy(make_input(w)).cuda()
    plan = plan_for(w)
    try:
        nf = fb.fm_n_frames(plan, w.T)
        n = w.B * w.n_mels * nf
        buf = torch.full((n + 4096,), float("nan"), device="cuda")
        buf[n:] = 12345.0
        fb.fm_mel_forward(plan, x.data_ptr(), w.B, w.T, buf.data_ptr(), 0)
        torch.cuda.synchronize()
        assert torch.isfinite(buf[:n]).all()
        assert torch.all(buf[n:] == 12345.0)
    finally:
        fb.fm_plan_destroy(plan)


def test_deterministic():
    w = WORKLOADS["speech"].resized(B=2, T=30000)
    x = make_input(w)
    a, b = run_gpu(w, x), run_gpu(w, x)
    assert np.array_equal(a, b)


def test_int16_and_f16_inputs_convert_exactly():
    """int16 x / 32768 and f16 widen exactly: same output bits as f32 input."""
    w16 = W(in_dtype="i16", recipe="pcm16", T=9000)
    xi = make_input(w16)
    a = run_gpu(w16, xi)
    b = run_gpu(W(T=9000), (xi.astype(np.float64) / 32768.0).astype(np.float32))
    assert np.array_equal(a, b)
    wh = W(in_dtype="f16", recipe="music16", T=9000)
    xh = make_input(wh)
    c = run_gpu(wh, xh)
    d = run_gpu(W(T=9000), xh.astype(np.float32))
    assert np.array_equal(c, d)


@pytest.mark.parametrize("tag", ["f32", "i16", "f16"])
def test_unaligned_input_pointer(tag):
    """Rows that start off any vector boundary (odd element offsets)."""
    import torch

    recipe = {"f32": "normal", "i16": "pcm16", "f16": "music16"}[tag]
    w = W(in_dtype=tag, recipe=recipe, B=3, T=4001)
    x = make_input(w)
    big = torch.zeros(w.B * w.T + 3, dtype=torch_dtype(tag), device="cuda")
    big[1 : 1 + w.B * w.T] = torch.from_numpy(x.reshape(-1)).cuda()
    plan = plan_for(w)
    try:
        nf = fb.fm_n_frames(plan, w.T)
        out = torch.empty((w.B, w.n_mels, nf), device="cuda")
        fb.fm_mel_forward(plan, big.data_ptr() + big.element_size(), w.B, w.T, out.data_ptr(), 0)
        torch.cuda.synchronize()
        check_close(out.double().cpu().numpy(), oracle_for(w, x), "f32", tag)
    finally:
        fb.fm_plan_destroy(plan)


def test_side_stream_and_transform_module():
    import torch

    from mel_spectrogram_gb300 import MelSpectrogram

    w = W(B=6, T=8000)
    x = make_input(w)
    s = torch.cuda.Stream()
    got = run_gpu(w, x, stream=s)
    check_close(got, oracle_for(w, x), "f32", "side stream")
    mel = MelSpectrogram(sample_rate=16000, n_fft=400, hop_length=160, n_mels=80, f_max=8000.0)
    y = mel(torch.from_numpy(x.reshape(2, 3, w.T)).cuda())
    assert tuple(y.shape) == (2, 3, 80, 1 + w.T // 160)
    check_close(y.reshape(6, 80, -1).double().cpu().numpy(), oracle_for(w, x), "f32", "module")
    with pytest.raises(ValueError):
        mel(torch.zeros(10, 1000))
    mel.close()


def test_transform_module_refusals_dtypes_and_empty_batch():
    """MelSpectrogram refuses what it cannot compute (autograd input, float64,
    a signal too short to reflect, a mismatched out=) and runs int16 / f16
    inputs, f16 output and an empty batch through the same C-ABI path."""
    import torch

    from mel_spectrogram_gb300 import MelSpectrogram

    w = WORKLOADS["tiny"].resized(B=2, T=4003)
    mel = MelSpectrogram(sample_rate=16000, n_fft=400, hop_length=160, n_mels=80, f_max=8000.0)
    mel16 = MelSpectrogram(sample_rate=16000, n_fft=400, hop_length=160, n_mels=80, f_max=8000.0,
                           dtype=torch.float16)
    try:
        x = torch.from_numpy(make_input(w)).cuda().requires_grad_(True)
        with pytest.raises(RuntimeError):
            mel(x)
        with torch.no_grad():
            y = mel(x)
        check_close(y.double().cpu().numpy(), oracle_for(w, make_input(w)), "f32", "no_grad input")
        with pytest.raises(TypeError):
            mel(torch.zeros(2, 4000, dtype=torch.float64, device="cuda"))
        with pytest.raises(fb.FmError):
            mel(torch.zeros(1, 200, device="cuda"))  # reflect padding needs T > n_fft / 2
        with pytest.raises(ValueError):
            mel(x.detach(), out=torch.empty(2, 80, 10, device="cuda"))
        for tag, recipe in (("i16", "pcm16"), ("f16", "music16")):
            wt = dataclasses.replace(w, in_dtype=tag, recipe=recipe)
            xt = make_input(wt)
            got = mel(torch.from_numpy(xt).cuda()).double().cpu().numpy()
            check_close(got, oracle_for(wt, xt), "f32", f"module {tag} input")
        xf = make_input(w)
        got16 = mel16(torch.from_numpy(xf).cuda())
        assert got16.dtype == torch.float16
        check_close(got16.double().cpu().numpy(), oracle_for(w, xf), "f16", "module f16 output")
        y0 = mel(torch.zeros(0, 4003, device="cuda"))
        assert tuple(y0.shape) == (0, 80, 26)
    finally:
        mel.close()
        mel16.close()


def test_host_buffer_entry_point_matches_device_path():
    import torch

    w = WORKLOADS["speech"].resized(B=2, T=24000)
    x = make_input(w)
    plan = plan_for(w)
    try:
        nf = fb.fm_n_frames(plan, w.T)
        h_in = torch.from_numpy(x).pin_memory()
        h_out = torch.empty((w.B, w.n_mels, nf), dtype=torch.float32).pin_memory()
        d_in = torch.empty((w.B, w.T), device="cuda")
        d_out = torch.empty((w.B, w.n_mels, nf), device="cuda")
        s = torch.cuda.current_stream()
        fb.fm_mel_forward_host(plan, h_in.data_ptr(), w.B, w.T, h_out.data_ptr(), d_in.data_ptr(),
                               d_out.data_ptr(), s.cuda_stream)
        s.synchronize()
        assert np.array_equal(h_out.numpy().astype(np.float64), run_gpu(w, x, plan=plan))
    finally:
        fb.fm_plan_destroy(plan)


@pytest.mark.parametrize("B", [1, 3, 5, 9])
def test_host_buffer_entry_point_orders_with_the_stream(B):
    """The chunked copy-in / kernel / copy-out pipeline starts after the work
    already queued on the caller's stream and the stream waits for all of it:
    here the input reaches its pinned host buffer through a device-to-host copy
    queued just before the call, on a side stream, and two calls in a row
    reuse the buffers."""
    import torch

    # 1.44 MB of input + output per signal: B = 1 runs on the caller's stream,
    # B = 3, 5, 9 make 2, 3 and 4 chunks of uneven sizes
    w = WORKLOADS["speech"].resized(B=B, T=200000 + 37 * B)
    plan = plan_for(w)
    try:
        nf = fb.fm_n_frames(plan, w.T)
        s = torch.cuda.Stream()
        d_in = torch.empty((w.B, w.T), device="cuda")
        d_out = torch.full((w.B, w.n_mels, nf), float("nan"), device="cuda")
        h_in = torch.zeros((w.B, w.T), dtype=torch.float32).pin_memory()
        h_out = torch.zeros((w.B, w.n_mels, nf), dtype=torch.float32).pin_memory()
        for seed in (3, 4):
            x = make_input(dataclasses.replace(w, seed=seed))
            src = torch.from_numpy(x).cuda()
            torch.cuda.synchronize()
            with torch.cuda.stream(s):
                torch.cuda._sleep(2_000_000)  # the copy below lands well after the call returns
                h_in.copy_(src, non_blocking=True)
                fb.fm_mel_forward_host(plan, h_in.data_ptr(), w.B, w.T, h_out.data_ptr(), d_in.data_ptr(),
                                       d_out.data_ptr(), s.cuda_stream)
            s.synchronize()
            assert np.array_equal(h_out.numpy().astype(np.float64), run_gpu(w, x, plan=plan)), seed
    finally:
        fb.fm_plan_destroy(plan)


def test_host_buffer_entry_point_in_a_cuda_graph():
    """The plan's three streams fork from and join the capturing stream, so a
    multi-chunk call records into a CUDA graph whose replays recompute h_out."""
    import torch

    w = WORKLOADS["speech"].resized(B=4, T=480000)
    plan = plan_for(w)
    try:
        nf = fb.fm_n_frames(plan, w.T)
        x1, x2 = make_input(w), make_input(dataclasses.replace(w, seed=9))
        h_in = torch.from_numpy(x1).pin_memory()
        h_out = torch.zeros((w.B, w.n_mels, nf), dtype=torch.float32).pin_memory()
        d_in = torch.empty((w.B, w.T), device="cuda")
        d_out = torch.empty((w.B, w.n_mels, nf), device="cuda")
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fb.fm_mel_forward_host(plan, h_in.data_ptr(), w.B, w.T, h_out.data_ptr(), d_in.data_ptr(),
                                   d_out.data_ptr(), torch.cuda.current_stream().cuda_stream)
        for x in (x1, x2):
            h_in.copy_(torch.from_numpy(x))
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(h_out.numpy().astype(np.float64), run_gpu(w, x, plan=plan))
    finally:
        fb.fm_plan_destroy(plan)


def test_host_buffer_entry_point_from_two_threads():
    """Calls on one plan from two host threads, each with its own stream and
    buffers: the plan serialises their queuing and every result is right."""
    import threading

    import torch

    w = WORKLOADS["speech"].resized(B=3, T=300000)
    plan = plan_for(w)
    nf = fb.fm_n_frames(plan, w.T)
    xs = [make_input(dataclasses.replace(w, seed=20 + i)) for i in range(2)]
    want = [run_gpu(w, x, plan=plan) for x in xs]
    errors = []

    def worker(i):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            h_in = torch.from_numpy(xs[i]).pin_memory()
            h_out = torch.zeros((w.B, w.n_mels, nf), dtype=torch.float32).pin_memory()
            d_in = torch.empty((w.B, w.T), device="cuda")
            d_out = torch.empty((w.B, w.n_mels, nf), device="cuda")
            for _ in range(20):
                h_out.zero_()
                fb.fm_mel_forward_host(plan, h_in.data_ptr(), w.B, w.T, h_out.data_ptr(), d_in.data_ptr(),
                                       d_out.data_ptr(), s.cuda_stream)
                s.synchronize()
                if not np.array_equal(h_out.numpy().astype(np.float64), want[i]):
                    errors.append(f"thread {i}: wrong output")
                    return
        except Exception as e:  # reported below
            errors.append(f"thread {i}: {e!r}")

    try:
        ts = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
        assert not errors, errors
    finally:
        fb.fm_plan_destroy(plan)


def test_plan_info():
    w = WORKLOADS["speech"]
    plan = plan_for(w)
    try:
        info = fb.fm_plan_get_info(plan)
        assert info["n_freqs"] == 201 and info["n_mels"] == 128
        assert info["grid_limit"] >= info["blocks_per_sm"] >= 1
        assert info["smem_bytes"] > 0 and info["threads_per_block"] % 32 == 0
        assert info["nnz"] > 0
    finally:
        fb.fm_plan_destroy(plan)


@pytest.mark.parametrize("kw", [
    dict(n_fft=400, hop=160, n_mels=128, T=16000, scale=12.0),  # two-frame kernel
    dict(n_fft=1024, hop=256, n_mels=80, T=20000, scale=8.0),
    dict(n_fft=2048, hop=512, n_mels=128, T=30000, scale=300.0, power=1.0, in_dtype="f16"),
    dict(n_fft=8192, hop=2048, n_mels=128, T=40000, scale=0.7),  # shared-memory passes
], ids=lambda k: f"n{k['n_fft']}")
def test_f16_output_saturates_to_inf(kw):
    """Loud signals whose mel values straddle the f16 range: +inf exactly where
    the float64 oracle overflows f16, the f16 tolerance elsewhere."""
    kw = dict(kw)
    scale = kw.pop("scale")
    in_dtype = kw.pop("in_dtype", "f32")
    w = W(out_dtype="f16", in_dtype=in_dtype, win_length=kw["n_fft"], **kw)
    x = (make_input(dataclasses.replace(w, in_dtype="f32", recipe="normal")).astype(np.float64) * scale)
    x = x.astype(np.float16 if in_dtype == "f16" else np.float32)
    ref = oracle_for(w, x)
    n_inf, n_fin = check_close_saturating(run_gpu(w, x), ref, str(kw))
    assert n_inf > 0 and n_fin > 0, (n_inf, n_fin)  # the case really straddles the range
