"""Helpers for the GPU tests: run the C-ABI path, compare with the oracle.

Tolerances (the bounds the path is held to, applied element by element):
  fp32 output: |gpu - oracle| <= 1e-4 * (1 + |oracle|)
  f16 output : |gpu - oracle| <= 2e-3 * (1 + |oracle|) everywhere, and
               <= 2e-3 * |oracle| wherever |oracle| >= 6.1e-5 (f16 normals)
"""
from __future__ import annotations

import numpy as np

import oracle.mel_oracle as o
from mel_spectrogram_gb300 import _binding as fb
from mel_spectrogram_gb300.workloads import Workload

TORCH_DTYPES = {"f32": "float32", "i16": "int16", "f16": "float16"}


def torch_dtype(tag):
    import torch

    return getattr(torch, TORCH_DTYPES[tag])


def plan_for(w: Workload, **over):
    p = dict(sr=w.sr, n_fft=w.n_fft, hop=w.hop, win_length=w.win_length, n_mels=w.n_mels, f_min=w.f_min,
             f_max=w.f_max, power=w.power, mel_scale=w.mel_scale, norm=w.norm, in_dtype=w.in_dtype,
             out_dtype=w.out_dtype)
    p.update(over)
    return fb.fm_plan_create(**p)


def run_gpu(w: Workload, x: np.ndarray, plan=None, stream=None) -> np.ndarray:
    """Upload x, launch fm_mel_forward through the C ABI, return float64 output."""
    import torch

    own = plan is None
    plan = plan_for(w) if own else plan
    try:
        xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
        B, T = x.shape
        nf = fb.fm_n_frames(plan, T)
        out = torch.full((B, w.n_mels, nf), float("nan"), dtype=torch_dtype(w.out_dtype), device="cuda")
        s = stream or torch.cuda.current_stream()
        fb.fm_mel_forward(plan, xd.data_ptr(), B, T, out.data_ptr(), s.cuda_stream)
        s.synchronize()
        return out.double().cpu().numpy()
    finally:
        if own:
            fb.fm_plan_destroy(plan)


def oracle_for(w: Workload, x: np.ndarray) -> np.ndarray:
    return o.mel_spectrogram(x, w.sr, w.n_fft, w.hop, w.n_mels, w.f_min, w.f_max, w.power, w.mel_scale, w.norm,
                             w.win_length)


def check_close(got: np.ndarray, ref: np.ndarray, out_dtype: str, what: str = "") -> float:
    """Assert the tolerance rule; return the worst error / allowed ratio."""
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    if got.size == 0:  # e.g. the finite part of an f16 output that saturates everywhere
        return 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite output (unwritten or overflow)"
    err = np.abs(got - ref)
    if out_dtype == "f32":
        allowed = 1e-4 * (1.0 + np.abs(ref))
    else:
        allowed = 2e-3 * (1.0 + np.abs(ref))
        normal = np.abs(ref) >= 6.1e-5
        allowed = np.where(normal, np.minimum(allowed, 2e-3 * np.abs(ref)), allowed)
    ratio = err / allowed
    worst = np.unravel_index(np.argmax(ratio), ratio.shape)
    assert ratio[worst] <= 1.0, (
        f"{what}: |gpu-oracle| = {err[worst]:.3e} > {allowed[worst]:.3e} at {worst} (oracle {ref[worst]:.6e})"
    )
    return float(ratio.max())


# f16 round-to-nearest-even overflows to inf from 65520 up (halfway between the
# largest finite f16, 65504, and 2^16)
F16_OVERFLOW = 65520.0


def check_close_saturating(got: np.ndarray, ref: np.ndarray, what: str = "") -> tuple[int, int]:
    """f16 output where the float64 oracle leaves the f16 range: +inf exactly
    where the oracle rounds to inf, the f16 tolerance elsewhere, and either
    in a narrow band (the f16 tolerance) around the overflow threshold, where
    fp32 and float64 may round to different sides (flashmel README
    "Development": values beyond fp16 range saturate to inf on both sides).
    Returns (elements that must be inf, elements that must be finite)."""
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    band = np.abs(np.abs(ref) - F16_OVERFLOW) <= 2e-3 * F16_OVERFLOW
    must_inf = (np.abs(ref) >= F16_OVERFLOW) & ~band
    must_fin = ~must_inf & ~band
    assert np.all(np.isinf(got[must_inf]) & (np.sign(got[must_inf]) == np.sign(ref[must_inf]))), (
        f"{what}: {int(np.sum(~np.isinf(got[must_inf])))} values beyond the f16 range did not saturate")
    check_close(got[must_fin], ref[must_fin], "f16", what)
    g, r = got[band], ref[band]
    ok = np.isinf(g) | (np.abs(g - r) <= 2e-3 * np.abs(r))
    assert np.all(ok), f"{what}: near the overflow threshold neither inf nor within tolerance"
    return int(must_inf.sum()), int(must_fin.sum())
