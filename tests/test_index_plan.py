"""The index plans of the two large-transform kernels, checked on the CPU.

A vectorised numpy model of the shared-memory index arithmetic of
`mel_kernel_big` (three autosorting passes over F = 32768 / n_fft frames) and
`mel_kernel_bigdif` (16-point DFTs over the frame, then two passes inside
each of 16 padded sub-frames per frame, each warp on its own sub-frames),
with the radix tables read from the kernel header, so that a change there is
modelled here. For every size it checks that:

  * every butterfly of every pass is taken by exactly one (thread, task);
  * every shared-memory index lies inside the buffer of the thread's group
    (the whole tile, or the warp's sub-frames);
  * every twiddle exponent lies in [0, M) (the two-row W_M table);
  * the transform equals numpy's FFT of the frame (to 1e-12), and the
    split's reads of Z[k] and Z[M - k] land on those values.

This is the check that ran before the first GPU launch of each plan; it
does not run the CUDA code (the GPU tests compare that with the oracle)."""
from __future__ import annotations

import os
import re

import numpy as np
import pytest

HDR = os.path.join(os.path.dirname(__file__), "..", "mel_spectrogram_gb300", "csrc")
THREADS = 512
R0 = 16  # the decimation-in-frequency kernel's first factor


def radix_table(fname: str, struct: str, fields: tuple[str, ...]) -> dict[int, tuple[int, ...]]:
    """{M: (radices...)} from the template specialisations of `struct` in a header."""
    text = open(os.path.join(HDR, fname)).read()
    pat = re.compile(r"struct\s+" + struct + r"<(\d+)>\s*\{\s*static constexpr int ([^;]+);")
    out = {}
    for m, body in pat.findall(text):
        vals = dict((k.strip(), int(v)) for k, v in (a.split("=") for a in body.split(",")))
        out[int(m)] = tuple(vals[f] for f in fields)
    return out


BIG = radix_table("fm_kernel_big.cuh", "BigRadices", ("R0", "R1", "R2"))
DIF = radix_table("fm_kernel_bigdif.cuh", "DifRadices", ("RA", "RB"))


def phys(i):
    return i + (i >> 4)


def frame_stride(m: int) -> int:
    return m + (m >> 4) + 1


def w(L: int, e) -> np.ndarray:
    return np.exp(-2j * np.pi * np.asarray(e) / L)


def stockham_pass(buf: np.ndarray, base: int, cap: int, frames: int, m: int, fs: int, r: int, ns: int,
                  threads: int, tw_scale: int, m_full: int) -> None:
    """One autosorting pass of radix r (ns = product of the earlier radices) over
    `frames` frames of m points at buf[base + f fs + phys(i)], done by `threads`
    threads that each take the tasks tid + t threads, as the kernel's pass does."""
    J = m // r
    assert (frames * J) % threads == 0
    task = np.arange(frames * J)  # tid + t * threads covers these once each
    tids = task % threads
    ts = task // threads
    assert np.array_equal(np.sort(tids + ts * threads), task)
    f, j = task // J, task % J
    rr = np.arange(r)
    src = base + f[:, None] * fs + phys(j[:, None] + rr[None, :] * J)
    assert src.min() >= base and src.max() < cap
    v = buf[src]
    if ns > 1:
        e = (j % ns) * (m // (ns * r))
        t = e[:, None] * rr[None, :] * tw_scale
        assert t.min() >= 0 and t.max() < m_full  # fine row t mod 64, coarse row t / 64
        v = v * w(m_full, t)
    v = np.fft.fft(v, axis=1)
    d = (j // ns) * ns * r + (j % ns)
    dst = base + f[:, None] * fs + phys(d[:, None] + rr[None, :] * ns)
    assert dst.min() >= base and dst.max() < cap
    assert len(np.unique(dst)) == dst.size  # in place: every slot written once
    buf[dst] = v


@pytest.mark.parametrize("n_fft", sorted(2 * m for m in BIG))
def test_three_pass_plan(n_fft):
    M, F = n_fft // 2, 32768 // n_fft
    rad = BIG[M]
    assert np.prod(rad) == M
    FS = frame_stride(M)
    rng = np.random.default_rng(n_fft)
    z = rng.standard_normal((F, M)) + 1j * rng.standard_normal((F, M))
    # two tile groups where the kernel runs them (F frames split, 256 threads each), and one
    for groups in (1, 2) if F >= 2 else (1,):
        Fg, TH = F // groups, THREADS // groups
        buf = np.full(F * FS, np.nan, complex)
        for g in range(groups):
            base = g * Fg * FS
            for f in range(Fg):
                buf[base + f * FS + phys(np.arange(M))] = z[g * Fg + f]
            ns = 1
            for r in rad:
                stockham_pass(buf, base, base + Fg * FS, Fg, M, FS, r, ns, TH, 1, M)
                ns *= r
        for f in range(F):
            got = buf[f * FS + phys(np.arange(M))]
            ref = np.fft.fft(z[f])
            assert np.abs(got - ref).max() <= 1e-12 * np.abs(ref).max()


@pytest.mark.parametrize("n_fft", sorted(2 * R0 * ms for ms in DIF))
def test_dif_plan(n_fft):
    M, F = n_fft // 2, 32768 // n_fft
    MS = M // R0
    RA, RB = DIF[MS]
    assert RA * RB == MS
    SFS = frame_stride(MS)
    NW = THREADS // 32
    SUB = F * R0 // NW  # sub-frames per warp
    cap = F * R0 * SFS
    rng = np.random.default_rng(n_fft + 1)
    z = rng.standard_normal((F, M)) + 1j * rng.standard_normal((F, M))
    buf = np.full(cap, np.nan, complex)
    # step A: task (f, n2) = divmod(tid + t THREADS, MS); value n1 = z[n1 MS + n2]
    task = np.arange(F * MS)
    assert (F * MS) % THREADS == 0
    f, n2 = task // MS, task % MS
    n1 = np.arange(R0)
    v = np.fft.fft(z[f[:, None], n1[None, :] * MS + n2[:, None]], axis=1)  # over n1 -> k1
    t = n2[:, None] * n1[None, :]
    assert t.max() < M
    v = v * w(M, t)
    dst = (f[:, None] * R0 + n1[None, :]) * SFS + phys(n2[:, None])
    assert dst.min() >= 0 and dst.max() < cap and len(np.unique(dst)) == dst.size
    buf[dst] = v
    # step B: warp k holds sub-frames k SUB .. k SUB + SUB - 1; below MS = 512 the
    # first pass runs on 32 RA / MS sub-frames at a time
    for warp in range(NW):
        base = warp * SUB * SFS
        g1 = 32 * RA // MS if MS < 512 else SUB
        for sf in range(0, SUB, g1):
            stockham_pass(buf, base + sf * SFS, cap, g1, MS, SFS, RA, 1, 32, R0, M)
        stockham_pass(buf, base, cap, SUB, MS, SFS, RB, RA, 32, R0, M)
    # the split's reads: Z[k] at sub-frame 16 f + k mod 16, position k / 16
    k = np.arange(M)
    for fr in range(F):
        zk = buf[(fr * R0 + (k & 15)) * SFS + phys(k >> 4)]
        ref = np.fft.fft(z[fr])
        assert np.abs(zk - ref).max() <= 1e-12 * np.abs(ref).max()
        km = (M - k) & (M - 1)
        zm = buf[(fr * R0 + (km & 15)) * SFS + phys(km >> 4)]
        assert np.allclose(zm, ref[km], rtol=0, atol=1e-12 * np.abs(ref).max())
    # the power tile (F rows of M + 1 floats) fits in the buffer it aliases
    assert F * (M + 1) <= 2 * cap


def test_tables_were_read():
    assert {512, 1024, 2048, 4096, 8192} <= set(BIG) and set(DIF) == {128, 256, 512}
