"""Host-only tests of the C ABI: no kernel runs here (no GPU needed)."""
from __future__ import annotations

import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle.mel_oracle as o
from mel_spectrogram_gb300 import _binding as fb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fm_mel.h")


@pytest.fixture(scope="module")
def L():
    from mel_spectrogram_gb300.build import build

    build()
    return fb.lib()


def declared_functions() -> list[str]:
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fm_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_what_the_binding_exports():
    assert declared_functions() == sorted(fb.EXPORTS)


def declared_prototypes() -> dict[str, tuple[str, list[str]]]:
    """name -> (return type, parameter types) of every function in the header."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for ret, name, params in re.findall(r"([A-Za-z_][\w ]*?\**)\s+\**(fm_[a-z_0-9]+)\s*\(([^)]*)\)\s*;", text):
        types = []
        for prm in params.split(","):
            prm = " ".join(prm.split())
            if not prm or prm == "void":
                continue
            # drop the parameter name, keep the type with its stars
            types.append(re.sub(r"\s*\b\w+$", "", prm).replace("const ", "").strip())
        out[name] = (ret.replace("const ", "").strip(), types)
    return out


def _ctype_for(t: str):
    """The ctypes type the binding must use for a C parameter type."""
    if t.endswith("*") or t == "fm_stream_t":
        return "pointer"
    return {"int": C.c_int, "int64_t": C.c_int64, "double": C.c_double, "fm_status": C.c_int,
            "fm_mel_scale": C.c_int, "fm_norm": C.c_int, "fm_dtype": C.c_int}[t]


def test_binding_signatures_match_the_header(L):
    protos = declared_prototypes()
    assert sorted(protos) == declared_functions()
    for name, (ret, params) in protos.items():
        fn = getattr(L, name)
        assert len(fn.argtypes) == len(params), name
        for i, (t, a) in enumerate(zip(params, fn.argtypes)):
            want = _ctype_for(t)
            if want == "pointer":
                assert a is C.c_void_p or a is C.c_char_p or issubclass(a, C._Pointer), (name, i, t, a)
            else:
                assert a is want, (name, i, t, a)
        if ret.endswith("*"):
            assert fn.restype in (C.c_char_p, C.c_void_p), name
        else:
            assert fn.restype is _ctype_for(ret), (name, ret, fn.restype)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings(L):
    assert fb.status_string(fb.FM_OK) == "FM_OK"
    assert fb.status_string(fb.FM_ERR_KERNEL_TIMEOUT) == "FM_ERR_KERNEL_TIMEOUT"
    assert fb.status_string(99) == "FM_ERR_UNKNOWN"


CSR_CASES = [
    (16000, 400, 80, 0.0, 8000.0, "htk", None),
    (16000, 400, 128, 0.0, 8000.0, "htk", None),
    (16000, 1024, 80, 0.0, 8000.0, "htk", None),
    (22050, 2048, 128, 0.0, 11025.0, "slaney", "slaney"),
    (16000, 512, 40, 125.0, 7600.0, "slaney", None),
    (44100, 256, 256, 30.0, 0.0, "htk", "slaney"),
    (8000, 64, 1, 0.0, 4000.0, "htk", None),
]


@pytest.mark.parametrize("case", CSR_CASES)
def test_host_filterbank_matches_oracle(L, case):
    sr, n_fft, n_mels, f_min, f_max, scale, norm = case
    start, ln, off, w = fb.fm_mel_filterbank_csr(sr, n_fft, n_mels, f_min, f_max, scale, norm)
    F = o.mel_filterbank(n_fft, sr, n_mels, f_min, f_max if f_max > 0 else sr / 2, scale, norm)
    dense = np.zeros_like(F)
    assert off[0] == 0 and off[-1] == len(w)
    for m in range(n_mels):
        assert off[m + 1] - off[m] == ln[m]
        dense[m, start[m] : start[m] + ln[m]] = w[off[m] : off[m + 1]]
    tol = 1e-6 * F.max()
    assert np.abs(dense - F).max() <= tol
    # support: every oracle weight above rounding level is inside the stored run
    big = F > 1e-9 * F.max()
    assert np.all(dense[big] > 0)


def test_empty_filters_have_zero_length(L):
    # HTK, 128 mels over 201 bins at 40 Hz spacing: the lowest filters are
    # narrower than a bin and some contain none.
    start, ln, off, w = fb.fm_mel_filterbank_csr(16000, 400, 128, 0.0, 8000.0, "htk", None)
    F = o.mel_filterbank(400, 16000, 128, 0.0, 8000.0, "htk", None)
    empty = np.nonzero(F.max(axis=1) == 0)[0]
    assert empty.size > 0
    assert np.all(ln[empty] == 0)


@pytest.mark.parametrize(
    "kw",
    [
        dict(sr=0), dict(n_fft=0), dict(hop=0), dict(n_mels=0), dict(win_length=500), dict(f_min=-1.0),
        dict(f_max=9000.0), dict(f_min=5000.0, f_max=4000.0), dict(power=0.0), dict(power=float("nan")),
        dict(out_dtype=1), dict(in_dtype=7), dict(mel_scale=5), dict(norm=3),
    ],
)
def test_plan_create_rejects_invalid(L, kw):
    args = dict(sr=16000, n_fft=400, hop=160, win_length=400, n_mels=80, f_min=0.0, f_max=8000.0, power=2.0,
                mel_scale=0, norm=0, in_dtype=0, out_dtype=0)
    args.update(kw)
    h = C.c_void_p(1234)
    st = L.fm_plan_create(C.byref(h), *args.values())
    assert st == fb.FM_ERR_INVALID_ARG
    assert h.value is None


@pytest.mark.parametrize("kw", [dict(n_fft=300), dict(n_fft=32768), dict(n_fft=32), dict(n_mels=257)])
def test_plan_create_reports_unsupported(L, kw):
    args = dict(sr=16000, n_fft=400, hop=160, win_length=0, n_mels=80, f_min=0.0, f_max=0.0, power=2.0,
                mel_scale=0, norm=0, in_dtype=0, out_dtype=0)
    args.update(kw)
    h = C.c_void_p()
    assert L.fm_plan_create(C.byref(h), *args.values()) == fb.FM_ERR_UNSUPPORTED


def _params(**kw):
    p = dict(sr=16000, n_fft=400, hop=160, win_length=400, n_mels=80, f_min=0.0, f_max=8000.0, power=2.0,
             mel_scale=0, norm=0, in_dtype=0, out_dtype=0, center=1, pad_mode=0, pad=0, normalized=0)
    p.update(kw)
    return fb.fm_plan_params(*p.values())


@pytest.mark.parametrize("kw", [dict(pad_mode=4), dict(pad_mode=-1), dict(pad=-1), dict(pad=(1 << 20) + 1),
                                dict(normalized=3), dict(normalized=-1), dict(n_fft=0), dict(power=-1.0)])
def test_plan_create_ex_rejects_invalid(L, kw):
    h = C.c_void_p(1234)
    p = _params(**kw)
    assert L.fm_plan_create_ex(C.byref(h), C.byref(p)) == fb.FM_ERR_INVALID_ARG
    assert h.value is None
    assert L.fm_plan_create_ex(C.byref(h), None) == fb.FM_ERR_INVALID_ARG
    assert L.fm_plan_create_ex(None, C.byref(p)) == fb.FM_ERR_INVALID_ARG


def test_plan_params_layout_matches_header():
    # int x5, double x3, int x8 with natural alignment
    assert C.sizeof(fb.fm_plan_params) == 5 * 4 + 4 + 3 * 8 + 8 * 4
    assert fb.fm_plan_params.f_min.offset == 24 and fb.fm_plan_params.mel_scale.offset == 48


def _c_layout(struct: str, fields: list[str], tmp_path) -> dict:
    """sizeof and offsetof of a struct from include/fm_mel.h, as the C compiler
    lays it out (a small program compiled with the host's cc)."""
    import shutil
    import subprocess

    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "fm_mel.h"', 'int main(void) {',
             f'  printf("size %zu\\n", sizeof({struct}));']
    lines += [f'  printf("{f} %zu\\n", offsetof({struct}, {f}));' for f in fields]
    lines += ['  return 0;', '}']
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-I", os.path.join(root, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    return {k: int(v) for k, v in (ln.split() for ln in out.splitlines())}


def test_binding_constants_match_the_header(tmp_path):
    """Every FM_* constant the binding defines has the header's value (the C
    compiler evaluates the header's enums and macros)."""
    import shutil
    import subprocess

    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    names = [n for n in dir(fb) if n.startswith("FM_") and isinstance(getattr(fb, n), int)]
    assert len(names) >= 20
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    body = "\n".join(f'  printf("{n} %lld\\n", (long long)({n}));' for n in names)
    src = tmp_path / "consts.c"
    src.write_text('#include <stdio.h>\n#include "fm_mel.h"\nint main(void) {\n' + body + "\n  return 0;\n}\n")
    exe = tmp_path / "consts"
    subprocess.run([cc, "-std=c99", "-I", os.path.join(root, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = {k: int(v) for k, v in (ln.split() for ln in out.splitlines())}
    for n in names:
        assert got[n] == getattr(fb, n), n


@pytest.mark.parametrize("name", ["fm_plan_params", "fm_plan_info"])
def test_binding_structs_match_the_c_layout(name, tmp_path):
    cls = getattr(fb, name)
    fields = [f for f, _ in cls._fields_]
    got = _c_layout(name, fields, tmp_path)
    assert got["size"] == C.sizeof(cls)
    for f in fields:
        assert got[f] == getattr(cls, f).offset, f


def test_null_arguments(L):
    assert L.fm_plan_create(None, 16000, 400, 160, 400, 80, 0.0, 0.0, 2.0, 0, 0, 0, 0) == fb.FM_ERR_INVALID_ARG
    assert L.fm_mel_forward(None, None, 1, 1000, None, None) == fb.FM_ERR_INVALID_ARG
    assert L.fm_plan_destroy(None) == fb.FM_OK
    assert L.fm_n_frames(None, 100) == -1
    assert L.fm_plan_get_info(None, None) == fb.FM_ERR_INVALID_ARG
    assert L.fm_plan_poll_error(None) == fb.FM_ERR_INVALID_ARG
    # the host-buffer entry points and the diagnostic refuse a missing plan
    # before any CUDA call
    assert L.fm_mel_forward_host(None, None, 1, 1000, None, None, None, None) == fb.FM_ERR_INVALID_ARG
    assert L.fm_mel_forward_host_noalloc(None, None, 1, 1000, None, None) == fb.FM_ERR_INVALID_ARG
    done, us = C.c_int(-1), C.c_double(-1.0)
    for kind in (0, 1, 2):
        assert L.fm_selftest_wait_timeout(None, kind, 4, None, C.byref(done), C.byref(us)) == fb.FM_ERR_INVALID_ARG
    assert done.value == -1 and us.value == -1.0  # nothing written on refusal
    nnz = C.c_int64(0)
    assert L.fm_mel_filterbank_csr(16000, 400, 80, 0.0, 0.0, 0, 0, None, None, None, None, None) == \
        fb.FM_ERR_INVALID_ARG
    # too small a weights buffer is refused
    buf = (C.c_float * 3)()
    nnz = C.c_int64(3)
    assert L.fm_mel_filterbank_csr(16000, 400, 80, 0.0, 0.0, 0, 0, None, None, None, buf, C.byref(nnz)) == \
        fb.FM_ERR_INVALID_ARG
    assert nnz.value > 3
