"""Ahead-of-time build of libfm_mel.so for sm_103a with nvcc.

Each translation unit compiles in its own nvcc process (in parallel), then
the objects are linked into ``mel_spectrogram_gb300/libfm_mel.so`` beside this
file. Rebuilds only what changed (source or header newer than the object).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfm_mel.so")
# the debug build (every guarded access index-checked, see FM_IN in fm_internal.h)
BUILD_CHECK = os.path.join(PKG, "_build_check")
LIB_CHECK = os.path.join(PKG, "libfm_mel_check.so")
CHECK_FLAGS = ["-DFM_BOUNDS_CHECK"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC,-O2",
          f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfm_mel.so")


def _sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _headers() -> list[str]:
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(INCLUDE, "*.h"))


def _obj(src: str, build_dir: str = BUILD) -> str:
    return os.path.join(build_dir, os.path.basename(src) + ".o")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, extra: list[str], build_dir: str = BUILD) -> str:
    out = _obj(src, build_dir)
    cmd = [nvcc(), *ARCH, *COMMON, *extra, "-c", src, "-o", out]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stderr


def build(verbose: bool = False, extra: list[str] | None = None, jobs: int | None = None,
          check: bool = False) -> str:
    """Compile and link libfm_mel.so (check=True: the index-checked debug
    build libfm_mel_check.so, in its own object directory); returns its path."""
    return build_many([check], verbose, extra, jobs)[0]


def build_many(checks: list[bool], verbose: bool = False, extra: list[str] | None = None,
               jobs: int | None = None) -> list[str]:
    """Build several of the libraries (release / debug) in one pool of nvcc
    processes; returns their paths in order."""
    extra = list(extra or [])
    hdrs = _headers()
    targets = [(BUILD_CHECK, LIB_CHECK, extra + CHECK_FLAGS) if c else (BUILD, LIB, extra) for c in checks]
    todo = []
    for bdir, _, flags in targets:
        os.makedirs(bdir, exist_ok=True)
        todo += [(s, flags, bdir) for s in _sources() if extra or _stale(_obj(s, bdir), [s, *hdrs, __file__])]
    if todo:
        n = jobs or min(len(todo), max(1, os.cpu_count() or 1))
        with cf.ThreadPoolExecutor(n) as ex:
            for (src, _, _), log in zip(todo, ex.map(lambda t: _compile(*t), todo)):
                if verbose and log.strip():
                    print(f"[{os.path.basename(src)}]\n{log}", file=sys.stderr)
    for bdir, lib, _ in targets:
        objs = [_obj(s, bdir) for s in _sources()]
        if any(t[2] == bdir for t in todo) or _stale(lib, objs):
            tmp = lib + ".tmp"
            cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
            os.replace(tmp, lib)
    return [lib for _, lib, _ in targets]


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []
    print(build(verbose=v or bool(extra), extra=extra, check="--check" in sys.argv))
