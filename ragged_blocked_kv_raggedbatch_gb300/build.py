"""Build ``libds_ragged.so`` (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel; the result lands in
``ragged_blocked_kv_raggedbatch_gb300/_build/``.  Rebuilds only what changed.
Extra nvcc flags (e.g. -D overrides of the decode CTA shape) can be given in
the DSR_NVCC_FLAGS environment variable.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libds_ragged.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libds_ragged.so")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _compile(src: str, verbose_ptxas: bool, out_dir: str = OUT_DIR, extra_flags: str = "") -> str:
    obj = os.path.join(out_dir, os.path.basename(src) + ".o")
    newest_dep = max([os.path.getmtime(src)] + [os.path.getmtime(h) for h in _headers()])
    stamp = obj + ".flags"
    extra = (os.environ.get("DSR_NVCC_FLAGS", "") + " " + extra_flags).strip()
    same_flags = os.path.exists(stamp) and open(stamp).read() == extra
    if os.path.exists(obj) and os.path.getmtime(obj) >= newest_dep and same_flags:
        return obj
    flags = list(NVCC_FLAGS) + extra.split()
    if verbose_ptxas and src.endswith(".cu"):
        flags += ["-Xptxas", "-v"]
    cmd = [_nvcc()] + flags + ["-c", src, "-o", obj + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    os.replace(obj + ".tmp", obj)
    with open(stamp, "w") as f:
        f.write(extra)
    return obj


def build(verbose_ptxas: bool = False, jobs: int = 0, out_dir: str = OUT_DIR, extra_flags: str = "") -> str:
    """Compile and link the library into out_dir (the package's _build/ by
    default); extra_flags are added nvcc flags (e.g. a test build's -D)."""
    os.makedirs(out_dir, exist_ok=True)
    lib = os.path.join(out_dir, os.path.basename(LIB))
    srcs = _sources()
    jobs = jobs or min(len(srcs), max(1, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, out_dir, extra_flags), srcs))
    if os.path.exists(lib) and os.path.getmtime(lib) >= max(os.path.getmtime(o) for o in objs):
        return lib
    tmp = lib + ".tmp.%d" % os.getpid()
    cmd = [_nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv))
