"""Build the CUDA library ``libconvfwd.so`` in-tree for sm_103a.

Each ``csrc/*.cu`` is compiled to an object in parallel with
``nvcc -gencode arch=compute_103a,code=sm_103a -O3 -lineinfo`` and the objects
are linked into one shared library next to this file.  No fast-math: the
tensor-core path's operand split relies on exact fp32 subtraction.

``build(debug=True)`` builds the same sources with ``-DCONVFWD_DEBUG`` into
``libconvfwd_debug.so``: host-side plan assertions and device-side bounds
checks that record into the status word instead of trapping (the binding
loads it when ``CONVFWD_DEBUG=1``).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
SO = os.path.join(HERE, "libconvfwd.so")
SO_DEBUG = os.path.join(HERE, "libconvfwd_debug.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
           "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA library cannot be built")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stamp(extra=()):
    h = hashlib.sha256()
    for f in sorted(_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) +
                    glob.glob(os.path.join(INCLUDE, "*.h"))):
        h.update(f.encode())
        h.update(open(f, "rb").read())
    h.update(" ".join(ARCH + NVFLAGS + list(extra)).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False, debug: bool = False) -> str:
    out_dir = os.path.join(BUILD, "debug") if debug else BUILD
    so = SO_DEBUG if debug else SO
    os.makedirs(out_dir, exist_ok=True)
    stamp_file = os.path.join(out_dir, "stamp")
    extra = ["-Xptxas", "-v"] if ptxas_v else []
    if debug:
        extra = extra + ["-DCONVFWD_DEBUG"]
    stamp = _stamp(extra)
    if not force and os.path.exists(so) and os.path.exists(stamp_file) and open(stamp_file).read() == stamp:
        return so
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc] + ARCH + NVFLAGS + extra + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        if verbose or ptxas_v:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = so + f".tmp{os.getpid()}"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, so)
    open(stamp_file, "w").write(stamp)
    return so


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_v="-v" in sys.argv, debug="--debug" in sys.argv))
