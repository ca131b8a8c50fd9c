"""Builds the CUDA library ``_lib/libmt_rowreduce.so`` in-tree with nvcc.

Targets sm_103a only (``-gencode arch=compute_103a,code=sm_103a``).  The
translation units compile in parallel; a stamp over the sources and flags
skips the build when nothing changed.  ``ptxas -v`` resource lines (registers,
spills, shared memory per kernel) are kept in ``_lib/ptxas.txt``.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT, "libmt_rowreduce.so")
HEADER = os.path.join(ROOT, "include", "mt_rowreduce.h")

OPS = ("rmsnorm", "layernorm", "residual_layernorm", "softmax", "row_sum",
       "cross_entropy", "residual_rmsnorm", "log_softmax")
DTYPES = ("f32", "f16", "bf16")
SOURCES = (["api.cpp", "planner.cpp", "mean.cu", "probe.cu"] +
           [f"ops_{op}_{dt}.cu" for op in OPS for dt in DTYPES])
DEPENDS = ["mt_internal.h", "mt_kernels.cuh", "mt_stage.cuh", "plan_table.inc"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler",
          "-fPIC,-fvisibility=hidden", "-Xptxas", "-v"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"),
                 "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put it on PATH)")


def _stamp(nvcc: str) -> str:
    h = hashlib.sha256()
    for name in SOURCES + DEPENDS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    with open(HEADER, "rb") as f:
        h.update(f.read())
    h.update(" ".join([nvcc] + ARCH + CFLAGS).encode())
    h.update(os.uname().machine.encode())
    return h.hexdigest()


def _compile(nvcc: str, src: str, obj: str) -> str:
    cmd = [nvcc, "-c", os.path.join(CSRC, src), "-o", obj] + ARCH + CFLAGS
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return r.stderr


def build(force: bool = False, jobs: int | None = None,
          verbose: bool = False) -> str:
    """Compile and link the library if sources changed; returns its path."""
    nvcc = _nvcc()
    os.makedirs(os.path.join(OUT, "obj"), exist_ok=True)
    stamp = _stamp(nvcc)
    stamp_file = os.path.join(OUT, "build.stamp")
    if (not force and os.path.exists(LIB) and os.path.exists(stamp_file)
            and open(stamp_file).read().strip() == stamp):
        return LIB
    objs = [os.path.join(OUT, "obj", s.rsplit(".", 1)[0] + ".o")
            for s in SOURCES]
    for name in os.listdir(os.path.join(OUT, "obj")):   # stale objects
        path = os.path.join(OUT, "obj", name)
        if path not in objs:
            os.remove(path)
    # Largest translation units first so the parallel build ends sooner.
    order = sorted(range(len(SOURCES)),
                   key=lambda i: not SOURCES[i].endswith(".cu"))
    jobs = jobs or min(len(SOURCES), max(1, os.cpu_count() or 1))
    logs = [""] * len(SOURCES)
    with cf.ThreadPoolExecutor(jobs) as ex:
        futs = {ex.submit(_compile, nvcc, SOURCES[i], objs[i]): i
                for i in order}
        for fut in cf.as_completed(futs):
            logs[futs[fut]] = fut.result()
    with open(os.path.join(OUT, "ptxas.txt"), "w") as f:
        for s, log in zip(SOURCES, logs):
            f.write(f"== {s}\n{log}\n")
    vers = os.path.join(OUT, "exports.map")
    with open(vers, "w") as f:
        f.write("{ global: mt_*; local: *; };\n")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", "-o", tmp] + objs + ARCH + [
        "-Xlinker", f"--version-script={vers}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp_file, "w") as f:
        f.write(stamp + "\n")
    if verbose:
        print(f"built {LIB}", file=sys.stderr)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
