"""Build the in-tree CUDA library ``libqgemm.so`` for sm_103a with nvcc.

Run ``python -m quantized_weight_gemm_run_b300.build`` (or call ``build()``).
Objects go to ``_build/`` beside the package; the shared library is written
next to this file so that it travels with the source tree.  Rebuilds only
what changed (source or header newer than the object).  ``--checked`` (or
``build(checked=True)``) builds ``libqgemm_checked.so`` instead: the same
sources with ``-DQGEMM_CHECKED`` (index tests in every kernel), objects in
``_build/checked/``.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libqgemm.so")
LIB_CHECKED = os.path.join(PKG, "libqgemm_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hs.append(os.path.join(ROOT, "include", "qgemm.h"))
    return hs


def _compile(nvcc, src, obj, verbose_ptxas, checked=False):
    cmd = [nvcc, *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
           "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-c", src, "-o", obj]
    if checked:
        cmd.insert(1, "-DQGEMM_CHECKED")
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{res.stderr}")
    return res.stderr


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int = 8,
          checked: bool = False) -> str:
    nvcc = nvcc_path()
    bdir = os.path.join(BUILD, "checked") if checked else BUILD
    lib = LIB_CHECKED if checked else LIB
    os.makedirs(bdir, exist_ok=True)
    hdr_time = max(os.path.getmtime(h) for h in headers())
    todo = []
    objs = []
    for src in sources():
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or not os.path.exists(obj) or os.path.getmtime(obj) < max(
                os.path.getmtime(src), hdr_time):
            todo.append((src, obj))
    logs = []
    if todo:
        with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
            futs = [ex.submit(_compile, nvcc, s, o, verbose_ptxas, checked) for s, o in todo]
            for f in futs:
                logs.append(f.result())
    if todo or force or not os.path.exists(lib):
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", lib, *objs,
               "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stderr}")
    if verbose_ptxas:
        for log in logs:
            sys.stderr.write(log)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv,
                checked="--checked" in sys.argv))
