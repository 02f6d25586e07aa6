"""Build libmfd.so (sm_103a) in-tree with nvcc: one object per .cu file,
compiled in parallel, linked with -shared.  libmfd_checked.so is the same
library with the tree builder compiled with -DMFD_CHECKED, the bounds-checked
build (an index out of range is clamped and reported as MFD_ERR_CHECK instead
of being used).
Run: python -m tree_verified_speculative_gb300.build"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libmfd.so")
LIB_CHECKED = os.path.join(BUILD, "libmfd_checked.so")
SOURCES = ["lmhead.cu", "topk.cu", "tree.cu", "verify.cu", "analytics.cu", "mfd_api.cu"]
CHECKED_SOURCES = ["tree.cu"]  # the sources with bounds checks under -DMFD_CHECKED
HEADERS = ["lmhead.h", "mfd_device.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _newest_input() -> float:
    paths = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    paths.append(os.path.join(HERE, "..", "include", "mfd.h"))
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def _compile(job: tuple[str, bool]) -> tuple[str, str]:
    src, checked = job
    obj = os.path.join(BUILD, src.replace(".cu", "_checked.o" if checked else ".o"))
    cmd = [nvcc(), *ARCH, *FLAGS, *(["-DMFD_CHECKED"] if checked else []), "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def _link(objs: list[str], out: str) -> None:
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)


def build(force: bool = False, verbose: bool = False) -> str:
    """Both libraries; returns the path of libmfd.so."""
    os.makedirs(BUILD, exist_ok=True)
    newest = _newest_input()
    if (not force and all(os.path.exists(p) and os.path.getmtime(p) >= newest for p in (LIB, LIB_CHECKED))):
        return LIB
    # the checks live in tree.cu; the checked library shares every other object
    jobs = [(s, False) for s in SOURCES] + [(s, True) for s in CHECKED_SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(_compile, jobs))
    log = "\n".join(err for _, err in results[:len(SOURCES)])
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        f.write(log)
    if verbose:
        print(log)
    plain = [o for o, _ in results[:len(SOURCES)]]
    checked = {src: o for (src, _), (o, _) in zip(jobs[len(SOURCES):], results[len(SOURCES):])}
    _link(plain, LIB)
    _link([checked.get(src, o) for src, o in zip(SOURCES, plain)], LIB_CHECKED)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
