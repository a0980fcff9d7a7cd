"""Build libloom.so in-tree with nvcc for sm_103a.

Each CUDA translation unit under csrc/ is compiled in parallel into
_build/, then linked into int8_dequant_dot_gb300/libloom.so.  The same
objects, with the host layer (loom_api.cu) compiled again with
LOOM_TEST_HOOKS, also link into libloom_test.so, the build the fault tests
load (it adds loom_test_inject_stall, csrc/test_hooks.h).  Usage:

    python int8_dequant_dot_gb300/build.py        (or __graft_entry__.build())

It is loaded by file path rather than as a package submodule, because
importing the package requires the library this script produces.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libloom.so")
TEST_LIB = os.path.join(HERE, "libloom_test.so")
SOURCES = ["loom_api.cu", "row_sum.cu", "dequant_dot.cu", "dot_tc.cu", "dot_tc_rows.cu", "packed_dot.cu", "lane_sum.cu", "routed.cu", "stage.cu", "stream_floor.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: set NVCC or put the CUDA toolkit on PATH")


def _deps() -> list[str]:
    out = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    out += [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))]
    return out


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile (if stale) and link libloom.so and libloom_test.so; returns the path of
    libloom.so."""
    deps = _deps()
    if not force and not _stale(LIB, deps) and not _stale(TEST_LIB, deps):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                    "-I", os.path.join(ROOT, "include"), "--ftz=false", "--prec-div=true",
                    "--prec-sqrt=true", "--fmad=true"]
    if ptxas_info:
        flags += ["-Xptxas", "-v"]

    def compile_one(job: tuple[str, str, list[str]]) -> tuple[str, str]:
        src, obj_name, extra = job
        obj = os.path.join(BUILD, obj_name)
        cmd = [cc] + flags + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    jobs = [(src, src.replace(".cu", ".o"), []) for src in SOURCES]
    jobs.append(("loom_api.cu", "loom_api_test.o", ["-DLOOM_TEST_HOOKS"]))
    with ThreadPoolExecutor(len(jobs)) as ex:
        results = list(ex.map(compile_one, jobs))
    if verbose or ptxas_info:
        for _, log in results[:len(SOURCES)]:
            if log.strip():
                print(log, file=sys.stderr)
    objs = [o for o, _ in results[:len(SOURCES)]]
    test_objs = [results[-1][0] if os.path.basename(o) == "loom_api.o" else o for o in objs]
    for target, members in ((LIB, objs), (TEST_LIB, test_objs)):
        tmp = target + ".tmp%d" % os.getpid()
        cmd = [cc] + ARCH + ["-shared", "-o", tmp] + members
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, target)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="-v" in sys.argv))
