"""Builds libfa_gb300.so from csrc/ with nvcc for sm_103a (in-tree).

Each translation unit is compiled in parallel into ``_build/`` and the objects
are linked into ``libfa_gb300.so`` next to this file.  Objects are rebuilt
when their source or any header is newer.
"""
from __future__ import annotations

import os
import platform
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OBJDIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libfa_gb300.so")
SOURCES = ["prefill_d512.cu", "prefill_d128.cu", "prefill_d256.cu", "prefill_d96.cu",
           "prefill_d64.cu", "decode.cu", "selftest.cu", "api.cu", "decode_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
                "-I", CSRC, "-I", INCLUDE]


def _options():
    """Build options from the environment: FA_PREFILL_TRACE=1 compiles the
    prefill kernel's debug clock trace (off by default: it costs registers)."""
    return ["-DFA_PREFILL_TRACE=1"] if os.environ.get("FA_PREFILL_TRACE") == "1" else []


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    hs.append(os.path.join(INCLUDE, "fa.h"))
    return hs


def build(force: bool = False, jobs: int | None = None, verbose: bool = False) -> str:
    os.makedirs(OBJDIR, exist_ok=True)
    # objects from another host architecture (or toolchain) are never reused
    stamp = os.path.join(OBJDIR, "host.txt")
    host = f"{platform.machine()} {platform.system()} {' '.join(_options())}"
    if not os.path.exists(stamp) or open(stamp).read() != host:
        force = True
    nvcc = _nvcc()
    newest_header = max(os.path.getmtime(h) for h in _headers())

    def compile_one(src):
        s = os.path.join(CSRC, src)
        o = os.path.join(OBJDIR, src.replace(".cu", ".o"))
        if (not force and os.path.exists(o)
                and os.path.getmtime(o) >= max(os.path.getmtime(s), newest_header)):
            return o, False
        cmd = [nvcc] + FLAGS + _options() + ["-c", s, "-o", o + ".tmp"]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        os.replace(o + ".tmp", o)
        return o, True

    jobs = jobs or min(len(SOURCES), os.cpu_count() or 4)
    with ThreadPoolExecutor(max_workers=jobs) as ex:
        results = list(ex.map(compile_one, SOURCES))
    objs = [o for o, _ in results]
    relink = (force or any(changed for _, changed in results) or not os.path.exists(LIB_PATH)
              or os.path.getmtime(LIB_PATH) < max(os.path.getmtime(o) for o in objs))
    if relink:
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs + [
            "-Xlinker", "-rpath," + os.path.join(os.path.dirname(os.path.dirname(
                os.path.realpath(nvcc) if os.path.sep in nvcc else "/usr/local/cuda/bin/nvcc")),
                "lib64")]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB_PATH)
    with open(stamp, "w") as f:
        f.write(host)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
