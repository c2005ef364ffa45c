"""Build libpagedkv.so (CUDA for sm_103a) in-tree with nvcc.

Each source (.cu kernels and C ABI, .cpp host code) compiles to an object in parallel, then one link step makes the
shared library next to this file.  No torch extension machinery: the library
exports a plain C ABI (include/pagedkv.h).
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libpagedkv.so")
SOURCES = ["api.cu", "kv_write.cu", "decode.cu", "decode_noalloc.cu", "kv_copy.cu", "prefill.cu",
           "prefill_fp8.cu", "prefill_fp4.cu",
           "block_manager.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps() -> list[str]:
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    inc = os.path.join(os.path.dirname(HERE), "include")
    hdrs += [os.path.join(inc, f) for f in os.listdir(inc) if f.endswith(".h")]
    return hdrs


def stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    files = [os.path.join(CSRC, s) for s in SOURCES] + _deps()
    return any(os.path.getmtime(f) > t for f in files)


def start_objects(verbose: bool = False) -> list[tuple[str, subprocess.Popen]]:
    os.makedirs(BUILD_DIR, exist_ok=True)
    procs = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc(), *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((obj, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    return procs


def finish(procs, verbose: bool = False) -> str:
    logs = []
    objs = []
    for obj, proc in procs:
        out, _ = proc.communicate()
        text = out.decode(errors="replace")
        logs.append(text)
        if proc.returncode != 0:
            raise RuntimeError(f"nvcc failed for {obj}:\n{text}")
        objs.append(obj)
    tmp = LIB_PATH + ".tmp"
    link = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if res.returncode != 0:
        raise RuntimeError("link failed:\n" + res.stdout.decode(errors="replace"))
    os.replace(tmp, LIB_PATH)
    log = "\n".join(logs)
    with open(os.path.join(BUILD_DIR, "ptxas.log"), "w") as f:
        f.write(log)
    if verbose:
        print(log)
    return log


def build(verbose: bool = False) -> str:
    return finish(start_objects(verbose), verbose)


if __name__ == "__main__":
    build(verbose="-v" in sys.argv)
    print(LIB_PATH)
