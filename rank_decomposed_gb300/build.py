"""Build liblr.so (the CUDA path) and libsynth.so (the GPU input generator).

Both are compiled in-tree for sm_103a only, with nvcc, one translation unit
per process so a build takes well under a minute.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "liblr.so")
SYNTH_SRC = os.path.join(ROOT, "synth", "synth_gen.cu")
SYNTH_LIB = os.path.join(ROOT, "synth", "libsynth.so")
SYNTH_HOST_SRC = os.path.join(ROOT, "synth", "synth_host.c")
SYNTH_HOST_LIB = os.path.join(ROOT, "synth", "libsynth_host.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found")
    return exe


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed: %s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
    return r.stdout + r.stderr


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    exe = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    jobs = []
    for src in sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        jobs.append(([exe, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj], obj))
    synth_cmd = [exe, *ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                 SYNTH_SRC, "-o", SYNTH_LIB]
    host_cmd = [shutil.which("gcc") or "gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared",
                SYNTH_HOST_SRC, "-o", SYNTH_HOST_LIB]
    logs = []
    with cf.ThreadPoolExecutor(max_workers=min(8, len(jobs) + 1)) as ex:
        futs = [ex.submit(_run, cmd) for cmd, _ in jobs]
        futs.append(ex.submit(_run, synth_cmd))
        futs.append(ex.submit(_run, host_cmd))
        for f in futs:
            logs.append(f.result())
    _run([exe, *ARCH, "-shared", "-o", LIB, *[o for _, o in jobs], "-lcudart_static"])
    out = "\n".join(l for l in logs if l)
    if verbose and out:
        print(out)
    return out


if __name__ == "__main__":
    import sys
    print(build(verbose=True, ptxas_info="-v" in sys.argv) or "built")
