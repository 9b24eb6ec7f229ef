"""Builds the sm_103a shared library in-tree with nvcc (no torch extension).

    python -m causal_gqa_prefill_gb300.build [--force] [--debug]

Output: ``causal_gqa_prefill_gb300/lib/libattn_prefill.so`` plus the ptxas
resource report ``lib/ptxas.log`` (registers, spills, shared memory). With
``debug=True``: ``lib/libattn_prefill_debug.so``, the same sources compiled
with ATTN_DEBUG, whose forward kernels check their TMA coordinates, tensor
memory and shared-memory addresses and mbarrier phases as they run
(``lib/ptxas_debug.log``). ``build_all()`` compiles both in parallel.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "lib")
LIBNAME = "libattn_prefill.so"
DEBUG_LIBNAME = "libattn_prefill_debug.so"
SOURCES = ["attn_prefill.cu", "attn_decode.cu", "attn_backward.cu", "attn_host.cu"]
HEADERS = [os.path.join(CSRC, "sm103_ptx.cuh"), os.path.join(INCLUDE, "attn_prefill.h")]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def library_path(debug: bool = False) -> str:
    return os.path.join(LIBDIR, DEBUG_LIBNAME if debug else LIBNAME)


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _elf_machine(path: str) -> int:
    with open(path, "rb") as f:
        head = f.read(20)
    if len(head) < 20 or head[:4] != b"\x7fELF":
        return -1
    return int.from_bytes(head[18:20], "little")


def _host_machine() -> int:
    return _elf_machine(sys.executable if os.path.exists(sys.executable) else "/bin/sh")


def _stale(out: str) -> bool:
    if not os.path.exists(out):
        return True
    if _elf_machine(out) != _host_machine():    # built on another architecture
        return True
    t = os.path.getmtime(out)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile the library (the ATTN_DEBUG one with ``debug``) if it is missing
    or older than its sources; return its path."""
    out = library_path(debug)
    if not force and not _stale(out):
        return out
    os.makedirs(LIBDIR, exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    cmd = [_nvcc(), "-shared", "-Xcompiler", "-fPIC", "-O3", "-std=c++17", "-lineinfo", ARCH,
           "-Xptxas", "-v", "-I" + INCLUDE, "-I" + CSRC]
    if debug:
        cmd.append("-DATTN_DEBUG")
    cmd += [os.path.join(CSRC, s) for s in SOURCES]
    cmd += ["-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(LIBDIR, "ptxas_debug.log" if debug else "ptxas.log"), "w") as f:
        f.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        if os.path.exists(tmp):
            os.remove(tmp)
        raise RuntimeError("nvcc failed:\n" + res.stderr[-4000:])
    os.replace(tmp, out)
    if verbose:
        print(res.stderr)
    return out


def build_all(force: bool = False) -> tuple:
    """Both libraries, compiled in parallel; returns (release path, debug path)."""
    from concurrent.futures import ThreadPoolExecutor

    with ThreadPoolExecutor(max_workers=2) as ex:
        rel = ex.submit(build, force, False, False)
        dbg = ex.submit(build, force, False, True)
        return rel.result(), dbg.result()


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))
