"""Compile the CUDA library (libuly.so) in-tree for sm_103a with nvcc.

Three translation units are compiled in parallel and linked into
``_build/libuly.so``; the CUDA runtime is linked statically so the library
loads without a runtime search path.  Rebuilds only when a source is newer
than the library.  ``checked=True`` builds ``_build/libuly_checked.so`` with
-DULY_CHECKED=1 instead: the same kernels with index checks (include/uly.h,
uly_checked_violations)."""
from __future__ import annotations

import glob
import os
import subprocess
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libuly.so")
LIB_CHECKED = os.path.join(OUT, "libuly_checked.so")
UNITS = ("layout.cu", "attn.cu", "uly_abi.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")]
_lock = threading.Lock()


def _sources():
    return ([os.path.join(CSRC, u) for u in UNITS] + glob.glob(os.path.join(CSRC, "*.cuh"))
            + [os.path.join(ROOT, "include", "uly.h")])


def up_to_date(checked: bool = False) -> bool:
    lib = LIB_CHECKED if checked else LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(s) <= t for s in _sources())


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    lib = LIB_CHECKED if checked else LIB
    with _lock:
        if not force and up_to_date(checked):
            return lib
        os.makedirs(OUT, exist_ok=True)
        nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
        if not os.path.exists(nvcc):
            nvcc = "nvcc"
        procs = []
        objs = []
        for u in UNITS:
            obj = os.path.join(OUT, u.replace(".cu", "_checked.o" if checked else ".o"))
            objs.append(obj)
            cmd = [nvcc] + ARCH + FLAGS + (["-DULY_CHECKED=1"] if checked else []) + \
                (["-Xptxas", "-v"] if verbose else []) + ["-c", os.path.join(CSRC, u), "-o", obj]
            procs.append((u, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        logs = []
        failed = []
        for u, p in procs:
            out, _ = p.communicate()
            logs.append(out.decode(errors="replace"))
            if p.returncode:
                failed.append(u)
        if failed:
            raise RuntimeError("nvcc failed for %s:\n%s" % (failed, "\n".join(logs)))
        tmp = lib + ".%d.tmp" % os.getpid()
        subprocess.check_call([nvcc] + ARCH + ["-shared", "-o", tmp] + objs)
        os.replace(tmp, lib)
        if verbose:
            print("\n".join(logs))
        return lib
