"""Build libfa.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Each translation unit under csrc/ is compiled in parallel, then linked into
io_aware_exact_02_gb300/libfa.so with the CUDA runtime linked statically, so
the library loads on a machine without a GPU (only its entry points need
one).  Run as ``python -m io_aware_exact_02_gb300.build``; ``--checked``
builds the bounds-checked variant libfa_checked.so instead (-DFA_CHECKS),
which the binding loads when FA_CHECKED=1.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libfa.so")
# The bounds-checked build (-DFA_CHECKS): every kernel range-checks the
# tile, mask and row indices it computes and reports FA_ERR_BOUNDS instead of
# using one that is out of range.
LIB_CHECKED = os.path.join(HERE, "libfa_checked.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
UNITS = ["fa_api.cu", "fa_fwd.cu", "fa_fwd_pair.cu", "fa_bwd.cu", "fa_noalloc.cu", "fa_fp8.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler",
         "-fvisibility=default", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa.so")


def sources():
    srcs = [os.path.join(CSRC, u) for u in UNITS]
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    deps.append(os.path.join(INCLUDE, "fa.h"))
    return srcs, deps


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    _, deps = sources()
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in deps)


def build(force: bool = False, verbose: bool = False, checked: bool | None = None) -> str:
    """Build libfa.so, or libfa_checked.so when `checked` (default: when the
    environment sets FA_CHECKED=1, as the binding does to load it)."""
    if checked is None:
        checked = os.environ.get("FA_CHECKED") == "1"
    lib = LIB_CHECKED if checked else LIB
    if not force and up_to_date(lib):
        return lib
    srcs, _ = sources()
    cc = nvcc()
    tmp = tempfile.mkdtemp(prefix="fa_build_")
    try:
        procs = []
        objs = []
        for s in srcs:
            obj = os.path.join(tmp, os.path.basename(s) + ".o")
            cmd = [cc, *ARCH, *FLAGS, *(["-DFA_CHECKS"] if checked else []), "-I", INCLUDE,
                   "-c", s, "-o", obj]
            if verbose:
                cmd += ["-Xptxas", "-v"]
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
            objs.append(obj)
        failed = []
        for cmd, pr in procs:
            out, _ = pr.communicate()
            text = out.decode(errors="replace")
            if pr.returncode != 0:
                failed.append(" ".join(cmd) + "\n" + text)
            elif verbose and text:
                sys.stdout.write(text)
        if failed:
            raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
        out_tmp = lib + ".%d.tmp" % os.getpid()
        subprocess.run([cc, *ARCH, "-shared", "-cudart", "static", *objs, "-o", out_tmp],
                       check=True)
        os.replace(out_tmp, lib)
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                checked=True if "--checked" in sys.argv else None))
