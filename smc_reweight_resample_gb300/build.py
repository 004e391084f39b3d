"""Build the CUDA library ``libsmcsd.so`` in-tree for sm_103a (GB300).

Each translation unit is compiled in its own nvcc process, in parallel, then linked into one
shared library with the CUDA runtime linked statically. Objects go to ``_build/`` beside this
file; the library is written next to this file. Run ``python -m smc_reweight_resample_gb300.build``
or call ``build()``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsmcsd.so")
SOURCES = ["api.cu", "verify_stream.cu", "stream_tma.cu", "finish.cu", "sd_sample.cu", "resample_pacer.cu",
           "static_scratch.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def _flags():
    return ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC",
            "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "smcsd.h")]
    return any(os.path.getmtime(d) > t for d in deps)


# The library with the opt-in device self-checks (-DSMCSD_CHECKS): every check site records its
# code and the offending value in the workspace instead of making the access. Built on request
# (build_checks) into its own folder, for the tests that run the parity cases against it.
CHECKS_BUILD = os.path.join(HERE, "_build_checks")
CHECKS_LIB = os.path.join(CHECKS_BUILD, "libsmcsd_checks.so")


def build_checks(force: bool = False, verbose: bool = False) -> str:
    return build(force, verbose, extra_flags=("-DSMCSD_CHECKS",), out=CHECKS_LIB,
                 objdir=CHECKS_BUILD)


def build(force: bool = False, verbose: bool = False, extra_flags=(), out: str = LIB,
          objdir: str = BUILD) -> str:
    if not force and not _stale(out):
        return out
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [cc, *_flags(), *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, pr in procs:
        log, _ = pr.communicate()
        if verbose or pr.returncode != 0:
            sys.stdout.write(log.decode(errors="replace"))
        if pr.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call([cc, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
