"""Build libpa.so (the C-ABI library) and libpa_probe.so (its measurement and
test aids) from csrc/ with nvcc for sm_103a.

Each translation unit compiles in parallel; the objects link into shared
libraries with the CUDA runtime linked statically, so they load with ctypes
and need nothing but the driver. Outputs stay in-tree:
``paged_kv_cache_176_gb300/_build/`` and ``paged_kv_cache_176_gb300/lib*.so``.

A build is reused only when a stamp written beside the objects matches the
sources, the flags and the host machine's architecture; anything else (a
changed source, a copy of the tree on another machine) rebuilds.
"""
from __future__ import annotations

import concurrent.futures as fut
import glob
import hashlib
import json
import os
import platform
import shutil
import subprocess
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpa.so")
PROBE_LIB = os.path.join(HERE, "libpa_probe.so")
STAMP = os.path.join(BUILD, "stamp")
RECORD = os.path.join(BUILD, "record.json")  # what the last compilation built, where and when
ROOT = os.path.dirname(HERE)
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _sources() -> tuple[list[str], list[str]]:
    lib = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    probe = sorted(glob.glob(os.path.join(CSRC, "probe", "*.cu")))
    return lib, probe


def _stamp(extra_flags) -> str:
    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(CSRC, "**", "*"), recursive=True)
                   + glob.glob(os.path.join(ROOT, "include", "*.h")) + [os.path.abspath(__file__)])
    for f in files:
        if os.path.isfile(f):
            h.update(os.path.relpath(f, ROOT).encode())
            with open(f, "rb") as fh:
                h.update(fh.read())
    h.update(" ".join([*ARCH, *NVCC_FLAGS, *extra_flags, platform.machine()]).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    stamp = _stamp(extra_flags)
    if (not force and os.path.exists(LIB) and os.path.exists(PROBE_LIB) and os.path.exists(STAMP)
            and open(STAMP).read().strip() == stamp):
        sys.stderr.write(f"libpa: reusing the build of these sources on {platform.machine()} "
                         f"(stamp {stamp[:16]})\n")
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    lib_srcs, probe_srcs = _sources()
    exe = nvcc()

    def compile_one(src: str) -> str:
        sub = "probe_" if os.path.basename(os.path.dirname(src)) == "probe" else ""
        obj = os.path.join(BUILD, sub + os.path.splitext(os.path.basename(src))[0] + ".o")
        cmd = [exe, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    srcs = lib_srcs + probe_srcs
    with fut.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    for out, o in ((LIB, objs[:len(lib_srcs)]), (PROBE_LIB, objs[len(lib_srcs):])):
        tmp = out + ".tmp"
        cmd = [exe, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *o]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, out)
    with open(STAMP, "w") as f:
        f.write(stamp + "\n")
    with open(RECORD, "w") as f:
        json.dump({"stamp": stamp[:16], "machine": platform.machine(), "units": len(srcs),
                   "compiled_unix_s": round(time.time(), 1)}, f)
    sys.stderr.write(f"libpa: compiled {len(srcs)} translation units for sm_103a "
                     f"on {platform.machine()}\n")
    return LIB


def build_record() -> dict:
    """Whether libpa.so was built from these sources on this machine, and when
    it was compiled (for run records: a library carried over from another
    machine or older sources shows here)."""
    cur = _stamp(())
    rec = {"stamp": cur[:16], "machine": platform.machine(), "matches_sources": False}
    if os.path.exists(STAMP):
        rec["matches_sources"] = open(STAMP).read().strip() == cur
    if os.path.exists(RECORD):
        with open(RECORD) as f:
            rec["last_compile"] = json.load(f)
    return rec


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []
    print(build(force=True, verbose=v or bool(extra), extra_flags=extra))
