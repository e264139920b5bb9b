"""Build libmx.so in-tree with nvcc for sm_103a (no CMake, no torch extension).

Each translation unit is compiled in parallel, then linked into a shared
library next to this file; the Python binding loads it from there.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmx.so")
# Timeline build: the same sources with -DMX_TIMELINE (per-CTA %globaltimer
# stamps of every GEMM launch, read back with mx_timeline_read); diagnostic only.
TIMELINE_LIB = os.path.join(HERE, "libmx_timeline.so")
TIMELINE_BUILD = os.path.join(HERE, "_build_timeline")
SOURCES = ["api.cu", "quantize.cu", "gemm.cu", "wo_a.cu", "chain.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    deps = [src] + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    deps.append(os.path.join(HERE, "..", "include", "mx.h"))
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def build(verbose: bool = False, force: bool = False, extra: list[str] | None = None,
          lib: str = LIB, build_dir: str = BUILD) -> str:
    """Compile the sources (in parallel) and link `lib`; objects go to build_dir.
    `extra` adds nvcc flags (e.g. -DMX_TIMELINE for the timeline build, which
    needs its own lib and build_dir)."""
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, s):
            cmd = [cc, *ARCH, *FLAGS, *(extra or []), "-c", s, "-o", o]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    errors = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            errors.append(f"--- {src}\n{text}")
        elif verbose and text.strip():
            print(text, file=sys.stderr)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    if force or procs or not os.path.exists(lib):
        tmp = lib + ".tmp"
        cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
        os.replace(tmp, lib)
    return lib


def build_timeline(verbose: bool = False) -> str:
    return build(verbose=verbose, extra=["-DMX_TIMELINE"], lib=TIMELINE_LIB, build_dir=TIMELINE_BUILD)


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
