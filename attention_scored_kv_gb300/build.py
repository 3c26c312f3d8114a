"""Build libkvs.so in-tree with nvcc for sm_103a (GB300).

Each CUDA translation unit is compiled in parallel to an object under _build/, then
linked into attention_scored_kv_gb300/_lib/libkvs.so.  The same sources built with
-DKVS_DEBUG (device-side bounds checks, NaN-poisoned scratch) give _lib/libkvs_debug.so,
which the binding loads when KVS_LIB_VARIANT=debug.  No cmake, no torch extension
machinery: plain nvcc, one -gencode.  Rebuilds only what changed (by mtime).
"""

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "libkvs.so")
LIB_DEBUG = os.path.join(LIBDIR, "libkvs_debug.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc():
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvs")
    return exe


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hdrs.append(os.path.join(INCLUDE, "kvs.h"))
    return max(os.path.getmtime(h) for h in hdrs)


def _compile(src, extra, objdir=BUILD):
    obj = os.path.join(objdir, os.path.basename(src) + ".o")
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), _deps()):
        return obj, ""
    cmd = [nvcc()] + ARCH + FLAGS + extra + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
    return obj, r.stderr


def _link(objs, lib):
    if not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs):
        cmd = [nvcc()] + ARCH + ["-shared", "-Xcompiler", "-fPIC", "-o", lib] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))


def build(verbose=False, ptxas_info=False, debug=True):
    """Compile every translation unit and link libkvs.so (and, with debug, the checked
    variant libkvs_debug.so); returns the release library's path."""
    dbg_dir = os.path.join(BUILD, "debug")
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(dbg_dir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    srcs = sources()
    jobs = [(src, extra, BUILD) for src in srcs]
    if debug:
        jobs += [(src, ["-DKVS_DEBUG"], dbg_dir) for src in srcs]
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(16, len(jobs))) as ex:
        results = list(ex.map(lambda j: _compile(*j), jobs))
    if verbose:
        for _, log in results:
            if log:
                sys.stderr.write(log)
    n = len(srcs)
    _link([o for o, _ in results[:n]], LIB)
    if debug:
        _link([o for o, _ in results[n:]], LIB_DEBUG)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv))
