"""Builds libpa.so (the C-ABI library) for sm_103a with nvcc, in-tree.

Each .cu file under csrc/ is compiled to an object in parallel, then linked
into ``paged_kv_cache_gb300/_build/libpa.so`` with the CUDA runtime linked
statically and only the ``pa_*`` symbols exported.  Usage:
``python -m paged_kv_cache_gb300.build [--force] [--verbose] [--trace]``.
``--trace`` builds the profiling variant ``_build_trace/libpa_trace.so``
instead: the same library with globaltimer marks in the decode kernels and
two more exports that read them (``decode_trace.py`` uses it).
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libpa.so")
TRACE_DIR = os.path.join(HERE, "_build_trace")
TRACE_LIB = os.path.join(TRACE_DIR, "libpa_trace.so")
TRACE_EXPORTS = ("pa_trace_decode_reset", "pa_trace_decode_read")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpa.so")
    return path


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def deps():
    extra = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".map"))]
    return extra + [os.path.join(INCLUDE, "pa.h"), os.path.abspath(__file__)]


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in sources() + deps())


def _compile(src: str, verbose: bool, out_dir: str = OUT_DIR, defines=()) -> str:
    obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
           "--expt-relaxed-constexpr", *["-D" + d for d in defines], "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s\n%s" % (src, r.stdout, r.stderr))
    if verbose:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles and links libpa.so if missing or stale; returns its path."""
    if not force and not needs_build():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    srcs = sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), srcs))
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs,
           "-Xlinker", "--version-script=" + os.path.join(CSRC, "exports.map")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    return LIB


def build_trace(verbose: bool = False) -> str:
    """Compiles and links the profiling variant libpa_trace.so; returns its path."""
    os.makedirs(TRACE_DIR, exist_ok=True)
    srcs = sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, TRACE_DIR, ("PA_DECODE_TRACE=1",)), srcs))
    exports = open(os.path.join(CSRC, "exports.map")).read().replace(
        "  local:", "".join("    %s;\n" % name for name in TRACE_EXPORTS) + "  local:")
    map_path = os.path.join(TRACE_DIR, "exports_trace.map")
    with open(map_path, "w") as f:
        f.write(exports)
    tmp = TRACE_LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-Xlinker", "--version-script=" + map_path]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, TRACE_LIB)
    return TRACE_LIB


if __name__ == "__main__":
    if "--trace" in sys.argv:
        print(build_trace(verbose="--verbose" in sys.argv))
    else:
        print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
