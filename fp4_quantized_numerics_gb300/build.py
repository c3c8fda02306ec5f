"""Build libufp4.so (the CUDA library behind include/ufp4.h) for sm_103a.

In-tree build: objects go to fp4_quantized_numerics_gb300/_build/, the shared
library to fp4_quantized_numerics_gb300/libufp4.so.  Translation units are
compiled in parallel with nvcc; a unit is rebuilt when it or any header is
newer than its object.  No cmake, no torch extension machinery.
"""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libufp4.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
    "-Xcompiler", "-fPIC,-fvisibility=hidden",
    "-I", os.path.join(ROOT, "include"),
]


def nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libufp4 needs the CUDA toolkit to build")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, extra, build_dir=BUILD, deps=()):
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    if _stale(obj, [src] + _headers() + list(deps)):
        cmd = [nvcc(), *NVCC_FLAGS, *extra, "-c", src, "-o", obj + ".tmp"]
        subprocess.check_call(cmd)
        os.replace(obj + ".tmp", obj)
    return obj


def _link(lib, objs):
    if _stale(lib, objs):
        tmp = lib + ".tmp.%d" % os.getpid()
        subprocess.check_call([nvcc(), *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, lib)
    return lib


def build(verbose=False, extra_flags=()):
    """Compile every .cu under csrc/ and link libufp4.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, list(extra_flags)), srcs))
    _link(LIB, objs)
    if verbose:
        print(LIB)
    return LIB


def build_variant(lib, build_dir, flags, sources, include_dir):
    """A test-only variant of the library: `sources` (file names under csrc/)
    recompiled with `flags` and -I include_dir (whose files they may include)
    into build_dir, linked with the library's other objects into `lib`.
    Builds the library's objects first.  Returns the variant's path."""
    os.makedirs(build_dir, exist_ok=True)
    deps = glob.glob(os.path.join(include_dir, "*"))
    extra = list(flags) + ["-I", include_dir]
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    mine = [s for s in srcs if os.path.basename(s) in sources]
    # the library and the variant's own objects compile side by side
    with cf.ThreadPoolExecutor(max_workers=1 + len(mine)) as ex:
        lib_job = ex.submit(build)
        jobs = {s: ex.submit(_compile, s, extra, build_dir, deps) for s in mine}
        lib_job.result()
        objs = [jobs[s].result() if s in jobs else os.path.join(BUILD, os.path.basename(s) + ".o")
                for s in srcs]
    return _link(lib, objs)


if __name__ == "__main__":
    build(verbose=True)
