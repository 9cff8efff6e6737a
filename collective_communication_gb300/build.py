"""Build librar.so (the C-ABI library of sm_103a CUDA kernels) in-tree.

nvcc compiles each translation unit for sm_103a only, in parallel, then links
the shared library next to this file. Run as a script or through
__graft_entry__.build().
"""
import concurrent.futures
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "librar.so")
# the debug variant: the same sources with RAR_DEBUG (device-side slice bounds checks)
BUILD_DEBUG = os.path.join(HERE, "_build", "debug")
LIB_DEBUG = os.path.join(HERE, "librar_debug.so")
SOURCES = ["rar_api.cu", "ring_simple.cu", "ring_ll.cu", "oneshot.cu", "oneshot_staged.cu", "rar_static_ws.cu"]
HEADERS = ["rar_device.cuh", "rar_geometry.h", "rar_launch.h"]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-I", os.path.join(ROOT, "include"), "-I", CSRC,
]


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, verbose_ptxas=False, debug=False):
    obj = os.path.join(BUILD_DEBUG if debug else BUILD, src.replace(".cu", ".o"))
    deps = [os.path.join(CSRC, src)] + [os.path.join(CSRC, h) for h in HEADERS] + \
        [os.path.join(ROOT, "include", "rar.h")]
    if not _stale(obj, deps) and not verbose_ptxas:
        return obj, ""
    cmd = [NVCC, *FLAGS, *(["-DRAR_DEBUG"] if debug else []), "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose_ptxas: bool = False, debug: bool = False) -> str:
    """Compile and link librar.so (debug=True: librar_debug.so); returns its path."""
    build_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    if force:
        for s in SOURCES:
            o = os.path.join(build_dir, s.replace(".cu", ".o"))
            if os.path.exists(o):
                os.remove(o)
    with concurrent.futures.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose_ptxas, debug), SOURCES))
    objs = [o for o, _ in results]
    if verbose_ptxas:
        for _, log in results:
            sys.stderr.write(log)
    return _link(lib, objs, force)


def build_all(force: bool = False) -> list:
    """Both variants, compiled side by side: [librar.so, librar_debug.so]."""
    with concurrent.futures.ThreadPoolExecutor(2) as ex:
        return list(ex.map(lambda d: build(force=force, debug=d), (False, True)))


def _link(LIB, objs, force):
    if _stale(LIB, objs) or force:
        tmp = LIB + ".tmp%d" % os.getpid()
        cmd = [NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", tmp, *objs,
               "-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    if "--all" in sys.argv:
        print(build_all(force="--force" in sys.argv))
    else:
        print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, debug="--debug" in sys.argv))
