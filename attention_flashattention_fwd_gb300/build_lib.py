"""Build ``libgbattn.so`` (the CUDA library behind include/gbattn.h) in-tree.

Each ``csrc/*.cu`` file is compiled for sm_103a only, in parallel, then
linked into a shared library with the CUDA runtime linked statically, so the
library needs nothing but the NVIDIA driver at run time.  ``debug=True``
builds ``libgbattn_debug.so`` instead: the same sources with GBATTN_DEBUG
defined, whose kernels check every direct global-memory index against its
buffer and report an out-of-range one instead of making the access.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libgbattn.so")
LIB_DEBUG = os.path.join(HERE, "libgbattn_debug.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE,
         "-Xptxas", "-v", "--expt-relaxed-constexpr"]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "gbattn.h")]


def up_to_date(lib=LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    lib = LIB_DEBUG if debug else LIB
    if not force and up_to_date(lib):
        return lib
    nvcc = _nvcc()
    objdir = os.path.join(HERE, "_build_debug" if debug else "_build")
    os.makedirs(objdir, exist_ok=True)
    defines = ["-DGBATTN_DEBUG"] if debug else []

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src).replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, *defines, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        with open(obj + ".ptxas.txt", "w") as f:
            f.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(_sources())) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        for o in objs:
            print(open(o + ".ptxas.txt").read())
    return lib


def build_all(force: bool = False) -> None:
    """The release and the debug library, compiled side by side."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        list(ex.map(lambda dbg: build(force=force, debug=dbg), (False, True)))


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                debug="--debug" in sys.argv))
