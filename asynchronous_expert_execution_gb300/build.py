"""Build the in-tree shared libraries for sm_103a.

``libmoe_async.so`` is the release library; ``libmoe_async_debug.so`` is the same code
compiled with MOE_DEBUG_BOUNDS, which checks every bucket, slot and k index the kernels read
back from device state and latches MOE_ERR_BOUNDS instead of touching memory out of range
(loaded when the environment sets MOE_DEBUG_BOUNDS=1).  nvcc compiles every translation unit
of both under ``csrc/`` in parallel and links each set into one shared object next to this
file.  A rebuild is skipped when a library is newer than every source and header.
"""
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libmoe_async.so")
LIB_DEBUG = os.path.join(HERE, "libmoe_async_debug.so")
BUILD_DIR = os.path.join(ROOT, "_build")
VARIANTS = {"release": (LIB, []), "debug": (LIB_DEBUG, ["-DMOE_DEBUG_BOUNDS=1"])}

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE]
# The tcgen05 kernel must not spill: it holds an SM's whole register file, and a build of a
# variant that spilled faulted on the GPU.  ptxas turns a spill into a build error.
FILE_FLAGS = {"moe_ffn_tc.cu": ["-Xptxas", "--warn-on-spills,--warning-as-error"]}


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe_async.so")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(lib):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return any(os.path.getmtime(p) > t for p in deps)


def build(force=False, verbose=False, variants=("release", "debug")):
    """Compile and link the requested libraries (all translation units of all of them in
    parallel); returns the release library's path."""
    todo = [v for v in variants if force or _stale(VARIANTS[v][0])]
    if not todo:
        return LIB
    nvcc = _nvcc()
    procs, objs = [], {}
    for v in todo:
        bdir = os.path.join(BUILD_DIR, v)
        os.makedirs(bdir, exist_ok=True)
        objs[v] = []
        for src in sources():
            obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
            cmd = [nvcc, *ARCH, *NVCC_FLAGS, *FILE_FLAGS.get(os.path.basename(src), []), *VARIANTS[v][1],
                   "-c", src, "-o", obj]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
            objs[v].append(obj)
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((src, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"), file=sys.stderr)
    if failed:
        msg = "\n".join(f"--- {s}\n{o}" for s, o in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    for v in todo:
        lib = VARIANTS[v][0]
        tmp = lib + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs[v]]
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
