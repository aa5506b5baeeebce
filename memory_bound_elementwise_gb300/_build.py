"""Build ``libew.so`` (the C ABI of include/ew.h) in-tree with nvcc for sm_103a.

The translation units are compiled in parallel, then linked into
``memory_bound_elementwise_gb300/_lib/libew.so`` with the CUDA runtime linked
statically.  Floating-point flags keep IEEE behaviour: no flush-to-zero, no
contraction of separate multiplies and adds, IEEE division and square root
(the kernels spell out their rounding in PTX anyway).
"""
import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libew.so")
OBJ_DIR = os.path.join(OUT_DIR, "obj")

SOURCES = ["ew_api.cu", "ew_kernels_f32.cu", "ew_kernels_f16.cu", "ew_kernels_bf16.cu", "ew_tma.cu",
           "ew_gather_fixed.cu", "ew_gather_fixed_wide.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "-ftz=false", "-prec-div=true", "-prec-sqrt=true", "-fmad=false",
              "-I", INCLUDE, "-I", CSRC]


def nvcc():
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found")


def _kernel_digest():
    """SHA-256 over the CUDA sources (kernels and dispatch) and the compiler
    flags, independent of where the repository sits on disk.  Profiler figures
    are tied to it."""
    h = hashlib.sha256()
    files = [os.path.join(CSRC, name) for name in sorted(os.listdir(CSRC))
             if name.endswith((".cu", ".cuh", ".h"))]
    for path in files:
        h.update(os.path.relpath(path, ROOT).encode())
        with open(path, "rb") as f:
            h.update(f.read())
    flags = [f for f in ARCH + NVCC_FLAGS if f not in (INCLUDE, CSRC)]
    h.update(" ".join(flags).encode())
    return h.hexdigest()


def source_digest():
    """SHA-256 over the kernel sources and flags (what profiler figures were taken on)."""
    return _kernel_digest()


def _inputs_digest():
    """Build stamp: the kernel sources and flags plus the public header."""
    h = hashlib.sha256(_kernel_digest().encode())
    with open(os.path.join(INCLUDE, "ew.h"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile and link libew.so unless an up-to-date build exists."""
    stamp = os.path.join(OUT_DIR, "build.sha256")
    digest = _inputs_digest() + ("|" + " ".join(extra_flags) if extra_flags else "")
    if (not force and os.path.exists(LIB) and os.path.exists(stamp)
            and open(stamp).read().strip() == digest):
        return LIB
    os.makedirs(OBJ_DIR, exist_ok=True)
    exe = nvcc()

    def compile_one(src):
        obj = os.path.join(OBJ_DIR, src.replace(".cu", ".o"))
        cmd = [exe, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s" % (src, r.stdout))
        return obj, r.stdout

    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            sys.stdout.write(log)
    objs = [o for o, _ in results]
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [exe, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s" % r.stdout)
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(digest)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
