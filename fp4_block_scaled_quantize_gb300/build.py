"""Build libfp4gb300.so for sm_103a (GB300) with nvcc, in-tree.

Each CUDA translation unit is compiled in parallel into _build/, then linked
into fp4_block_scaled_quantize_gb300/_lib/libfp4gb300.so.  The quantizer
units are built with -fmad=false so no multiply-add is contracted into an FMA
(their arithmetic is specified as separately rounded binary32 operations).
"""
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libfp4gb300.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC,
          "--expt-relaxed-constexpr"]
UNITS = {
    "abi.cu": [],
    "amax.cu": ["-fmad=false"],
    "quantize.cu": ["-fmad=false"],
    "remap.cu": ["-fmad=false"],
    "convert.cu": ["-fmad=false"],
    "dequant.cu": ["-fmad=false"],
    "gemm.cu": [],
    "gemm2.cu": [],
    "mmarate.cu": [],
}


def nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _stale(obj, deps):
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose=False, extra=()):
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    headers.append(os.path.join(INCLUDE, "fp4.h"))
    procs, objs = [], []
    for unit, flags in UNITS.items():
        src = os.path.join(CSRC, unit)
        obj = os.path.join(BUILD, unit.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            cmd = [nvcc()] + ARCH + COMMON + flags + list(extra) + ["-c", src, "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            procs.append((unit, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                 stderr=subprocess.STDOUT, text=True)))
    failed = []
    for unit, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            sys.stdout.write(out)
        if p.returncode:
            failed.append(unit)
    if failed:
        raise RuntimeError("nvcc failed for " + ", ".join(failed))
    if force or procs or not os.path.exists(LIB) or _stale(LIB, objs):
        tmp = LIB + ".tmp"
        subprocess.run([nvcc()] + ARCH + ["-shared", "-o", tmp] + objs, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
