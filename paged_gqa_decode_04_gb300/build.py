"""Build libpaged_gqa.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

Each translation unit is compiled by nvcc in parallel into ``_build/``, then
linked into ``libpaged_gqa.so`` beside this file.  No torch, no cmake.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpaged_gqa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["api.cpp", "block_manager.cpp", "decode_simple.cu", "decode_tma_d64.cu",
           "decode_tma_d128.cu", "decode_tma_d128_share.cu", "decode_tma_d128_sep.cu",
           "decode_tma_fp8.cu", "decode_tma_fp8_share.cu", "decode_tma_fp8_sep.cu",
           "decode_tma_i8.cu", "decode_tma_i8_share.cu", "decode_tma_i8_sep.cu",
           "decode_tma_fp8pb.cu", "decode_tma_fp8pb_share.cu", "decode_tma_fp8pb_sep.cu",
           "decode_tma_i8pb.cu", "decode_tma_i8pb_share.cu", "decode_tma_i8pb_sep.cu",
           "kv_write.cu", "merge.cu", "noalloc.cu", "selftest.cu"]


def nvcc():
    path = shutil.which("nvcc")
    if path:
        return path
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return (ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                    "-I" + INCLUDE, "-I" + CSRC] + list(extra))


def _stale(lib, deps):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose=False, extra_flags=()):
    """Compile and link if any source or header is newer than the library."""
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    deps.append(os.path.abspath(__file__))
    if not force and not _stale(LIB, deps):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [cc] + _flags(extra_flags) + ["-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cu"):
            cmd += ["-Xptxas", "-v"] if verbose else []
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), res.stderr))
        return obj, res.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for obj, log in results:
            if log.strip():
                print(log)
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), res.stderr))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
