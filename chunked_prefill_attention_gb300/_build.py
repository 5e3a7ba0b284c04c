"""Build libq8attn.so in-tree with nvcc for sm_103a (one -gencode, parallel TUs)."""

import concurrent.futures
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libq8attn.so")
SOURCES = ["api.cu", "quantize.cu", "state.cu", "chunk_step.cu", "pipeline.cu", "graph.cu"]
HEADERS = ["ptx.cuh", "internal.h"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libq8attn.so")
    return cand


def _flags():
    # no fast-math anywhere: the quantiser and the finaliser rely on IEEE divides
    return [ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
            "-I", os.path.join(ROOT, "include"), "-Xptxas", "-v"]


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, s) for s in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "q8attn.h"),
                                                                   os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose=False):
    """Compile every translation unit in parallel and link the shared library."""
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *_flags(), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            if log.strip():
                print(log)
    tmp = LIB + ".tmp"
    cmd = [nvcc, ARCH, "-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


SANITIZED_LIB = os.path.join(PKG, "libq8attn_sanitized.so")
HOST_SOURCES = ["api.cu", "pipeline.cu", "graph.cu"]   # the C-ABI layer: validation, streams, events, graphs


def build_sanitized():
    """libq8attn_sanitized.so: the same library with the host code of the C-ABI
    layer built with AddressSanitizer and UndefinedBehaviorSanitizer (the
    kernels are unchanged).  Load it with the sanitizer runtime preloaded."""
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    # one flag per -Xcompiler: nvcc splits its arguments at commas
    san = [f"-Xcompiler={f}" for f in ("-fsanitize=address", "-fsanitize=undefined",
                                        "-fno-omit-frame-pointer", "-fno-sanitize-recover=all")]

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + (".san.o" if src in HOST_SOURCES else ".o"))
        if src not in HOST_SOURCES and os.path.exists(obj) and os.path.getmtime(obj) > os.path.getmtime(
                os.path.join(CSRC, src)):
            return obj
        cmd = [nvcc, *_flags(), *(san if src in HOST_SOURCES else []), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = SANITIZED_LIB + ".tmp"
    cmd = [nvcc, ARCH, "-shared", "-Xcompiler=-fsanitize=address", "-Xcompiler=-fsanitize=undefined", "-o",
           tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, SANITIZED_LIB)
    return SANITIZED_LIB


def ensure_built():
    if _stale():
        build()
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
