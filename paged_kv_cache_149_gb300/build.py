"""Build libpa.so in-tree with nvcc for sm_103a (GB300).

Each source is compiled in its own nvcc process (in parallel), then linked into
``paged_kv_cache_149_gb300/libpa.so``.  ``python -m paged_kv_cache_149_gb300.build``
does the same from the command line.
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libpa.so")
SOURCES = ["pa_api.cu", "pa_decode.cu", "pa_decode_fp8.cu", "pa_decode_int4.cu", "pa_decode_append.cu",
           "pa_decode_append_fp8.cu", "pa_decode_append_int4.cu", "pa_decode_timed.cu",
           "pa_prefill.cu", "pa_cache_ops.cu", "pa_fixed_scratch.cu", "pa_pool.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpa.so")
    return path


def _compile(src, verbose):
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    cmd = [nvcc(), "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O3", "-c",
           os.path.join(CSRC, src), "-o", obj, "-I", os.path.join(ROOT, "include")]
    if src.endswith(".cu"):
        cmd[1:1] = ARCH
        if verbose:
            cmd += ["-Xptxas", "-v"]
    else:
        cmd += ["-x", "c++"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
    return obj, r.stderr


def build(verbose=False, force=False):
    """Compile every source and link libpa.so; returns the library path."""
    os.makedirs(BUILD, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    deps.append(os.path.join(ROOT, "include", "pa.h"))
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(d) for d in deps)):
        return LIB
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp] + [o for o, _ in results] + ["-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
