"""Build libhq.so (the C-ABI library) for sm_103a with nvcc, in-tree.

Translation units compile in parallel; the objects go to _build/ and the
shared library next to this file.  Only nvcc and a host C++ compiler are used.
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libhq.so")
# The debug build: the same sources with HQ_DEBUG_BOUNDS, whose device-side index checks record HQ_ERR_BOUNDS in the
# workspace status and skip the access instead of trapping.  The binding loads it when HQ_LIBRARY=debug.
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libhq_debug.so")
SOURCES = ["hq_api.cu", "hq_pack.cu", "hq_route.cu", "hq_gemm_int4.cu", "hq_gemm_nvfp4.cu", "hq_gemm_mxfp4.cu", "hq_gemm_mxfp4a.cu", "hq_gemm_mxfp4x.cu", "hq_gemm_mxfp4x_comb.cu", "hq_gemm_small.cu", "hq_gemm_small_fmt.cu", "hq_gemm_small_bits.cu", "hq_splitk.cu", "hq_noalloc.cu", "hq_act_quant.cu", "hq_moe_combine.cu", "hq_gemm_int4_comb.cu", "hq_gemm_nvfp4_comb.cu", "hq_gemm_mxfp4_comb.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden"]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libhq.so")
    return cand


def _stale(obj, src_files):
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(s) > t for s in src_files)


def build(verbose=False, force=False, debug=False):
    """Compile every translation unit and link libhq.so (debug: libhq_debug.so); returns the library path."""
    out_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    flags = FLAGS + (["-DHQ_DEBUG_BOUNDS=1"] if debug else [])
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(os.path.dirname(HERE), "include", "hq.h"))
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(out_dir, src.replace(".cu", ".o"))
        if force or _stale(o, [s] + headers):
            jobs.append([nvcc, *ARCH, *flags, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        if verbose:
            sys.stdout.write(r.stdout + r.stderr)
        return cmd[-1]

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        list(ex.map(run, jobs))
    objs = [os.path.join(out_dir, s.replace(".cu", ".o")) for s in SOURCES]
    if force or jobs or not os.path.exists(lib):
        cmd = [nvcc, *ARCH, "-shared", "-o", lib, *objs, "-lcudart_static", "-ldl", "-lrt", "-lpthread"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, debug="--debug" in sys.argv))
