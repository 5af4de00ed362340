"""Builds libcf.so (the C-ABI CUDA library) in-tree for sm_103a.

    python -m co_prefill_decode_gb300.build        # or build(verbose=True)

Each translation unit is compiled by nvcc in parallel, then linked into
co_prefill_decode_gb300/libcf.so.  Objects go to co_prefill_decode_gb300/_build/.
"""
import concurrent.futures as cf_futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libcf.so")
SOURCES = ["engine.cu", "gemm.cu", "decode_attn.cu", "prefill_attn.cu", "rowops.cu", "decode_noalloc.cu",
           "latency.cpp", "dispatch.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newer(src_paths, dst) -> bool:
    if not os.path.exists(dst):
        return True
    t = os.path.getmtime(dst)
    return any(os.path.getmtime(p) > t for p in src_paths)


def build(verbose: bool = False, ptxas_verbose: bool = False, force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(ROOT, "include", "cf.h"))
    jobs = []
    for src in SOURCES:
        sp = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        if force or _newer([sp] + headers, obj):
            cmd = [cc, *ARCH, *FLAGS, "-c", sp, "-o", obj]
            if ptxas_verbose:
                cmd += ["-Xptxas", "-v"]
            jobs.append((src, cmd))

    def run(job):
        src, cmd = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, r

    failed = []
    with cf_futures.ThreadPoolExecutor(max_workers=min(8, max(1, len(jobs)))) as ex:
        for src, r in ex.map(run, jobs):
            if verbose or ptxas_verbose or r.returncode:
                sys.stderr.write(f"--- {src}\n{r.stdout}{r.stderr}")
            if r.returncode:
                failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    objs = [os.path.join(BUILD, os.path.splitext(s)[0] + ".o") for s in SOURCES]
    if force or jobs or _newer(objs, LIB):
        cmd = [cc, *ARCH, "-shared", "-o", LIB, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode:
            raise RuntimeError(f"link failed:\n{r.stdout}{r.stderr}")
    return LIB


if __name__ == "__main__":
    build(verbose=True, ptxas_verbose="-v" in sys.argv, force="-f" in sys.argv)
    print(LIB)
