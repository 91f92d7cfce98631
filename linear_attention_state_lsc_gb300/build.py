"""Build liblsc.so (sm_103a) in-tree with nvcc: one object per translation unit,
compiled in parallel, linked with the static CUDA runtime.

    python -m linear_attention_state_lsc_gb300.build [--force] [--ptxas-info]
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "liblsc.so")
SOURCES = ["lsc_host.cu", "lsc_copy.cu", "lsc_gdn.cu", "lsc_rec128.cu", "lsc_chunked_tc.cu", "lsc_chunk_prep.cu", "lsc_noalloc.cu", "lsc_decode_f32.cu", "lsc_decode_bf16.cu",
           "lsc_prefill.cu", "lsc_kv.cu", "lsc_prefix_cache.cpp", "lsc_store.cpp"]
HEADERS = [os.path.join(CSRC, h) for h in ("lsc_internal.h", "lsc_ptx.h", "lsc_tc.h", "lsc_chunk.h", "lsc_gdn_common.cuh", "lsc_decode.cuh")] + \
    [os.path.join(INCLUDE, h) for h in ("lsc.h", "lsc_prefix_cache.h", "lsc_kv.h", "lsc_store.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if ptxas_info:
        flags += ["-Xptxas", "-v"]
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        if force or ptxas_info or _stale(o, [s] + HEADERS):
            jobs.append([cc] + flags + ["-c", s, "-o", o])
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs))
    for cmd, r in zip(jobs, results):
        if r.returncode != 0 or ptxas_info:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed: " + " ".join(cmd))
    objs = [os.path.join(BUILD, os.path.splitext(s)[0] + ".o") for s in SOURCES]
    if force or jobs or _stale(LIB, objs):
        subprocess.run([cc] + ARCH + ["-shared", "-o", LIB + ".tmp"] + objs, check=True)
        os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, ptxas_info="--ptxas-info" in sys.argv))
