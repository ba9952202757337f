"""Build libsvpa.so in-tree with nvcc for sm_103a (GB300).

Translation units are compiled in parallel; spec_accept.cu is compiled with
-fmad=false so that the acceptance product is never fused into a
multiply-add.  Run ``python -m speculative_verify_paged_attn_gb300.build``.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "libsvpa.so")
BUILD = os.path.join(HERE, "_build")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "--expt-relaxed-constexpr", "-diag-suppress", "177"]
SOURCES = {
    "svpa_api.cu": [],
    "paged_verify_attn.cu": [],
    "paged_verify_attn_tc.cu": [],
    "paged_verify_attn_f8.cu": [],
    "spec_accept.cu": ["-fmad=false"],
    "block_table_commit.cu": [],
    "kv_append.cu": ["-fmad=false"],
    "gamma_control.cu": ["-fmad=false"],
    "svpa_noalloc.cu": [],
    "svpa_logits_api.cu": [],
    "svpa_step_api.cu": [],
    "wait_selftest.cu": [],
}


def _stamp() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(HERE, "..", "include", "svpa.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(OUT) and os.path.getmtime(OUT) >= _stamp():
        return OUT
    os.makedirs(BUILD, exist_ok=True)

    def compile_one(item):
        src, extra = item
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [NVCC, *ARCH, *COMMON, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES.items()))
    tmp = OUT + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
