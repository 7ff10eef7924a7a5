"""Builds libxs.so in-tree with nvcc for sm_103a (no CMake, no torch extension).

Each translation unit is compiled in parallel into ``_build/`` and linked into
``comm_comp_fusion_gb300/libxs.so`` with the CUDA runtime linked statically.
The attention kernels use ``setmaxnreg`` to move registers between
warpgroups; that is only safe if the kernel launches with exactly 128
registers per thread (512 threads x 128 = the whole register file), so the
build reads ptxas' report and refuses a library where that does not hold.
"""
from __future__ import annotations

import os
import re
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libxs.so")
ROOT = os.path.dirname(PKG)

SOURCES = ["xs_attn_d128.cu", "xs_attn_f8.cu", "xs_attn_d256.cu", "xs_attn_d96.cu", "xs_attn_d64.cu", "xs_attn.cu", "xs_permute.cu", "xs_api.cpp", "xs_schedule.cpp",
           "xs_noalloc.cu", "xs_burst.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newest_input_mtime() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths += [os.path.join(ROOT, "include", "xs.h"), __file__]
    return max(os.path.getmtime(p) for p in paths if os.path.exists(p))


def _compile(src: str) -> tuple[str, str]:
    nvcc = _nvcc()
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc, "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC,-O2", "-Xptxas", "-v",
           "-I", os.path.join(ROOT, "include"), "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stdout + r.stderr


def check_attention_registers(ptxas_log: str) -> None:
    """Every attn_fwd_kernel instance must report exactly 128 registers."""
    current = None
    seen = 0
    for line in ptxas_log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and current and "attn_fwd_kernel" in current:
            seen += 1
            if int(m.group(1)) != 128:
                raise RuntimeError(f"{current} uses {m.group(1)} registers; the setmaxnreg split needs 128")
    if seen == 0:
        raise RuntimeError("ptxas report has no attention kernel entries")


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input_mtime():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    log = "\n".join(r[1] for r in results)
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        f.write(log)
    if verbose:
        print(log)
    check_attention_registers(log)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [_nvcc(), "-shared", *ARCH, "-cudart", "static", "-o", tmp] + [r[0] for r in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
