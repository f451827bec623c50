"""Builds libmtp.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel; the result is
``mtp_speculative_decoding_gb300/libmtp.so``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
# per-machine build folder: objects and the library of another architecture never mix
BUILD = os.path.join(PKG, "_build", platform.machine())
LIB = os.path.join(BUILD, "libmtp.so")

# (object name, source, extra defines): the draft kernel's variants are one
# source compiled once per (weight type, head dimension, tensor-core paths)
UNITS = [("api", "api.cu", []), ("verify", "verify.cu", []), ("noalloc", "noalloc.cu", []),
         ("draft_dispatch", "draft_dispatch.cu", [])]
for _hd in (32, 64, 128, 256, 512):
    for _name, _bf, _tc in (("f32", 0, 0), ("bf16_cc", 1, 0), ("bf16_tc", 1, 1)):
        UNITS.append((f"draft_{_name}_{_hd}", "draft_inst.cu",
                      [f"-DMTP_WT_BF16={_bf}", f"-DMTP_HD={_hd}", f"-DMTP_TC={_tc}"]))
for _hd in (64, 128, 256):   # Q8_0 and Q4_0 projections
    UNITS.append((f"draft_q8_{_hd}", "draft_inst.cu", ["-DMTP_WT_BF16=1", f"-DMTP_HD={_hd}", "-DMTP_TC=0", "-DMTP_Q8=1"]))
    UNITS.append((f"draft_q4_{_hd}", "draft_inst.cu", ["-DMTP_WT_BF16=1", f"-DMTP_HD={_hd}", "-DMTP_TC=0", "-DMTP_Q4=1"]))
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.sep not in c or os.path.exists(c)):
            return c
    return "nvcc"


def _flags() -> list[str]:
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2,-ffp-contract=off", "-I", INCLUDE, "-I", CSRC,
                   "--expt-relaxed-constexpr"]


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    deps = [src] + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    deps.append(os.path.join(INCLUDE, "mtp.h"))
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    jobs = []
    for name, s, defs in UNITS:
        src = os.path.join(CSRC, s)
        obj = os.path.join(BUILD, name + ".o")
        if force or _stale(obj, src):
            cmd = [nvcc] + _flags() + defs + (["-Xptxas", "-v"] if ptxas_info else []) + ["-c", src, "-o", obj]
            jobs.append((name, cmd))
    if jobs:
        def run(job):
            name, cmd = job
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {name}:\n{r.stderr}")
            return name, r.stderr
        with cf.ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
            for name, err in ex.map(run, jobs):
                if verbose and err:
                    print(f"--- {name}\n{err}")
    objs = [os.path.join(BUILD, name + ".o") for name, _, _ in UNITS]
    # relink also when an object is newer than the library (a link that failed after its compiles)
    if force or jobs or not os.path.exists(LIB) or any(os.path.getmtime(o) > os.path.getmtime(LIB) for o in objs):
        cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", LIB + ".tmp"] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
