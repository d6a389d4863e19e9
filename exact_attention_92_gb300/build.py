"""Build libfa.so (the sm_103a CUDA library) in-tree with nvcc.

Each .cu file compiles to an object under ``_build/`` in parallel; the
objects link into ``exact_attention_92_gb300/libfa.so`` with the CUDA runtime
linked statically, so the library needs no libcudart at run time and loads on
a machine without a GPU driver (the tensor-map encoder is fetched from the
driver at first use).
"""

from __future__ import annotations

import concurrent.futures
import os
import re
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfa.so")

SOURCES = ["fa_api.cu", "fa_fwd.cu", "fa_fwd256.cu", "fa_bwd.cu", "fa_bwd_pair.cu", "fa_bwd256.cu", "fa_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libfa.so")
    return cand


def _flags(extra=()):
    return ["-O3", "-std=c++17", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
            "-I", INCLUDE, "-I", CSRC, *extra]


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "fa.h"), __file__]
    return max(os.path.getmtime(f) for f in files)


# Kernels that read tensor memory with tcgen05.ld: the destination registers
# of such a load are only valid after tcgen05.wait::ld, so a register spill
# between the two would store garbage.  The build refuses any spill in them.
NO_SPILL_KERNELS = ("fa_fwd_kernel", "fa_fwd256_kernel", "fa_bwd_dkdv_kernel", "fa_bwd_dkdv_pair_kernel",
                    "fa_bwd_dq_kernel", "fa_bwd256_kv_kernel", "fa_bwd256_dq_kernel")


# Kernels that move registers between warpgroups with setmaxnreg, and the
# per-thread count they must be launched with.  The split's shares are
# static_asserted against this count in the source; if ptxas gave the entry
# fewer registers, the warpgroup that asks for more would wait forever.
REG_SPLIT_KERNELS = {"fa_fwd_kernel": 168, "fa_bwd_dkdv_kernel": 168, "fa_bwd_dkdv_pair_kernel": 168,
                     "fa_bwd_dq_kernel": 168}


def check_spills(ptxas_log: str) -> None:
    entry = None
    for line in ptxas_log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            entry = m.group(1)
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and entry and any(k in entry for k in NO_SPILL_KERNELS):
            if int(m.group(1)) or int(m.group(2)):
                raise RuntimeError(f"register spills in {entry}: {line.strip()}")
        m = re.search(r"Used (\d+) registers", line)
        if m and entry:
            for k, regs in REG_SPLIT_KERNELS.items():
                if k in entry and int(m.group(1)) != regs:
                    raise RuntimeError(f"{entry} starts with {m.group(1)} registers, its register split needs {regs}")


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile and link libfa.so if any source is newer than it; return its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps() and not ptxas_verbose:
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc, *_flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    for _, log in results:
        check_spills(log)
    if verbose or ptxas_verbose:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    tmp = LIB + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of libfa.so failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="--ptxas-v" in sys.argv))
