"""Build the CUDA library ``libw4a8.so`` in-tree (``w4a8_block_quantized_gb300/_build``).

sm_103a only: every translation unit is compiled with
``-gencode arch=compute_103a,code=sm_103a``.  The units compile in parallel and the
build is skipped when the library is newer than every source and header.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import re
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libw4a8.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libw4a8.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        [os.path.join(ROOT, "include", "w4a8.h"), os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _deps())


# Kernels that re-split registers between warpgroups (setmaxnreg) need exactly this many
# registers per thread at launch: the split in gemm.cu is sized against it, and a smaller
# launch allocation would leave setmaxnreg.inc waiting for registers that never come.  Keys
# are matched against the mangled entry names; the debug instantiation of the 256-token
# kernel (template argument true, "ILb1E") does not re-split and is not checked.
REGISTER_SPLIT_KERNELS = {"gemm_kernel": 96, "gemm_wide_kernelILb0E": 96, "gemm_packed_kernel": 96}


def check_register_split(ptxas_log: str) -> None:
    """Fail the build if a register-split kernel was not compiled with its launch count."""
    current = None
    seen = 0
    for line in ptxas_log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and current:
            for name, want in REGISTER_SPLIT_KERNELS.items():
                if name in current:
                    seen += 1
                    if int(m.group(1)) != want:
                        raise RuntimeError(f"{current}: ptxas used {m.group(1)} registers per thread, "
                                           f"the warpgroup register split needs exactly {want}")
            current = None
    if seen == 0:
        raise RuntimeError("register check: no register-split kernel found in the ptxas report")


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
                     "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")]
    if ptxas_verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        split = os.path.basename(src) == "gemm.cu"
        cmd = [cc, *common, *([] if ptxas_verbose or not split else ["-Xptxas", "-v"]), "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if split:
            check_register_split(r.stdout + r.stderr)
        if verbose or ptxas_verbose:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=4) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv))
