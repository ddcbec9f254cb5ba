"""Build the C-ABI library ``_build/libua_gb300.so`` in-tree for sm_103a.

Each translation unit compiles in parallel (nvcc for ``.cu``, g++ for the
host-only planner), then nvcc links a shared library with the CUDA runtime
linked statically, so the library needs no ``libcudart`` at load time and
loads (without running anything) on machines that have no GPU.

    python -m paged_varlen_attention_gb300.build_lib [--force]
"""
from __future__ import annotations

import concurrent.futures as cf
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
LIB = os.path.join(BUILD, "libua_gb300.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr"]
CXX_FLAGS = ["-O2", "-fPIC", "-std=c++17", "-Wall"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    cu = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    cpp = sorted(f for f in os.listdir(CSRC) if f.endswith(".cpp"))
    return cu, cpp


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def _compile(cmd, log_path):
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(log_path, "w") as fh:
        fh.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}{r.stderr}")
    return log_path


# Register ceilings of the kernels: both prefill kernels run 384 threads on one
# SM, so a thread may hold at most 65536 / 384 -> 168 registers; a build where
# ptxas goes past that is refused.
LAUNCH_REGS = {"ua_prefill_kernel": 168, "ua_prefill_pair_kernel": 168}


def _registers_by_kernel(log_text: str) -> dict:
    out, current = {}, None
    for line in log_text.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and current:
            out[current] = int(m.group(1))
    return out


def _check_launch_registers(log_path: str):
    regs = _registers_by_kernel(open(log_path).read())
    for mangled, n in regs.items():
        for name, want in LAUNCH_REGS.items():
            if name in mangled and n > want:
                raise RuntimeError(f"{name}: ptxas chose {n} registers per thread, more than "
                                   f"the {want} its launch allows; refusing to build")


def build(force: bool = False, verbose: bool = False, prefill=None, pair=None) -> str:
    """Compile every CUDA / C++ source of the library; return the .so path.

    prefill=False builds a library whose planner sends every row tile to the
    decode kernel (used to cross-check the two kernels against each other);
    pair=False runs head-size-128 prefill rows on one SM per work item instead
    of on SM pairs.  None keeps the setting of the existing build (both on by
    default).
    """
    stamp = os.path.join(BUILD, "prefill_flag")
    os.makedirs(BUILD, exist_ok=True)
    old_flag = open(stamp).read() if os.path.exists(stamp) else ""
    old_defs = old_flag.split()
    if prefill is None:
        prefill = "-DUA_PREFILL_ENABLED=0" not in old_defs
    if pair is None:
        pair = "-DUA_PREFILL_PAIR=0" not in old_defs
    defines = [f"-DUA_PREFILL_ENABLED={int(bool(prefill))}", f"-DUA_PREFILL_PAIR={int(bool(pair))}"]
    if (not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime()
            and old_flag == " ".join(defines)):
        return LIB
    nvcc = _nvcc()
    cu, cpp = _sources()
    jobs = []
    objs = []
    for f in cu:
        obj = os.path.join(BUILD, f + ".o")
        objs.append(obj)
        jobs.append(([nvcc, *ARCH, *NVCC_FLAGS, *defines, "-I", INCLUDE, "-I", CSRC, "-c",
                      os.path.join(CSRC, f), "-o", obj], obj + ".log"))
    cxx = os.environ.get("CXX", "g++")
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "include")
    for f in cpp:
        obj = os.path.join(BUILD, f + ".o")
        objs.append(obj)
        jobs.append(([cxx, *CXX_FLAGS, *defines, "-I", INCLUDE, "-I", CSRC, "-I", cuda_inc, "-c",
                      os.path.join(CSRC, f), "-o", obj], obj + ".log"))
    with cf.ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
        logs = list(ex.map(lambda j: _compile(*j), jobs))
    if verbose:
        for lg in logs:
            sys.stdout.write(open(lg).read())
    for lg in logs:
        _check_launch_registers(lg)
    tmp = LIB + ".tmp"
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lpthread", "-ldl", "-lrt"]
    _compile(link, os.path.join(BUILD, "link.log"))
    os.replace(tmp, LIB)
    with open(stamp, "w") as fh:
        fh.write(" ".join(defines))
    return LIB


if __name__ == "__main__":
    pf = False if "--no-prefill" in sys.argv else (True if "--prefill" in sys.argv else None)
    pr = False if "--no-pair" in sys.argv else (True if "--pair" in sys.argv else None)
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, prefill=pf, pair=pr))
