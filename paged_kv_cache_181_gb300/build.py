"""Build libpagedkv.so in-tree: nvcc for the CUDA sources (sm_103a), g++ for host code.

    python -m paged_kv_cache_181_gb300.build [-v]

Translation units compile in parallel; the library links the CUDA runtime
statically, so it loads on a machine without a GPU (calls then fail with
PKV_ERR_CUDA) and needs no libcuda at link time (the TMA encode entry point is
fetched from the driver at run time).
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
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpagedkv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_SOURCES = ["device.cu", "kv_write.cu", "attn_simt.cu", "attn_tc.cu", "noalloc.cu", "selftest.cu"]
HOST_SOURCES = ["host.cpp"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd: list[str], verbose: bool, log: str | None = None) -> str:
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if verbose and res.stdout.strip():
        print(res.stdout, flush=True)
    if res.returncode != 0:
        raise RuntimeError(f"build step failed ({res.returncode}): {' '.join(cmd)}\n{res.stdout}")
    if log:
        with open(log, "w") as f:
            f.write(res.stdout)
    return res.stdout


# The tensor-core attention kernel hands registers between its warpgroups with setmaxnreg, a split
# sized for exactly the register count the kernel is compiled to; that count is checked here, from
# ptxas's report, so that a toolchain which allocates differently fails the build instead of every
# bf16/f16 call at run time (the launcher keeps the same check as a backstop).
TC_SOURCE = "attn_tc.cu"
TC_KERNEL = "attn_tc_kernel"
# Sources whose ptxas report is kept beside their object (`<source>.ptxas.txt`): the tensor-core kernel's for
# the gate below, the CUDA-core kernel's for its spill check (it runs at 252-254 registers, where a
# toolchain that allocated differently would start spilling: slower, not wrong).
PTXAS_LOGGED = (TC_SOURCE, "attn_simt.cu")


def expected_tc_registers(source: str) -> int:
    m = re.search(r"constexpr\s+int\s+kLaunchRegs\s*=\s*(\d+)", source)
    if not m:
        raise RuntimeError(f"{TC_SOURCE}: kLaunchRegs not found")
    return int(m.group(1))


def check_tc_registers(ptxas_log: str, expected: int) -> int:
    """Every instantiation of the tensor-core kernel in a ``-Xptxas -v`` log uses ``expected`` registers;
    returns how many instantiations were checked, raises RuntimeError otherwise."""
    seen = 0
    current = None
    for line in ptxas_log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and current is not None:
            if TC_KERNEL in current:
                seen += 1
                if int(m.group(1)) != expected:
                    raise RuntimeError(
                        f"{TC_SOURCE}: {current} compiled to {m.group(1)} registers per thread, but its warpgroup "
                        f"register split (setmaxnreg) is sized for {expected}; adjust kLaunchRegs/kRegsLow/"
                        f"kRegsHigh or the kernel's register use")
            current = None
    if seen == 0:
        raise RuntimeError(f"{TC_SOURCE}: no register report for {TC_KERNEL} in the ptxas output")
    return seen


def spills(ptxas_log: str, kernel: str) -> list[tuple[str, int, int]]:
    """(function, spill store bytes, spill load bytes) of every instantiation of ``kernel`` in a
    ``-Xptxas -v`` log."""
    out = []
    current = None
    for line in ptxas_log.splitlines():
        m = re.search(r"(?:Compiling entry function|Function properties for) '?([^' ]+)'?", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and current is not None and kernel in current:
            out.append((current, int(m.group(1)), int(m.group(2))))
            current = None
    return out


def _stale(obj: str, deps: list[str]) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile every source that changed and link libpagedkv.so; return its path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "pagedkv.h"))
    jobs = []
    objs = []
    tc_log = os.path.join(OUT_DIR, TC_SOURCE + ".ptxas.txt")
    for src in CUDA_SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(OUT_DIR, src + ".o")
        objs.append(obj)
        log = os.path.join(OUT_DIR, src + ".ptxas.txt") if src in PTXAS_LOGGED else None
        if force or _stale(obj, [path, *headers]) or (log is not None and _stale(log, [obj])):
            cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                   "-I", INCLUDE, "-I", CSRC, "-c", path, "-o", obj]
            if ptxas_verbose or log is not None:
                cmd += ["-Xptxas", "-v"]
            jobs.append((cmd, log))
    for src in HOST_SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(OUT_DIR, src + ".o")
        objs.append(obj)
        if force or _stale(obj, [path, *headers]):
            jobs.append((["g++", "-O2", "-std=c++17", "-fPIC", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC, "-c",
                          path, "-o", obj], None))
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for f in [ex.submit(_run, cmd, verbose, log) for cmd, log in jobs]:
                f.result()
    with open(os.path.join(CSRC, TC_SOURCE)) as f:
        expected = expected_tc_registers(f.read())
    with open(tc_log) as f:
        try:
            check_tc_registers(f.read(), expected)
        except RuntimeError:
            os.remove(tc_log)  # the next build compiles the kernel again
            raise
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + ".tmp"
        _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-lpthread", "-ldl", "-lrt"], verbose)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    v = "-v" in sys.argv
    print(build(verbose=v, force="-f" in sys.argv, ptxas_verbose="--ptxas" in sys.argv))
