"""Build the C-ABI library ``libgpuos.so`` (and the injectable op cubin) in-tree.

Only sm_103a is targeted. nvcc cross-compiles without a GPU, so this runs on
any machine with CUDA 13; each machine rebuilds it for its own host architecture.
Translation units compile in parallel; the whole build takes well under a
minute.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import re
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgpuos.so")
EXT_CUBIN = os.path.join(HERE, "gpuos_ext_ops.cubin")
# relocatable build of the executor: op modules are linked with it at run time
EXEC_RDC = os.path.join(HERE, "gpuos_exec_rdc.cubin")
# native host-thread contention measurement (links libgpuos.so)
PRODUCERS = os.path.join(HERE, "gpuos_producers")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc")
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-I" + INCLUDE, "-I" + CSRC]

SOURCES = ["gpuos_device.cu", "gpuos_host.cpp", "gpuos_nvrtc.cpp"]


def _run(cmd, log=None):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if log:
        with open(log, "w") as f:
            f.write(" ".join(cmd) + "\n" + r.stdout)
    if r.returncode != 0:
        sys.stderr.write(r.stdout)
        raise RuntimeError("build step failed: " + " ".join(cmd))
    return r.stdout


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def executor_regs(log_path=None) -> int:
    """Registers per thread of the executor kernel, from the ptxas report."""
    log_path = log_path or os.path.join(BUILD, "gpuos_device.ptxas.txt")
    txt = open(log_path).read()
    m = re.search(r"Function properties for gpuos_executor_kernel.*?Used (\d+) registers", txt, re.S)
    if not m:
        raise RuntimeError("executor register count not found in ptxas report")
    return int(m.group(1))


def build(force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, "gpuos_internal.h"), os.path.join(INCLUDE, "gpuos.h")]
    objs = []
    jobs = []
    for src in SOURCES:
        sp = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, src + ".o")
        objs.append(obj)
        if force or _stale(obj, [sp] + headers):
            cmd = [NVCC] + ARCH + COMMON + ["-Xcompiler", "-fPIC,-fvisibility=hidden", "-c", sp, "-o", obj]
            log = None
            if src.endswith(".cu"):
                cmd += ["-Xptxas", "-v"]
                log = os.path.join(BUILD, src.replace(".cu", ".ptxas.txt"))
            jobs.append((cmd, log))
    ext_src = os.path.join(CSRC, "gpuos_ext_ops.cu")
    dev_src = os.path.join(CSRC, "gpuos_device.cu")
    if force or _stale(EXEC_RDC, [dev_src] + headers):
        # every function of the relocatable build must fit the executor's
        # per-thread register budget (launch bounds: 384 threads, 1 block/SM)
        jobs.append(([NVCC] + ARCH + COMMON + ["-cubin", "-rdc=true", "-maxrregcount", "168", "-Xptxas", "-v",
                                               dev_src, "-o", EXEC_RDC + ".tmp"],
                     os.path.join(BUILD, "gpuos_exec_rdc.ptxas.txt")))
    with cf.ThreadPoolExecutor(max_workers=4) as ex:
        list(ex.map(lambda j: _run(*j), jobs))
    if os.path.exists(EXEC_RDC + ".tmp"):
        os.replace(EXEC_RDC + ".tmp", EXEC_RDC)
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + ".tmp"
        _run([NVCC] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs + ["-lpthread", "-ldl", "-lrt"])
        os.replace(tmp, LIB)
    # the native multi-producer measurement (C ABI only, pthreads)
    prod_src = os.path.join(CSRC, "gpuos_producers.cpp")
    if os.path.exists(prod_src) and (force or _stale(PRODUCERS, [prod_src, LIB, os.path.join(INCLUDE, "gpuos.h")])):
        cxx = shutil.which("g++") or "g++"
        _run([cxx, "-O2", "-std=c++17", "-I" + INCLUDE, prod_src, "-o", PRODUCERS + ".tmp", "-L" + HERE,
              "-lgpuos", "-Wl,-rpath,$ORIGIN", "-lpthread"])
        os.replace(PRODUCERS + ".tmp", PRODUCERS)
    # The example op module is a relocatable object (linked into the executor
    # at run time); it must not use more registers than the executor holds
    # per thread, so it is compiled with the executor's count as its cap.
    if os.path.exists(ext_src) and (force or _stale(EXT_CUBIN, [ext_src, LIB] + headers)):
        regs = min(executor_regs(), 168)
        tmp = EXT_CUBIN + ".tmp"
        log = os.path.join(BUILD, "gpuos_ext_ops.ptxas.txt")
        _run([NVCC] + ARCH + COMMON + ["-cubin", "-rdc=true", "-maxrregcount", str(regs), "-Xptxas", "-v",
                                      ext_src, "-o", tmp], log)
        os.replace(tmp, EXT_CUBIN)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
