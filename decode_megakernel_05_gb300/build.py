"""Builds the CUDA library (libmk.so) in-tree for sm_103a.

Each .cu translation unit is compiled in parallel with
``nvcc -gencode arch=compute_103a,code=sm_103a -O3 -lineinfo -Xptxas -v`` and the
objects are linked into ``decode_megakernel_05_gb300/_build/libmk.so`` with the
CUDA runtime linked statically, so the library loads without any other CUDA
shared object.  The ptxas resource report (registers, spills, shared memory)
is kept in ``_build/ptxas.log``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libmk.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
SOURCES = ["mk_api.cu", "mk_aux.cu", "mk_perop.cu", "mk_prefill.cu", "mk_noalloc.cu"]
# (head_dim, query heads per KV group, hidden / 256) of the fused kernel, one
# object each; keep in sync with MK_VARIANTS in csrc/mk_api.cu
VARIANTS = [(64, 2, 1), (64, 4, 2), (64, 4, 4), (64, 4, 8), (64, 4, 16), (128, 4, 4), (128, 4, 8), (128, 4, 16)]
# long-context builds (attention on the tensor cores), launched for steps whose context gives
# each CTA at least MK_ATTN_TC_MIN_PER_CTA positions; keep in sync with MK_LC_VARIANTS in
# csrc/mk_api.cu
LC_VARIANTS = [(64, 4, 2), (64, 4, 8), (128, 4, 4), (128, 4, 16)]
# weight-only INT8 builds (-DMK_WB_V=1) of the standard and long-context kernels; keep in sync
# with MK_Q8_VARIANTS and MK_Q8_LC_VARIANTS in csrc/mk_api.cu
Q8_VARIANTS = [(64, 2, 1), (64, 4, 8), (128, 4, 16)]
Q8_LC_VARIANTS = [(64, 4, 8)]
# weight-only INT4 builds (-DMK_WB_V=0); keep in sync with MK_Q4_VARIANTS and MK_Q4_LC_VARIANTS
Q4_VARIANTS = [(64, 2, 1), (64, 4, 8), (128, 4, 16)]
Q4_LC_VARIANTS = [(64, 4, 8), (128, 4, 16)]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def _deps():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(INCLUDE, "mk.h"))
    deps.append(os.path.abspath(__file__))
    return deps


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
                    "-I", INCLUDE, "-I", CSRC]
    jobs = [(src, os.path.join(BUILD, src.replace(".cu", ".o")), []) for src in SOURCES]
    kernels = ([v + (0, 2) for v in VARIANTS] + [v + (1, 2) for v in LC_VARIANTS] +
               [v + (0, 1) for v in Q8_VARIANTS] + [v + (1, 1) for v in Q8_LC_VARIANTS] +
               [v + (0, 0) for v in Q4_VARIANTS] + [v + (1, 0) for v in Q4_LC_VARIANTS])
    for hd, g, mh, lc, wb in kernels:
        for tr in (False, True):   # each without and with the segment trace compiled in
            sfx = ("_lc" if lc else "") + {2: "", 1: "_q8", 0: "_q4"}[wb] + ("_trace" if tr else "")
            jobs.append(("mk_kernel.cu", os.path.join(BUILD, f"mk_kernel_{hd}_{g}_{mh}{sfx}.o"),
                         [f"-DMK_HD_V={hd}", f"-DMK_G_V={g}", f"-DMK_MH_V={mh}", f"-DMK_LC_V={lc}",
                          f"-DMK_WB_V={wb}"] + ([] if tr else ["-DMK_NO_TRACE"])))

    def compile_one(job):
        src, obj, defs = job
        cmd = [cc, *flags, *defs, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src} {defs}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(min(len(jobs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, jobs))
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        for (obj, log), (src, _, defs) in zip(results, jobs):
            f.write(f"==== {src} {' '.join(defs)}\n{log}\n")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        print(open(os.path.join(BUILD, "ptxas.log")).read())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
