"""Build the CUDA library in-tree: sparse_attention_indexer_sm_gb300/_build/libtopk_transform.so.

Every object is compiled for sm_103a only, all of them in parallel, then linked
against the shared CUDA runtime (so that the process keeps a single runtime
together with PyTorch). Run ``python -m sparse_attention_indexer_sm_gb300.build``.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libtopk_transform.so")

SOURCES = ("topk_select.cu", "topk_api.cu")
# The kernel source is compiled once per (CTA size, form) and once per CTA size for
# the dispatch by form: ten objects that build in parallel.
KERNEL_OBJECTS = [(f"topk_select_{cta}_{form}", ["-DTOPK_CTA_THREADS=%d" % cta, "-DTOPK_FORM=%d" % form])
                  for cta in (512, 256) for form in range(4)]
KERNEL_OBJECTS += [(f"topk_select_{cta}", ["-DTOPK_CTA_THREADS=%d" % cta]) for cta in (512, 256)]
HEADERS = (os.path.join(CSRC, "topk_select.cuh"), os.path.join(INCLUDE, "topk_transform.h"))
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + list(HEADERS) + [__file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link if any source is newer than the library; return its path."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    exe = nvcc()
    procs, objs = [], []
    units = [(name, defs, "topk_select.cu") for name, defs in KERNEL_OBJECTS]
    units.append(("topk_api", [], "topk_api.cu"))
    for name, defs, src in units:
        obj = os.path.join(BUILD_DIR, name + ".o")
        cmd = [exe, *NVCC_FLAGS, *defs, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                            text=True)))
        objs.append(obj)
    for cmd, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed ({' '.join(cmd)}):\n{out}")
        if verbose and out:
            print(out, file=sys.stderr)
    tmp = LIB_PATH + f".{os.getpid()}.tmp"
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(exe))), "lib64")
    link = [exe, *ARCH, "-shared", "-cudart", "shared", "-Xlinker", "-rpath," + cuda_lib,
            "-o", tmp, *objs]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed ({' '.join(link)}):\n{r.stdout}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
