"""Build libdd.so in-tree for sm_103a (GB300) with nvcc.

Each translation unit is compiled in parallel, then linked into one shared
library next to this file.  Usage: ``python -m sparse_kv_prefetch_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(HERE, "libdd.so")
BUILD_DIR = os.path.join(ROOT, "_build")

SOURCES = ["api.cu", "score.cu", "topk.cu", "gather.cu", "attn.cu", "correct.cu", "noalloc.cu",
           "landmark.cu", "debug.cu", "hoststore.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src: str, extra: list[str], bdir: str = BUILD_DIR) -> str:
    obj = os.path.join(bdir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def build(verbose_ptxas: bool = False, out: str = OUT, defines=()) -> str:
    """Compile and link libdd.so into `out`.  `defines` are extra -D macros
    (compile-time geometry of the kernels, e.g. "DD_GATHER_STAGES=4"); a build
    with defines goes to its own object folder."""
    bdir = BUILD_DIR if not defines else os.path.join(
        BUILD_DIR, "_".join(d.replace("=", "-") for d in defines))
    os.makedirs(bdir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    extra += [f"-D{d}" for d in defines]
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, bdir), SOURCES))
    tmp = out + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", "-rpath=/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out



def is_stale(out: str = OUT) -> bool:
    """True if libdd.so is missing or older than any source or header."""
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + \
        [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return any(os.path.getmtime(p) > t for p in deps)


def ensure_built() -> str:
    return build() if is_stale() else OUT


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv))
