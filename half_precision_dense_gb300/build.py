"""Build the CUDA library ``lib/libhgemm.so`` in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel into ``_build/``; the shared
library links the CUDA runtime statically. A unit is recompiled only when it
or a header it may include is newer than its object.
"""

from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libhgemm.so")

SOURCES = ["hgemm_api.cu", "hgemm_tc_bf16.cu", "hgemm_tc_f16.cu", "hgemm_tc_tf32.cu", "hgemm_tc_fp8.cu", "hgemm_tc_fp8bs.cu",
           "hgemm_aux.cu",
           "hgemm_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
          f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return path


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _extra_flags() -> list[str]:
    """Extra nvcc flags from HGEMM_NVCC_FLAGS (e.g. -DHG_TRACE for a build that
    records kernel timelines)."""
    return os.environ.get("HGEMM_NVCC_FLAGS", "").split()


def _flags_stamp() -> str:
    return os.path.join(BUILD_DIR, "flags.txt")


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    try:
        with open(_flags_stamp()) as f:
            if f.read() != " ".join(_extra_flags()):
                return True
    except OSError:
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in [src, __file__] + _headers())


def _compile(src_name: str, verbose: bool) -> tuple[str, str]:
    src = os.path.join(CSRC, src_name)
    obj = os.path.join(BUILD_DIR, src_name.replace(".cu", ".o"))
    if not _stale(obj, src):
        return obj, ""
    cmd = [nvcc(), *ARCH, *CFLAGS, *_extra_flags(), "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src_name}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose:
        print(r.stderr)
    return obj, r.stderr


def build(verbose: bool = False) -> str:
    """Compile (if needed) and link the library; returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    with open(_flags_stamp(), "w") as f:
        f.write(" ".join(_extra_flags()))
    objs = [o for o, _ in results]
    if not os.path.exists(LIB_PATH) or any(os.path.getmtime(o) > os.path.getmtime(LIB_PATH) for o in objs):
        tmp = LIB_PATH + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-cudart", "static", *objs, "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def ptxas_report() -> str:
    """The -Xptxas -v lines of the last compilation of each unit (rebuilds all)."""
    for s in SOURCES:
        o = os.path.join(BUILD_DIR, s.replace(".cu", ".o"))
        if os.path.exists(o):
            os.remove(o)
    os.makedirs(BUILD_DIR, exist_ok=True)
    out = []
    for s in SOURCES:
        _, log = _compile(s, False)
        out.append(f"== {s}\n{log}")
    return "\n".join(out)


if __name__ == "__main__":
    print(build(verbose=True))
