"""Build libnvfp4.so (the C-ABI library) for sm_103a with nvcc.

Each translation unit in csrc/ is compiled in parallel, then linked into
``libnvfp4_<machine>.so`` next to this file (the library is machine specific:
the build host and the GB300 host differ in CPU architecture).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build", platform.machine())
SOURCES = ["api.cu", "kernels_amax.cu", "kernels_quantize.cu", "kernels_misc.cu",
           "kernels_gemm.cu", "kernels_rht.cu"]
HEADERS = ["device_common.cuh", "internal.h", "tile_pipeline.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--fmad=false", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-Xptxas", "-warn-spills", "-I", INCLUDE]


def library_path() -> str:
    return os.path.join(HERE, f"libnvfp4_{platform.machine()}.so")


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, extra) -> str:
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    deps = [os.path.join(CSRC, src), os.path.join(INCLUDE, "nvfp4.h")]
    deps += [os.path.join(CSRC, h) for h in HEADERS]
    if _stale(obj, deps) or extra:
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, extra=()) -> str:
    """Compile (if needed) and return the path of the shared library."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = list(extra)
    if force:
        for f in os.listdir(BUILD_DIR):
            os.unlink(os.path.join(BUILD_DIR, f))
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    out = library_path()
    if _stale(out, objs) or extra:
        fd, tmp = tempfile.mkstemp(suffix=".so", dir=HERE)
        os.close(fd)
        try:
            cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl",
                   "-lpthread", "-lrt"]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
            os.replace(tmp, out)
        finally:
            if os.path.exists(tmp):
                os.unlink(tmp)
    return out


if __name__ == "__main__":
    print(build(force=True))
