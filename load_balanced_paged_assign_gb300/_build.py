"""Builds libhpcdecode.so in the package directory (nvcc, sm_103a only).

The translation units are compiled in parallel and linked with the CUDA
runtime statically, so the library needs nothing at run time beyond the
NVIDIA driver.  Rebuilds only when a source or header is newer than the
library.
"""

from __future__ import annotations

import glob
import os
import shutil
import subprocess
import tempfile
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB_PATH = os.path.join(HERE, "libhpcdecode.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libhpcdecode.so")


def sources() -> list:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, defines=(), out: str | None = None) -> str:
    """Compile the library (to `out`, default the package's libhpcdecode.so).

    `defines` are extra -D settings, e.g. the pipeline shape of the attention
    kernels (HPC_BF16_STAGES, HPC_BF16_TPS, HPC_FP8_STAGES, HPC_FP8_TPS)."""
    target = out or LIB_PATH
    if not force and not defines and out is None and not is_stale():
        return LIB_PATH
    nvcc = _nvcc()
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                    "--expt-relaxed-constexpr"] + [f"-D{d}" for d in defines]
    with tempfile.TemporaryDirectory(prefix="hpcdecode_build_") as tmp:
        def compile_one(src):
            obj = os.path.join(tmp, os.path.basename(src) + ".o")
            cmd = [nvcc, *flags, "-c", src, "-o", obj]
            res = subprocess.run(cmd, capture_output=True, text=True)
            if res.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{res.stderr}")
            if verbose and res.stderr:
                print(res.stderr)
            return obj

        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as pool:
            objs = list(pool.map(compile_one, sources()))
        out_tmp = os.path.join(tmp, "libhpcdecode.so")
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", out_tmp, *objs]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stderr}")
        staged = target + f".{os.getpid()}.tmp"
        shutil.copyfile(out_tmp, staged)
        os.replace(staged, target)
    return target


if __name__ == "__main__":
    import argparse
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--define", "-D", action="append", default=[])
    ap.add_argument("--out", default=None)
    a = ap.parse_args()
    print(build(force=True, verbose=True, defines=a.define, out=a.out))
