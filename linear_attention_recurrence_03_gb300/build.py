"""Builds ``libgdn.so`` -- the CUDA library behind include/gdn.h -- in the package
directory with nvcc, for sm_103a only. Each translation unit compiles in parallel;
the link is one ``nvcc -shared`` step. Objects go to ``_build/`` beside this file."""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgdn.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
    "-I", INCLUDE, "-I", CSRC,
]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _inputs():
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = srcs + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
    deps += glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]
    return srcs, deps


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    _, deps = _inputs()
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False,
          defines=(), lib_path: str | None = None) -> str:
    """Compile and link the library if any source is newer than it. Returns its path.

    ``defines`` (e.g. ``("GDN_TRACE",)``) and ``lib_path`` build a variant library
    elsewhere (profiling aids); the default build has neither."""
    out_lib = lib_path or LIB
    if not force and not defines and lib_path is None and up_to_date():
        return LIB
    build_dir = BUILD if not defines else BUILD + "_" + "_".join(d.lower() for d in defines)
    os.makedirs(build_dir, exist_ok=True)
    srcs, _ = _inputs()
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_v else []
    extra += [f"-D{d}" for d in defines]

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_v:
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = out_lib + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a",
                        *objs, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out_lib)
    return out_lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
