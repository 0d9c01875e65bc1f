"""Build step of the rope3d library: compiles the CUDA kernels for sm_103a and
the host C ABI, and links them into ``_build/librope3d.so`` inside this
package (in-tree, so the same file is what the tests and the benchmark load).

    python -m rope_rope3d_apply_gb300.build
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
DEBUG_BUILD = os.path.join(HERE, "_build_debug")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "librope3d.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = [
    os.path.join(CSRC, "rope3d_kernels.cu"),
    os.path.join(CSRC, "rope3d_noalloc.cu"),
    os.path.join(CSRC, "rope3d_patchify.cu"),
    os.path.join(CSRC, "rope3d_neox.cu"),
    os.path.join(CSRC, "rope3d_na3d.cu"),
    os.path.join(CSRC, "rope3d_api.cpp"),
    os.path.join(CSRC, "rope3d_internal.h"),
    os.path.join(INCLUDE, "rope3d.h"),
]


def _cuda_home() -> str:
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _nvcc() -> str:
    return os.path.join(_cuda_home(), "bin", "nvcc")


def commands(out_dir: str = BUILD, extra_nvcc: list[str] | None = None,
             debug_bounds: bool = False):
    """Compile and link commands. debug_bounds: every kernel checks each index
    it computes before the access (see rope3d_debug_bounds in rope3d.h)."""
    cuda = _cuda_home()
    dbg = ["-DROPE3D_DEBUG_BOUNDS=1"] if debug_bounds else []
    kern_o = os.path.join(out_dir, "rope3d_kernels.o")
    api_o = os.path.join(out_dir, "rope3d_api.o")
    nvcc_compile = [
        _nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-fmad=false", *dbg,
        "-Xcompiler", "-fPIC,-ffp-contract=off", "-Xptxas", "-v",
        *(extra_nvcc or []),
        "-c", os.path.join(CSRC, "rope3d_kernels.cu"), "-o", kern_o,
    ]
    noalloc_o = os.path.join(out_dir, "rope3d_noalloc.o")
    nvcc_noalloc = [
        _nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-fmad=false", *dbg,
        "-Xcompiler", "-fPIC,-ffp-contract=off",
        "-c", os.path.join(CSRC, "rope3d_noalloc.cu"), "-o", noalloc_o,
    ]
    patch_o = os.path.join(out_dir, "rope3d_patchify.o")
    nvcc_patch = [
        _nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", *dbg, "-Xcompiler", "-fPIC",
        "-Xptxas", "-v", "-c", os.path.join(CSRC, "rope3d_patchify.cu"), "-o", patch_o,
    ]
    neox_o = os.path.join(out_dir, "rope3d_neox.o")
    nvcc_neox = [
        _nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-fmad=false", *dbg,
        "-Xcompiler", "-fPIC,-ffp-contract=off", "-Xptxas", "-v",
        "-c", os.path.join(CSRC, "rope3d_neox.cu"), "-o", neox_o,
    ]
    na_o = os.path.join(out_dir, "rope3d_na3d.o")
    nvcc_na = [
        _nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-fmad=false", *dbg,
        "-Xcompiler", "-fPIC,-ffp-contract=off", "-Xptxas", "-v", *(extra_nvcc or []),
        "-c", os.path.join(CSRC, "rope3d_na3d.cu"), "-o", na_o,
    ]
    gxx_compile = [
        "g++", "-std=c++17", "-O2", "-fPIC", "-ffp-contract=off", "-fno-fast-math", *dbg,
        "-pthread", "-Wall", "-Wno-unused-function", f"-I{cuda}/include",
        "-c", os.path.join(CSRC, "rope3d_api.cpp"), "-o", api_o,
    ]
    link = [_nvcc(), *ARCH, "-shared", kern_o, api_o, noalloc_o, patch_o, neox_o, na_o,
            "-o", os.path.join(out_dir, "librope3d.so"), "-Xcompiler", "-pthread"]
    return [nvcc_compile, gxx_compile, nvcc_noalloc, nvcc_patch, nvcc_neox, nvcc_na], link


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(s) <= t for s in SOURCES)


def build(force: bool = False, verbose: bool = False, out_dir: str | None = None,
          extra_nvcc: list[str] | None = None, debug_bounds: bool = False) -> str:
    """Compile and link; returns the library path. The compiles run in parallel.
    debug_bounds builds the bounds-checking variant (into _build_debug unless
    out_dir says otherwise)."""
    if out_dir is None:
        out_dir = DEBUG_BUILD if debug_bounds else BUILD
    lib = os.path.join(out_dir, "librope3d.so")
    if not force and out_dir in (BUILD, DEBUG_BUILD) and up_to_date(lib):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    compiles, link = commands(out_dir, extra_nvcc, debug_bounds)
    procs = [subprocess.Popen(c, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
             for c in compiles]
    logs = []
    for c, p in zip(compiles, procs):
        out, _ = p.communicate()
        logs.append(out)
        if p.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(c)}\n{out}")
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(link)}\n{r.stdout}")
    with open(os.path.join(out_dir, "ptxas.log"), "w") as f:
        f.write("\n".join(logs))
    if verbose:
        print("\n".join(logs))
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
