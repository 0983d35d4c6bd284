"""Builds libsgemv.so in-tree from csrc/*.cu with nvcc for sm_103a.

Each translation unit is compiled in parallel; the shared library links the
CUDA runtime statically so that it carries no dependency on the runtime
that the calling process (e.g. PyTorch) happens to load.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsgemv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-Wall", "--expt-relaxed-constexpr",
              "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"),
                 "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith(".cu"))


def _stamp(files: list[str] | None = None) -> str:
    """Hash of the sources (all of csrc, or the named csrc files), the public
    header and the compiler flags.  A record taken on one kernel (a profile's
    traffic) names that kernel's files, so edits elsewhere keep it valid."""
    h = hashlib.sha256()
    if files is None:
        deps = sources() + sorted(
            os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh"))
    else:
        deps = [os.path.join(CSRC, f) for f in files]
    deps.append(os.path.join(INCLUDE, "sgemv.h"))
    for p in deps:
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode() + b"\0" + f.read())
    # flags without the machine-specific include path
    h.update(" ".join(f for f in ARCH + NVCC_FLAGS if f != INCLUDE).encode())
    return h.hexdigest()


# Build variants: the product library, and the checked build (a debugging
# aid: the product kernels validate every decoded code and index).
VARIANTS = {None: ([], LIB, BUILD),
            "checked": (["-DSGEMV_CHECKED"], os.path.join(HERE, "libsgemv_checked.so"),
                        os.path.join(HERE, "_build_checked"))}


def build(force: bool = False, verbose: bool = False,
          extra: list[str] | None = None, variant: str | None = None) -> str:
    vflags, lib, build_dir = VARIANTS[variant]
    if variant is None:
        lib, build_dir = LIB, BUILD
    stamp_path = os.path.join(build_dir, "stamp")
    stamp = _stamp() + " ".join(vflags + (extra or []))
    if (not force and os.path.exists(lib) and os.path.exists(stamp_path)
            and open(stamp_path).read() == stamp):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    flags = ARCH + NVCC_FLAGS + vflags + (extra or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        cmd = [cc, "-c", src, "-o", obj] + flags
        if verbose:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static",
                                                      "-Xcompiler", "-fPIC"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                variant="checked" if "--checked" in sys.argv else None))
