"""Build libgq.so in-tree with nvcc for sm_103a (GB300).

    python -m quantized_skinny_matmul_gb300._build [--force] [--verbose-ptxas] [--debug]

Each CUDA translation unit under csrc/ compiles in parallel to an object file;
nvcc then links them (with the static CUDA runtime) into
quantized_skinny_matmul_gb300/_lib/libgq.so.  No torch headers are involved, so
the library does not depend on the installed PyTorch version.

With --debug (build(debug=True)) the same sources compile with -DGQ_DEBUG into
_lib/libgq_debug.so: the kernels then check the indices they derive from their
arguments and record a failure in the device status word (gq_last_error returns
GQ_ERR_DEVICE_CHECK); nothing traps.  The binding loads it when GQ_LIBRARY names it.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
OBJ_DIR = os.path.join(OUT_DIR, "obj")
LIB_PATH = os.path.join(OUT_DIR, "libgq.so")
DEBUG_LIB_PATH = os.path.join(OUT_DIR, "libgq_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "gq.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


_ELF_MACHINE = {"x86_64": 62, "amd64": 62, "aarch64": 183, "arm64": 183}


def built_for_this_machine(path: str) -> bool:
    """Whether the ELF file at path targets this host's CPU (a copy built on another machine does not)."""
    want = _ELF_MACHINE.get(platform.machine().lower())
    try:
        with open(path, "rb") as f:
            head = f.read(20)
    except OSError:
        return False
    if len(head) < 20 or head[:4] != b"\x7fELF":
        return False
    return want is None or int.from_bytes(head[18:20], "little") == want


def up_to_date(path: str = LIB_PATH) -> bool:
    return (os.path.exists(path) and os.path.getmtime(path) >= _deps()
            and built_for_this_machine(path))


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None, debug: bool = False) -> str:
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    obj_dir = OBJ_DIR + ("_debug" if debug else "")
    if not force and up_to_date(lib_path):
        return lib_path
    os.makedirs(obj_dir, exist_ok=True)
    cc = nvcc()
    extra = (["-Xptxas", "-v"] if verbose_ptxas else []) + (["-DGQ_DEBUG"] if debug else [])

    def compile_one(src: str):
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, res

    srcs = _sources()
    objs = []
    failed = []
    with cf.ThreadPoolExecutor(max_workers=jobs or min(8, len(srcs))) as ex:
        for src, obj, res in ex.map(compile_one, srcs):
            if res.stdout or res.stderr:
                sys.stderr.write(res.stdout + res.stderr)
            if res.returncode != 0:
                failed.append(src)
            objs.append(obj)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(os.path.basename(f) for f in failed))
    tmp = lib_path + ".tmp"
    link = [cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs]
    res = subprocess.run(link, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError("link of " + os.path.basename(lib_path) + " failed")
    os.replace(tmp, lib_path)
    return lib_path


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    ap.add_argument("--debug", action="store_true", help="the GQ_DEBUG build (device-side bounds checks)")
    a = ap.parse_args()
    print(build(force=a.force, verbose_ptxas=a.verbose_ptxas, debug=a.debug))


if __name__ == "__main__":
    main()
