"""Build libattn.so in-tree with nvcc for sm_103a.

Each CUDA source compiles in its own nvcc process (in parallel), then one
link step produces ``attention_attn_prefill_gb300/libattn.so``.  A stamp over
the sources, headers, flags and host architecture skips the work when nothing
changed.  No cmake, no torch extension machinery.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import platform
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libattn.so")

SOURCES = ("api.cu", "prefill.cu", "prefill_cta2.cu", "prefill_host.cu", "decode.cu", "decode_noalloc.cu",
           "merge_emulated.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE,
                     "--expt-relaxed-constexpr"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattn.so")


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "attn.h"))
    return files


def _stamp(extra: list[str]) -> str:
    h = hashlib.sha256()
    for f in _inputs():
        h.update(f.encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(NVCC_FLAGS + extra).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          variant: str | None = None) -> str:
    """Compile and link libattn.so; returns its path.

    variant: a named build with extra_flags (for example a test-only variant), linked to
    _build/<variant>/libattn_<variant>.so instead of the package's libattn.so.
    """
    extra = list(extra_flags or [])
    build_dir = BUILD_DIR if variant is None else os.path.join(BUILD_DIR, variant)
    lib_path = LIB_PATH if variant is None else os.path.join(build_dir, f"libattn_{variant}.so")
    os.makedirs(build_dir, exist_ok=True)
    stamp_file = os.path.join(build_dir, "stamp")
    stamp = _stamp(extra)
    if not force and os.path.exists(lib_path) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read().strip() == stamp:
                return lib_path
    nvcc = nvcc_path()
    objs = []
    cmds = []
    for src in SOURCES:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmds.append([nvcc] + NVCC_FLAGS + extra + ["-c", os.path.join(CSRC, src), "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            print(" ".join(cmd))
            print(r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError(f"nvcc failed on {cmd[-3]}")
        return r

    with cf.ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        list(ex.map(run, cmds))
    tmp = lib_path + ".tmp"
    run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs)
    os.replace(tmp, lib_path)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return lib_path


if __name__ == "__main__":
    print(build(force=True, verbose=True))
