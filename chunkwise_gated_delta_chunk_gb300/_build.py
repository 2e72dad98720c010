"""Build ``libdnchunk.so`` in-tree with nvcc for sm_103a (GB300).

Each ``csrc/*.cu`` translation unit compiles in parallel into
``_build/*.o``; the objects link into one shared library next to this file.
The CUDA runtime is linked statically, so the library needs only the driver.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdnchunk.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I" + INCLUDE, "-I" + CSRC] + ARCH


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdnchunk.so")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(
        os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src: str, extra: list[str]) -> str:
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc()] + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
    if r.stderr.strip() and os.environ.get("DN_BUILD_VERBOSE"):
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, extra: list[str] | None = None) -> str:
    """Compile every kernel for sm_103a and link ``libdnchunk.so``."""
    if not force and not extra and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    extra = list(extra or [])
    with cf.ThreadPoolExecutor(max_workers=max(1, len(sources()))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), sources()))
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, LIB)
    return LIB


# Translation units that change in the failure-path test build.
STALL_SOURCES = ("dn_api.cu", "dn_tc.cu", "dn_tc_wide.cu", "dn_wy.cu")
STALL_LIB = os.path.join(BUILD, "stall", "libdnchunk_stall.so")


def build_stall_variant() -> str:
    """Build the failure-path test variant of the library (never the product
    library): dn_api.cu, dn_tc.cu, dn_tc_wide.cu and dn_wy.cu compiled with -DDN_TEST_STALL
    (2 ms wait limit, the dn_test_stall_next hook), linked with the other
    objects of the regular build, into ``_build/stall/libdnchunk_stall.so``."""
    build()
    out = os.path.dirname(STALL_LIB)
    os.makedirs(out, exist_ok=True)
    stall_srcs = [os.path.join(CSRC, f) for f in STALL_SOURCES]

    def one(src: str) -> str:
        obj = os.path.join(out, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc()] + NVCC_FLAGS + ["-DDN_TEST_STALL", "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s" % (src, r.stderr))
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(stall_srcs)) as ex:
        objs = list(ex.map(one, stall_srcs))
    objs += [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in sources()
             if os.path.basename(s) not in STALL_SOURCES]
    tmp = STALL_LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s" % r.stderr)
    os.replace(tmp, STALL_LIB)
    return STALL_LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
