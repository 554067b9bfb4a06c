"""Build the CUDA library (``lib/libattn_gb300.so``) in-tree with nvcc.

Every ``csrc/*.cu`` file is compiled for sm_103a only, in parallel, and the
objects are linked into one shared library that exports the C ABI of
``include/attn_gb300.h``.  No torch, no cmake.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIB_DIR, "libattn_gb300.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC,-O2", "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [
        os.path.join(ROOT, "include", "attn_gb300.h")]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


# Debug variant: every shared-memory staging tile (dS for the dQ MMA, the fp32
# dQ partial before its bulk reduction, the dK / dV epilogue tiles) is filled
# with NaN by each writer just before its real data, so a consumer that reads
# the tile before the writes have landed produces non-finite output.
POISON_LIB = os.path.join(LIB_DIR, "libattn_gb300_poison.so")

# Debug variant: per-tile bounds checks that record ATTN_E_INTERNAL and skip
# the access instead of trapping, and attn_debug_inject_stall(), which makes
# one bounded wait of one block's MMA issuer run out so that the kernels' own
# unwind paths (abort flag, drains, ATTN_E_TIMEOUT) run on the GPU.
CHECKED_LIB = os.path.join(LIB_DIR, "libattn_gb300_checked.so")


def build(force: bool = False, verbose: bool = False, extra_flags=(), variant=None) -> str:
    """variant None: the library; "poison": the poisoned-staging debug build;
    "checked": the bounds-check / stall-injection debug build."""
    out_lib, build_dir = LIB, BUILD
    if variant == "poison":
        out_lib, build_dir = POISON_LIB, os.path.join(BUILD, "poison")
        extra_flags = tuple(extra_flags) + ("-DATTN_POISON_SMEM",)
    elif variant == "checked":
        out_lib, build_dir = CHECKED_LIB, os.path.join(BUILD, "checked")
        extra_flags = tuple(extra_flags) + ("-DATTN_DEBUG_CHECKS",)
    elif variant is not None:
        raise ValueError("unknown build variant %r" % (variant,))
    if not force and up_to_date(out_lib):
        return out_lib
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = out_lib + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, out_lib)
    return out_lib


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "-v" in sys.argv else []))
