"""In-tree build of libw4a8.so for sm_103a (GB300).

Each ``csrc/*.cu`` translation unit is compiled by its own nvcc process (in parallel) and the
objects are linked into ``int4_quantized_linear_gb300/libw4a8.so`` next to this file.  The CUDA
runtime is linked statically, so the library needs nothing at load time beyond the driver.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libw4a8.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden", "-Xptxas", "-v",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    return "nvcc"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + [os.path.join(ROOT, "include", "w4a8.h"), os.path.abspath(__file__)])


def _extra_flags():
    # W4A8_EXTRA_NVCC_FLAGS: extra compiler options for this build (e.g. -DW4A8_TRACE to compile in
    # the pipeline timestamps, or a tuning constant such as -DW4A8_L2_PREFETCH_FILLS=4)
    return os.environ.get("W4A8_EXTRA_NVCC_FLAGS", "").split()


def _flags_path():
    return LIB_PATH + ".flags"


def up_to_date(check_flags: bool = True) -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    if not all(os.path.getmtime(d) <= t for d in _deps()):
        return False
    if not check_flags:
        return True
    # a library built with other extra options (a diagnostic build, say) is rebuilt
    try:
        with open(_flags_path()) as f:
            return f.read() == " ".join(_extra_flags())
    except OSError:
        return not _extra_flags()


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()

    extra = _extra_flags()

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + ARCH + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, _sources()))
    failed = [(s, r) for s, _, r in results if r.returncode != 0]
    for s, _, r in results:
        if verbose or r.returncode != 0:
            sys.stderr.write(f"--- {os.path.basename(s)}\n{r.stdout}{r.stderr}")
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(os.path.basename(s) for s, _ in failed))
    tmp = LIB_PATH + ".tmp%d" % os.getpid()
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + [o for _, o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB_PATH)
    with open(_flags_path(), "w") as f:
        f.write(" ".join(extra))
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
