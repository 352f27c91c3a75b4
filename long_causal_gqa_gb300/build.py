"""Build the sm_103a CUDA library libh3gqa.so in-tree with nvcc.

One translation unit, one -gencode (compute_103a -> sm_103a). The result
sits next to this file and is what the Python binding loads.
"""
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
SOURCES = [os.path.join(CSRC, "h3gqa_api.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in ("fwd_kernel.cuh", "ptx_sm103a.cuh", "prep_kernel.cuh")] + [
    os.path.join(INCLUDE, "h3gqa.h")]
LIB = os.path.join(HERE, "libh3gqa.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    p = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(p):
        return p
    raise RuntimeError("nvcc not found (CUDA 13 toolkit required)")


def build(force: bool = False, out: str = LIB, defines=(), verbose: bool = False) -> str:
    """Compile the library to `out` unless it is newer than every source."""
    if (not force and not defines and os.path.exists(out)
            and os.path.getmtime(out) >= max(os.path.getmtime(d) for d in DEPENDS)):
        return out
    tmp = out + ".tmp.%d" % os.getpid()
    cmd = [nvcc_path(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17",
           "-Xcompiler", "-fPIC", "-shared", "-I", INCLUDE,
           *["-D%s" % d for d in defines], "-o", tmp, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
