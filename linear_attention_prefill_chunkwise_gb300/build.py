"""Compile the sm_103a C-ABI library ``libla_prefill.so`` in-tree.

Six translation units (prefill; speculative-decoding ops; segmented prefill; its variant
with a built-in scratch buffer; backward pass; D = 256 prefill), one ``-gencode`` (sm_103a),
static CUDA runtime, no
link-time dependency on the driver library (the tensor-map encoder is fetched
through the runtime's driver entry-point query), so the library loads on a
machine without a GPU.
"""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libla_prefill.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
INCLUDE_DIR = os.path.join(os.path.dirname(HERE), "include")

SOURCES = ["la_prefill_api.cu", "la_decode_api.cu", "la_segment_api.cu", "la_segment_static_api.cu",
           "la_backward_api.cu", "la_d256_api.cu"]
DEPENDS = ["la_prefill_api.cu", "la_prefill_kernel.cuh", "sm103_ptx.cuh", "la_decode_api.cu", "la_decode_kernels.cuh",
           "la_segment_api.cu", "la_segment_kernels.cuh", "la_segment_static_api.cu", "la_host_common.h",
           "la_backward_api.cu", "la_verify_kernel.cuh", "la_prefill_internal.h", "la_d256_api.cu"]
HEADERS = ["la_prefill.h", "la_decode.h", "la_segment.h", "la_backward.h", "la_d256.h"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    cand = shutil.which("nvcc")
    if cand:
        return cand
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    return os.path.join(cuda_home, "bin", "nvcc")


def _stale(path: str) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    deps = [os.path.join(CSRC, d) for d in DEPENDS] + [os.path.join(INCLUDE_DIR, h) for h in HEADERS]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, wait_limit_ns: int = 0) -> str:
    """Build the library if any source is newer than it; return its path.

    wait_limit_ns > 0 builds the prefill entry point alone, as a separate file, with that
    limit on every pipeline wait instead of one second: ordinary waits then exceed it, so the
    kernels' timeout exit can be exercised on a healthy input."""
    if wait_limit_ns:
        out = os.path.join(BUILD_DIR, f"libla_prefill_wait{int(wait_limit_ns)}ns.so")
        sources = ["la_prefill_api.cu"]
    else:
        out = LIB_PATH
        sources = SOURCES
    if not force and not _stale(out):
        return out
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc_path(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           "-cudart", "static", "-I", INCLUDE_DIR, "-o", tmp] + [os.path.join(CSRC, s) for s in sources]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    if wait_limit_ns:
        cmd.insert(1, f"-DLA_WAIT_LIMIT_NS={int(wait_limit_ns)}ull")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    if verbose:
        print(res.stdout + res.stderr)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True, verbose=True))
