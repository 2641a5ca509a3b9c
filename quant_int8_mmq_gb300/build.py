"""Build libmmq_gb300.so in-tree: nvcc for sm_103a, one object per .cu, compiled in parallel."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libmmq_gb300.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)
SOURCES = ["api.cu", "prepass.cu", "pack.cu", "ggml.cu", "gemm.cu", "gemm_sb.cu", "gemm_small.cu", "gemm_ft.cu", "route.cu"]
PEAKS_SRC = "peaks.cu"
PEAKS_EXE = os.path.join(BUILD_DIR, "mmq_peaks")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH") or "/usr/local/cuda"
    cand = os.path.join(home, "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found: set CUDA_HOME")
    return found


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f != PEAKS_SRC]
    files += [os.path.join(INCLUDE, "mmq.h"), __file__]
    return [f for f in files if os.path.isfile(f)]


def _up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def compile_flags(ptxas_verbose: bool = False):
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                    "--expt-relaxed-constexpr"]
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]
    return flags


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    if not force and not ptxas_verbose and _up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = nvcc_path()
    flags = compile_flags(ptxas_verbose)

    def one(src):
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(one, SOURCES))
    if verbose or ptxas_verbose:
        for _, log in results:
            if log.strip():
                sys.stderr.write(log)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def build_peaks() -> str:
    """The throughput-probe program (roofline denominators), built on demand."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    src = os.path.join(CSRC, PEAKS_SRC)
    if os.path.exists(PEAKS_EXE) and os.path.getmtime(PEAKS_EXE) >= os.path.getmtime(src):
        return PEAKS_EXE
    cmd = [nvcc_path()] + compile_flags() + [src, "-o", PEAKS_EXE]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {PEAKS_SRC}:\n{r.stdout}\n{r.stderr}")
    return PEAKS_EXE


if __name__ == "__main__":
    build(force=True, verbose=True, ptxas_verbose="-v" in sys.argv)
    print(LIB_PATH)
