"""Build the CUDA libraries in-tree with nvcc (sm_103a only).

    libattn_fwd.so        the attention forward pass (C ABI: include/attn_fwd.h)
    libattn_fwd_trace.so  the same with the kernel's timeline recorded (-DATTN_TRACE; include/attn_fwd_trace.h)
    libattn_bwd.so        its backward (C ABI: include/attn_bwd.h)
    libattn_bwd_trace.so  the same with the backward kernels' timeline recorded (-DATTN_TRACE; include/attn_bwd_trace.h)
    libattn_probe.so      primitive checks of their building blocks (include/attn_fwd_probe.h)

The translation units compile in parallel; a library is rebuilt only when a
source or header is newer than it.  Usage: ``python -m attention_forward_06_gb300.build``.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "--use_fast_math", "-shared", "-Xcompiler", "-fPIC",
    "-cudart", "shared", "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC,
]

LIBS = {  # name -> (source, extra nvcc flags)
    "attn_fwd": (os.path.join(CSRC, "attn_fwd.cu"), []),
    "attn_fwd_trace": (os.path.join(CSRC, "attn_fwd.cu"), ["-DATTN_TRACE"]),
    "attn_bwd": (os.path.join(CSRC, "attn_bwd.cu"), []),
    "attn_bwd_trace": (os.path.join(CSRC, "attn_bwd.cu"), ["-DATTN_TRACE"]),
    "attn_probe": (os.path.join(CSRC, "probe.cu"), []),
}


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the attention library")
    return path


def lib_path(name: str) -> str:
    return os.path.join(BUILD_DIR, f"lib{name}.so")


def _deps() -> list[str]:
    return glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(name: str) -> bool:
    out = lib_path(name)
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in _deps())


def _compile(name: str, src: str, extra: list[str]) -> tuple[str, str]:
    out = lib_path(name)
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc()] + NVCC_FLAGS + extra + [src, "-o", tmp]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    log = proc.stdout + proc.stderr
    with open(os.path.join(BUILD_DIR, f"{name}.ptxas.log"), "w") as f:
        f.write(" ".join(cmd) + "\n" + log)
    if proc.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{log}")
    os.replace(tmp, out)
    return out, log


def build(force: bool = False, verbose: bool = False) -> dict[str, str]:
    """Compile every stale library; return {name: path}."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    todo = {n: s for n, s in LIBS.items() if force or _stale(n)}
    if todo:
        with ThreadPoolExecutor(max_workers=len(todo)) as ex:
            futs = {n: ex.submit(_compile, n, src, extra) for n, (src, extra) in todo.items()}
            for n, f in futs.items():
                _, log = f.result()
                if verbose:
                    sys.stdout.write(log)
    return {n: lib_path(n) for n in LIBS}


if __name__ == "__main__":
    for name, path in build(force="--force" in sys.argv, verbose=True).items():
        print(name, path)
