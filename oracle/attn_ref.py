"""fp64 CPU oracle for the exact attention forward pass -- Python side.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code with
the CUDA library and never imports it; the two meet only in the seeded inputs.

The arithmetic lives in ``attn_ref.c`` (plain C, fp64, OpenMP over rows): the
plain definition of softmax attention with its closed-form log-sum-exp normaliser
(page "AdaSplash-2: Faster Differentiable Sparse Attention", technical summary
section 1).  This wrapper only builds the C file, marshals numpy arrays and
returns fp64 results.

Inputs are raw bf16 bit patterns (``numpy.uint16``) in the layouts
``q [B,Hq,Sq,D]``, ``k, v [B,Hkv,Sk,D]``; ``causal`` is 0 (none), 1 (bottom-right:
key j allowed for row i iff ``j <= i + Sk - Sq``) or 2 (top-left: ``j <= i``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libattn_ref.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``attn_ref.c`` into ``_build/libattn_ref.so`` (gcc, OpenMP) and return its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-fopenmp", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # ATTN_REF_LIB names another build of attn_ref.c to load instead: the mutation test
            # (tests/test_oracle_mutants.py) runs the pin suites, in a child process, against copies of the
            # oracle with one planted mistake each, and requires every copy to fail a pin.
            override = os.environ.get("ATTN_REF_LIB")
            lib = ctypes.CDLL(override if override else build())
            u16p = ctypes.POINTER(ctypes.c_uint16)
            f64p = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_int64)
            lib.attn_ref_fwd.restype = ctypes.c_int
            lib.attn_ref_fwd.argtypes = [u16p, u16p, u16p, f64p, f64p] + [ctypes.c_int] * 7 + [
                ctypes.c_float, i64p, ctypes.c_int64]
            lib.attn_ref_fwd_masked.restype = ctypes.c_int
            lib.attn_ref_fwd_masked.argtypes = [u16p, u16p, u16p, f64p, f64p] + [ctypes.c_int] * 7 + [
                ctypes.c_float, ctypes.POINTER(ctypes.c_uint32)] + [ctypes.c_int] * 3 + [i64p, ctypes.c_int64]
            lib.attn_ref_bwd.restype = ctypes.c_int
            lib.attn_ref_bwd.argtypes = [u16p, u16p, u16p, u16p, f64p, f64p, f64p] + [ctypes.c_int] * 7 + [
                ctypes.c_float]
            lib.attn_ref_probs.restype = ctypes.c_int
            lib.attn_ref_probs.argtypes = [u16p, u16p, u16p, f64p, f64p, f64p] + [ctypes.c_int] * 4 + [
                ctypes.c_float]
            lib.attn_ref_num_threads.restype = ctypes.c_int
            lib.attn_ref_num_threads.argtypes = []
            _lib = lib
    return _lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"oracle inputs are bf16 bit patterns (uint16), got {a.dtype}")
    return a


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def num_threads() -> int:
    """Threads the oracle's OpenMP loop runs on."""
    return int(_load().attn_ref_num_threads())


def attention(q, k, v, causal: int, scale: float, rows=None, block_mask=None, block=(128, 128)):
    """Exact attention forward in fp64.

    Returns ``(o, lse)``.  With ``rows=None``: ``o [B,Hq,Sq,D]``, ``lse [B,Hq,Sq]``.
    With ``rows`` (flat ids ``(b*Hq + h)*Sq + i``): ``o [len(rows), D]``, ``lse [len(rows)]``.
    ``scale`` is rounded to fp32 first: the oracle uses the value the GPU receives.
    ``block_mask`` (optional): uint32 ``[B, 1 or Hq, ceil(Sq/bq), ceil(ceil(Sk/bk)/32)]``, bit ``kb % 32``
    of word ``kb // 32`` marking key block ``kb`` visible to a query block (``block = (bq, bk)``);
    it restricts the keys on top of ``causal`` (page "AdaSplash-2", technical summary section 2).
    """
    q, k, v = _u16(q), _u16(k), _u16(v)
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be 4-d [B, H, S, D]")
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    if k.shape != v.shape or Bk != B or Dk != D:
        raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape}")
    if rows is None:
        o = np.empty((B, Hq, Sq, D), np.float64)
        lse = np.empty((B, Hq, Sq), np.float64)
        rows_arr, nrows = None, 0
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.size
        o = np.empty((nrows, D), np.float64)
        lse = np.empty((nrows,), np.float64)
    rows_ptr = _ptr(rows_arr, ctypes.c_int64) if rows_arr is not None else None
    if block_mask is None:
        rc = _load().attn_ref_fwd(
            _ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
            _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
            B, Hq, Hkv, Sq, Sk, D, int(causal), float(np.float32(scale)), rows_ptr, nrows)
    else:
        bq, bk = block
        mask = np.ascontiguousarray(block_mask, dtype=np.uint32)
        words = (-(-Sk // bk) + 31) // 32
        if mask.ndim != 4 or mask.shape[0] != B or mask.shape[1] not in (1, Hq) or \
                mask.shape[2] != -(-Sq // bq) or mask.shape[3] != words:
            raise ValueError(f"block mask shape {mask.shape} does not fit B={B} Hq={Hq} Sq={Sq} Sk={Sk}")
        rc = _load().attn_ref_fwd_masked(
            _ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
            _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
            B, Hq, Hkv, Sq, Sk, D, int(causal), float(np.float32(scale)),
            _ptr(mask, ctypes.c_uint32), int(mask.shape[1]), int(bq), int(bk), rows_ptr, nrows)
    if rc != 0:
        raise ValueError(f"attn_ref_fwd failed with status {rc}")
    return o, lse


def probabilities(q, k, v, causal: int, scale: float):
    """One (b, h) slice: ``q [Sq,D]``, ``k, v [Sk,D]`` -> ``(p [Sq,Sk], o [Sq,D], lse [Sq])``."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    Sq, D = q.shape
    Sk = k.shape[0]
    p = np.empty((Sq, Sk), np.float64)
    o = np.empty((Sq, D), np.float64)
    lse = np.empty((Sq,), np.float64)
    rc = _load().attn_ref_probs(
        _ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
        _ptr(p, ctypes.c_double), _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
        Sq, Sk, D, int(causal), float(np.float32(scale)))
    if rc != 0:
        raise ValueError(f"attn_ref_probs failed with status {rc}")
    return p, o, lse


def backward(q, k, v, dout, causal: int, scale: float):
    """Gradients of the forward's O with respect to q, k, v for the upstream gradient ``dout`` (fp64).

    ``q, dout [B,Hq,Sq,D]``, ``k, v [B,Hkv,Sk,D]`` as bf16 bit patterns.  Returns ``(dq, dk, dv)``.
    """
    q, k, v, dout = _u16(q), _u16(k), _u16(v), _u16(dout)
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    if k.shape != v.shape or Bk != B or Dk != D or dout.shape != q.shape:
        raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape} dout{dout.shape}")
    dq = np.empty((B, Hq, Sq, D), np.float64)
    dk = np.empty((B, Hkv, Sk, D), np.float64)
    dv = np.empty((B, Hkv, Sk, D), np.float64)
    rc = _load().attn_ref_bwd(
        _ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16), _ptr(dout, ctypes.c_uint16),
        _ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double), _ptr(dv, ctypes.c_double),
        B, Hq, Hkv, Sq, Sk, D, int(causal), float(np.float32(scale)))
    if rc != 0:
        raise ValueError(f"attn_ref_bwd failed with status {rc}")
    return dq, dk, dv
