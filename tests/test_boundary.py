"""The C-ABI boundary on the host (no GPU needed): the libraries build for
sm_103a, load, export every symbol the headers declare, and reject bad
arguments with the documented status codes before touching any device.
"""
import ctypes
import os
import re
import subprocess

import pytest

from attention_forward_06_gb300 import build as B
from attention_forward_06_gb300 import _lib, ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = {"attn_fwd": "include/attn_fwd.h", "attn_fwd_trace": "include/attn_fwd_trace.h",
           "attn_bwd": "include/attn_bwd.h", "attn_bwd_trace": "include/attn_bwd_trace.h",
           "attn_probe": "include/attn_fwd_probe.h"}
TRACED = {"attn_fwd_trace": "attn_fwd", "attn_bwd_trace": "attn_bwd"}  # traced build -> the library it extends


@pytest.fixture(scope="module", autouse=True)
def built():
    return B.build()


def declared_functions(header):
    text = open(os.path.join(ROOT, header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


@pytest.mark.parametrize("name", sorted(HEADERS))
def test_library_exports_every_declared_symbol(name, built):
    funcs = declared_functions(HEADERS[name])
    assert funcs, "no declarations parsed"
    lib = ctypes.CDLL(built[name])
    for f in funcs:
        assert hasattr(lib, f), f"{f} declared in {HEADERS[name]} but not exported"
    # and the Python binding knows exactly these signatures (a traced build exports its library's as well)
    expected = set(funcs)
    if name in TRACED:
        expected |= set(declared_functions(HEADERS[TRACED[name]]))
        for f in declared_functions(HEADERS[TRACED[name]]):
            assert hasattr(lib, f), f"{f} missing from the traced build"
    assert sorted(_lib.SIGNATURES[name]) == sorted(expected)


@pytest.mark.parametrize("traced", sorted(TRACED))
def test_default_build_records_no_timeline(traced, built):
    lib = ctypes.CDLL(built[TRACED[traced]])
    for f in declared_functions(HEADERS[traced]):
        assert not hasattr(lib, f), f"{f} is exported by the default build"


def test_library_is_built_for_sm_103a_only(built):
    log = open(os.path.join(B.BUILD_DIR, "attn_fwd.ptxas.log")).read()
    assert "arch=compute_103a,code=sm_103a" in log
    assert "for 'sm_103a'" in log
    assert "sm_90" not in log and "sm_100" not in log


def test_version_and_strerror():
    lib = _lib.load()
    assert lib.attn_fwd_version() >= 100
    for code in range(0, 8):
        assert lib.attn_fwd_strerror(code)
    assert lib.attn_fwd_strerror(999) == b"unknown status"


# fake, 16-byte aligned addresses: validation never dereferences them
Q, K, V, O, L = 0x100000, 0x200000, 0x300000, 0x400000, 0x500000
GOOD = dict(B=1, Hq=4, Hkv=2, Sq=64, Sk=64, D=128, causal=1, scale=0.1)


def call(q=Q, k=K, v=V, o=O, lse=L, **kw):
    a = dict(GOOD)
    a.update(kw)
    return ops.attn_fwd_raw(q, k, v, o, lse, a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Sk"], a["D"], a["causal"],
                            a["scale"], 0)


@pytest.mark.parametrize("kw", [
    dict(D=96), dict(D=0), dict(D=256), dict(Hq=3, Hkv=2), dict(Hkv=0), dict(Hq=0), dict(causal=3),
    dict(causal=-1), dict(B=-1), dict(Sq=-5), dict(Sk=-1), dict(scale=float("nan")), dict(scale=float("inf")),
    dict(scale=0.0), dict(scale=-0.1),  # the masking takes scale > 0
])
def test_invalid_arguments(kw):
    assert call(**kw) == ops.ATTN_ERR_INVALID_ARG


def test_null_pointers():
    assert call(q=0) == ops.ATTN_ERR_NULL_PTR
    assert call(k=0) == ops.ATTN_ERR_NULL_PTR
    assert call(v=0) == ops.ATTN_ERR_NULL_PTR
    assert call(o=0) == ops.ATTN_ERR_NULL_PTR
    assert call(lse=0) == ops.ATTN_ERR_NULL_PTR


def test_misaligned_pointers():
    for kw in (dict(q=Q + 8), dict(k=K + 2), dict(v=V + 4), dict(o=O + 1), dict(lse=L + 4)):
        assert call(**kw) == ops.ATTN_ERR_MISALIGNED, kw


def test_overlapping_outputs_are_rejected():
    assert call(o=Q) == ops.ATTN_ERR_INVALID_ARG
    assert call(lse=K + 64) == ops.ATTN_ERR_INVALID_ARG
    assert call(o=V - 16) == ops.ATTN_ERR_INVALID_ARG


def test_empty_work_returns_ok_without_launching():
    # B == 0 or Sq == 0: nothing to compute, no CUDA call (passes on a machine without a GPU)
    assert call(B=0) == ops.ATTN_OK
    assert call(Sq=0) == ops.ATTN_OK
    assert call(q=0, o=0, lse=0, Sq=0) == ops.ATTN_OK or call(q=0, o=0, lse=0, Sq=0) == ops.ATTN_ERR_NULL_PTR


def test_keys_may_be_null_when_there_are_none():
    # Sk == 0 needs no k/v: validation passes; without a GPU the device query then fails with a CUDA error
    st = call(k=0, v=0, Sk=0)
    assert st in (ops.ATTN_OK, ops.ATTN_ERR_CUDA, ops.ATTN_ERR_UNSUPPORTED_DEVICE)


def test_oracle_and_library_share_no_code():
    # the oracle is plain C with no include of the library's headers, and the library never names the oracle
    src = open(os.path.join(ROOT, "oracle", "attn_ref.c")).read()
    assert "attn_fwd.h" not in src and "ptx.cuh" not in src
    for f in os.listdir(os.path.join(ROOT, "attention_forward_06_gb300", "csrc")):
        text = open(os.path.join(ROOT, "attention_forward_06_gb300", "csrc", f)).read()
        assert "attn_ref" not in text and "oracle" not in text
    for f in ("ops.py", "_lib.py", "build.py", "inputs.py", "__init__.py"):
        text = open(os.path.join(ROOT, "attention_forward_06_gb300", f)).read()
        assert "import oracle" not in text and "from oracle" not in text


def test_nm_lists_c_symbols_unmangled(built):
    out = subprocess.run(["nm", "-D", "--defined-only", built["attn_fwd"]], capture_output=True, text=True).stdout
    for f in declared_functions(HEADERS["attn_fwd"]):
        assert re.search(rf"\bT {f}$", out, flags=re.M), f


def test_splitkv_workspace_size_formula():
    for B, Hq, Sq, D, s in ((1, 2, 128, 64, 4), (2, 32, 513, 128, 7), (1, 1, 1, 128, 1)):
        rows = B * Hq * Sq
        o_bytes = s * rows * D * 4
        expect = ((o_bytes + 255) // 256) * 256 + s * rows * 4
        assert ops.splitkv_workspace_size(B, Hq, Sq, D, s) == expect
    assert ops.splitkv_workspace_size(1, 1, 1, 96, 1) == 0
    assert ops.splitkv_workspace_size(1, 1, 1, 128, 0) == 0
    assert ops.splitkv_workspace_size(1, 1, 1, 128, 257) == 0


def test_splitkv_invalid_arguments_before_any_device_work():
    lib = _lib.load()
    W = 0x600000
    for n_splits in (0, 257, -1):
        assert lib.attn_fwd_splitkv(Q, K, V, O, L, 1, 4, 2, 64, 64, 128, 1, 0.1, n_splits, W, 1 << 30, None) == \
            ops.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_splitkv(Q, K, V, O, L, 1, 4, 2, 64, 64, 96, 1, 0.1, 2, W, 1 << 30, None) == \
        ops.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_splitkv(0, K, V, O, L, 1, 4, 2, 64, 64, 128, 1, 0.1, 2, W, 1 << 30, None) == \
        ops.ATTN_ERR_NULL_PTR


def test_block_mask_words_formula():
    lib = _lib.load()
    for B, Hm, Sq, Sk in ((1, 1, 128, 128), (2, 4, 300, 5000), (1, 8, 1, 1), (3, 2, 257, 4097)):
        qb, kb = -(-Sq // 128), -(-Sk // 128)
        assert lib.attn_fwd_block_mask_words(B, Hm, Sq, Sk) == B * Hm * qb * ((kb + 31) // 32)
    assert lib.attn_fwd_block_mask_words(1, 0, 128, 128) == 0
    assert lib.attn_fwd_block_mask_words(-1, 1, 128, 128) == 0


def test_blocksparse_invalid_arguments_before_any_device_work():
    lib = _lib.load()
    M = 0x700000  # fake, aligned mask address
    args = lambda mask, heads: lib.attn_fwd_blocksparse(Q, K, V, O, L, 1, 4, 2, 64, 64, 128, 1, 0.1, mask, heads, None)
    assert args(M, 3) == ops.ATTN_ERR_INVALID_ARG       # neither 1 nor Hq
    assert args(M, 0) == ops.ATTN_ERR_INVALID_ARG
    assert args(0, 1) == ops.ATTN_ERR_NULL_PTR
    assert args(M + 2, 4) == ops.ATTN_ERR_MISALIGNED
    assert args(O, 1) == ops.ATTN_ERR_INVALID_ARG       # the mask overlaps the output


def test_tile_order_entries_formula():
    lib = _lib.load()
    for B, Ho, Sq, Sk in ((1, 1, 256, 128), (2, 4, 300, 5000), (1, 8, 1, 1), (3, 2, 513, 4097)):
        assert lib.attn_fwd_tile_order_entries(B, Ho, Sq, Sk) == B * Ho * -(-Sq // 256) * -(-Sk // 128)
    assert lib.attn_fwd_tile_order_entries(1, 0, 128, 128) == 0
    assert lib.attn_fwd_tile_order_entries(1, 1, -1, 128) == 0


def test_ordered_invalid_arguments_before_any_device_work():
    lib = _lib.load()
    T = 0x700000  # fake, aligned order address
    args = lambda order, heads, **kw: lib.attn_fwd_ordered(Q, K, V, O, L, 1, 4, 2, 64, 64, 128, 1,
                                                         kw.get("scale", 0.1), order, heads, None)
    assert args(T, 3) == ops.ATTN_ERR_INVALID_ARG       # neither 1 nor Hq
    assert args(T, 0) == ops.ATTN_ERR_INVALID_ARG
    assert args(0, 1) == ops.ATTN_ERR_NULL_PTR
    assert args(T + 2, 4) == ops.ATTN_ERR_MISALIGNED
    assert args(O, 1) == ops.ATTN_ERR_INVALID_ARG       # the order overlaps the output
    assert args(T, 1, scale=0.0) == ops.ATTN_ERR_INVALID_ARG


def test_bwd_workspace_formula_and_invalid_arguments():
    lib = _lib.load("attn_bwd")
    for B, Hq, Sq in ((1, 1, 1), (2, 16, 2048), (3, 5, 300)):
        one = B * Hq * (-(-Sq // 128) * 128) * 4
        assert lib.attn_bwd_workspace_size(B, Hq, Sq) == 2 * ((one + 255) // 256 * 256)
    W = 0x900000
    call = lambda **kw: lib.attn_bwd(*[kw.get(n, a) for n, a in zip(
        ("q", "k", "v", "o", "lse", "do", "dq", "dk", "dv"),
        (0x100000, 0x200000, 0x300000, 0x400000, 0x500000, 0x600000, 0x700000, 0x800000, 0x880000))],
        1, 4, kw.get("Hkv", 2), 64, 64, kw.get("D", 128), 1, kw.get("scale", 0.1), kw.get("ws", W), 1 << 20, None)
    assert call(D=96) == ops.ATTN_ERR_INVALID_ARG
    assert call(scale=0.0) == ops.ATTN_ERR_INVALID_ARG
    assert call(scale=-0.5) == ops.ATTN_ERR_INVALID_ARG
    assert call(Hkv=3) == ops.ATTN_ERR_INVALID_ARG
    assert call(dq=0) == ops.ATTN_ERR_NULL_PTR
    assert call(ws=0) == ops.ATTN_ERR_NULL_PTR
    assert call(dk=0x800008) == ops.ATTN_ERR_MISALIGNED
    assert call(dq=0x100000) == ops.ATTN_ERR_INVALID_ARG    # dq overlaps q
    assert call(dv=0x800000) == ops.ATTN_ERR_INVALID_ARG    # dv overlaps dk
