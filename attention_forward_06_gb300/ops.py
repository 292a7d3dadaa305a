"""Python binding of the C ABI (include/attn_fwd.h): marshals torch tensors into
pointers and sizes and calls the CUDA library.  Every step of the attention
computation runs in the library's kernel; torch only provides device memory and
streams here.
"""
from __future__ import annotations

import ctypes
import math

import torch

from ._lib import load

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_NULL_PTR = 2
ATTN_ERR_MISALIGNED = 3
ATTN_ERR_UNSUPPORTED_DEVICE = 4
ATTN_ERR_CUDA = 5
ATTN_ERR_DEVICE_TIMEOUT = 6
ATTN_ERR_TENSOR_MAP = 7


class AttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"attn_fwd status {status}: {message}")
        self.status = status


def _check(status: int) -> None:
    if status != ATTN_OK:
        msg = load().attn_fwd_strerror(status).decode()
        raise AttnError(status, msg)


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def attn_fwd_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int, Hq: int, Hkv: int,
                 Sq: int, Sk: int, D: int, causal: int, scale: float, stream: int) -> int:
    """Direct call of the C entry point with integer pointers; returns the status code."""
    return load().attn_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, Hq, Hkv, Sq, Sk, D, causal,
                           ctypes.c_float(scale), stream)


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: int = 1, scale: float | None = None,
             o: torch.Tensor | None = None, lse: torch.Tensor | None = None, stream=None):
    """Exact attention forward: returns ``(o, lse)``.

    q ``[B,Hq,Sq,D]``, k/v ``[B,Hkv,Sk,D]``: contiguous bf16 CUDA tensors.  ``causal`` is
    0 (none), 1 (bottom-right aligned) or 2 (top-left aligned).  ``scale`` defaults to
    1/sqrt(D).  ``o``/``lse`` may be given (``[B,Hq,Sq,D]`` bf16, ``[B,Hq,Sq]`` fp32) to
    avoid allocation.  Asynchronous on ``stream`` (default: torch's current stream).
    """
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-d bf16 CUDA tensor")
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or Dk != D:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    if o.shape != q.shape or o.dtype != torch.bfloat16 or not o.is_contiguous():
        raise ValueError("o must be a contiguous bf16 tensor shaped like q")
    if tuple(lse.shape) != (B, Hq, Sq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B, Hq, Sq]")
    _check(attn_fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                        B, Hq, Hkv, Sq, Sk, D, int(causal), float(scale), _stream_handle(stream)))
    return o, lse


def splitkv_workspace_size(B: int, Hq: int, Sq: int, D: int, n_splits: int) -> int:
    return int(load().attn_fwd_splitkv_workspace_size(B, Hq, Sq, D, n_splits))


def splitkv_suggest(B: int, Hq: int, Sq: int, Sk: int, D: int, causal: int) -> int:
    return int(load().attn_fwd_splitkv_suggest(B, Hq, Sq, Sk, D, causal))


def attn_fwd_splitkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: int = 1, scale: float | None = None,
                     n_splits: int | None = None, workspace: torch.Tensor | None = None,
                     o: torch.Tensor | None = None, lse: torch.Tensor | None = None, stream=None):
    """Split-key forward (same result as ``attn_fwd``): ``(o, lse)``.

    ``n_splits`` defaults to ``splitkv_suggest``; ``workspace`` (a CUDA tensor of at
    least ``splitkv_workspace_size`` bytes) is allocated here when not given.
    """
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-d bf16 CUDA tensor")
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or Dk != D:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if n_splits is None:
        n_splits = splitkv_suggest(B, Hq, Sq, Sk, D, int(causal))
    need = splitkv_workspace_size(B, Hq, Sq, D, n_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(load().attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                   B, Hq, Hkv, Sq, Sk, D, int(causal), ctypes.c_float(scale), int(n_splits),
                                   workspace.data_ptr(), ws_bytes, _stream_handle(stream)))
    return o, lse


def attn_fwd_splitkv_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: int = 1,
                             scale: float | None = None, n_splits: int = 1, o: torch.Tensor | None = None,
                             lse: torch.Tensor | None = None, stream=None):
    """Split-key forward with the library's fixed scratch instead of a workspace: ``(o, lse)``.

    For callers that get only their input and output buffers and may not allocate
    device memory; ``o``/``lse`` should then be given.  Work beyond the fixed
    scratch (32 MiB of partials) is rejected; overlapping calls on the GPU race.
    """
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    _check(load().attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                           B, Hq, Hkv, Sq, Sk, D, int(causal), ctypes.c_float(scale), int(n_splits),
                                           _stream_handle(stream)))
    return o, lse


MASK_BLOCK = 128  # query rows and keys per block of a block mask (ATTN_MASK_BLOCK)


def block_mask_words(B: int, mask_heads: int, Sq: int, Sk: int) -> int:
    return int(load().attn_fwd_block_mask_words(B, mask_heads, Sq, Sk))


def pack_block_mask(blocks: torch.Tensor) -> torch.Tensor:
    """Bit-pack a boolean block mask ``[B, H, ceil(Sq/128), ceil(Sk/128)]`` into int32 words
    ``[B, H, ceil(Sq/128), ceil(ceil(Sk/128)/32)]`` (bit ``kb % 32`` of word ``kb // 32``), on its device."""
    if blocks.dim() != 4 or blocks.dtype != torch.bool:
        raise ValueError("blocks must be a 4-d bool tensor [B, H, query blocks, key blocks]")
    B, H, QB, KB = blocks.shape
    W = (KB + 31) // 32
    padded = torch.zeros((B, H, QB, W * 32), dtype=torch.int64, device=blocks.device)
    padded[..., :KB] = blocks.to(torch.int64)
    weights = torch.tensor([1 << b for b in range(32)], dtype=torch.int64, device=blocks.device)
    words = (padded.view(B, H, QB, W, 32) * weights).sum(-1)
    return (words - (words >= (1 << 31)).to(torch.int64) * (1 << 32)).to(torch.int32).contiguous()


def attn_fwd_blocksparse(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, block_mask: torch.Tensor,
                         causal: int = 1, scale: float | None = None, o: torch.Tensor | None = None,
                         lse: torch.Tensor | None = None, stream=None):
    """Block-sparse forward: ``attn_fwd`` restricted to the marked (query block, key block) pairs.

    ``block_mask``: contiguous int32 (or uint32) CUDA tensor ``[B, 1 or Hq, ceil(Sq/128), W]`` of
    bit-packed words (see ``pack_block_mask``).  Returns ``(o, lse)``.
    """
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-d bf16 CUDA tensor")
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or Dk != D:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if block_mask.element_size() != 4 or not block_mask.is_cuda or not block_mask.is_contiguous() or \
            block_mask.dim() != 4:
        raise ValueError("block_mask must be a contiguous 4-d 32-bit CUDA tensor")
    Hm = block_mask.shape[1]
    W = (-(-Sk // MASK_BLOCK) + 31) // 32
    if tuple(block_mask.shape) != (B, Hm, -(-Sq // MASK_BLOCK), W):
        raise ValueError(f"block_mask shape {tuple(block_mask.shape)} does not fit q{tuple(q.shape)} k{tuple(k.shape)}")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    _check(load().attn_fwd_blocksparse(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                       B, Hq, Hkv, Sq, Sk, D, int(causal), ctypes.c_float(scale),
                                       block_mask.data_ptr(), int(Hm), _stream_handle(stream)))
    return o, lse


ORDER_ROWS = 256  # query rows sharing one key-tile order (ATTN_ORDER_ROWS)
ORDER_KEYS = 128  # keys per key tile of an order (ATTN_ORDER_KEYS)


def tile_order_entries(B: int, order_heads: int, Sq: int, Sk: int) -> int:
    return int(load().attn_fwd_tile_order_entries(B, order_heads, Sq, Sk))


def attn_fwd_ordered(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, tile_order: torch.Tensor,
                     causal: int = 1, scale: float | None = None, o: torch.Tensor | None = None,
                     lse: torch.Tensor | None = None, stream=None):
    """Forward with the key tiles of each 256-row query block visited in ``tile_order``'s order: ``(o, lse)``.

    ``tile_order``: contiguous int32 CUDA tensor ``[B, 1 or Hq, ceil(Sq/256), ceil(Sk/128)]`` of key-tile
    indices; each row is visited in order, entries outside the block's causal tile range passed over.
    """
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-d bf16 CUDA tensor")
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or Dk != D:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if tile_order.dtype != torch.int32 or not tile_order.is_cuda or not tile_order.is_contiguous() or \
            tile_order.dim() != 4:
        raise ValueError("tile_order must be a contiguous 4-d int32 CUDA tensor")
    Ho = tile_order.shape[1]
    if tuple(tile_order.shape) != (B, Ho, -(-Sq // ORDER_ROWS), -(-Sk // ORDER_KEYS)):
        raise ValueError(f"tile_order shape {tuple(tile_order.shape)} does not fit q{tuple(q.shape)} k{tuple(k.shape)}")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    _check(load().attn_fwd_ordered(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                   B, Hq, Hkv, Sq, Sk, D, int(causal), ctypes.c_float(scale),
                                   tile_order.data_ptr(), int(Ho), _stream_handle(stream)))
    return o, lse


def bwd_workspace_size(B: int, Hq: int, Sq: int) -> int:
    return int(load("attn_bwd").attn_bwd_workspace_size(B, Hq, Sq))


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
             dout: torch.Tensor, causal: int = 1, scale: float | None = None, dq: torch.Tensor | None = None,
             dk: torch.Tensor | None = None, dv: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
             stream=None):
    """Backward of ``attn_fwd``: ``(dq, dk, dv)`` for the upstream gradient ``dout`` of ``o``.

    ``o`` and ``lse`` are the forward's outputs for the same ``q, k, v, causal, scale``.
    """
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-d bf16 CUDA tensor")
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or Dk != D or o.shape != q.shape or dout.shape != q.shape:
        raise ValueError("shape mismatch")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, Sq) or not lse.is_contiguous():
        raise ValueError("lse must be the forward's contiguous fp32 [B, Hq, Sq]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = bwd_workspace_size(B, Hq, Sq)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    lib = load("attn_bwd")
    st = lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                      dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, Sq, Sk, D, int(causal),
                      ctypes.c_float(scale), workspace.data_ptr(), ws_bytes, _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, lib.attn_bwd_strerror(st).decode())
    return dq, dk, dv


def bwd_debug_status(stream=None) -> tuple[int, int]:
    """Synchronise ``stream`` and read/clear the backward kernels' timeout word: ``(status, site)``."""
    site = ctypes.c_int(0)
    st = load("attn_bwd").attn_bwd_debug_status(_stream_handle(stream), ctypes.byref(site))
    return st, site.value


def debug_status(stream=None) -> tuple[int, int]:
    """Synchronise ``stream`` and read/clear the kernel's timeout word: ``(status, site)``."""
    site = ctypes.c_int(0)
    st = load().attn_fwd_debug_status(_stream_handle(stream), ctypes.byref(site))
    return st, site.value


def version() -> int:
    return int(load().attn_fwd_version())
