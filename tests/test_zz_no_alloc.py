"""attn_fwd_splitkv_noalloc: the split-key forward for callers that are handed
only their input and output buffers and may not call cudaMalloc (its partials
live in a fixed array inside the library).  Called through the C ABI and checked
against attn_fwd_splitkv, which takes a caller workspace, on two calls in a row
(bit for bit: the same kernels run on the same key ranges); the second call uses
different inputs so stale scratch contents would show.
"""
import ctypes

import pytest
import torch

from attention_forward_06_gb300 import _lib, ops
from attention_forward_06_gb300.inputs import draw

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module")
def lib():
    from attention_forward_06_gb300 import build
    build.build()
    return _lib.load("attn_fwd")


def call_noalloc(lib, q, k, v, o, lse, causal, scale, n_splits):
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    return lib.attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                        B, Hq, Hkv, Sq, Sk, D, causal, ctypes.c_float(scale), n_splits,
                                        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("shape,causal,n_splits", [
    ((1, 8, 2, 256, 8192, 128), 1, 6),
    ((2, 4, 4, 130, 3000, 64), 0, 5),
])
def test_noalloc_matches_workspace_entry_point_twice(lib, shape, causal, n_splits):
    B, Hq, Hkv, Sq, Sk, D = shape
    scale = D ** -0.5
    for call, seed in enumerate((101, 202)):
        q, k, v = [t.cuda() for t in draw(B, Hq, Hkv, Sq, Sk, D, seed=seed + sum(shape))]
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, Hq, Sq), float("nan"), device="cuda")
        assert call_noalloc(lib, q, k, v, o, lse, causal, scale, n_splits) == ops.ATTN_OK, f"call {call}"
        o_ref, lse_ref = ops.attn_fwd_splitkv(q, k, v, causal=causal, scale=scale, n_splits=n_splits)
        torch.cuda.synchronize()
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        # the same two kernels run on the same key ranges; only where the partials live differs
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), f"call {call}"


def test_noalloc_rejects_work_beyond_its_fixed_scratch(lib):
    # 8 splits x 32768 rows x 129 floats x 4 bytes = 135 MB > 32 MiB: rejected before any device work
    q, k, v = [t.cuda() for t in draw(1, 64, 8, 512, 512, 128, seed=7)]
    o = torch.zeros_like(q)
    lse = torch.zeros((1, 64, 512), device="cuda")
    assert call_noalloc(lib, q, k, v, o, lse, 1, 0.088, 8) == ops.ATTN_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert o.abs().max().item() == 0.0
    # and a call that fits still works afterwards
    assert call_noalloc(lib, q[:, :4].contiguous(), k[:, :1].contiguous(), v[:, :1].contiguous(),
                        o[:, :4].contiguous(), lse[:, :4].contiguous(), 1, 0.088, 2) == ops.ATTN_OK
    torch.cuda.synchronize()
