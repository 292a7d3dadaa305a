"""Split-key forward (attn_fwd_splitkv): the same result as the single-pass
kernel, for shapes with few query blocks and long key ranges; partial results
per key range are merged by their log-sum-exp."""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_06_gb300 import ops
from attention_forward_06_gb300.inputs import bf16_bits, draw, sample_rows
from parity_util import compare

pytestmark = pytest.mark.gpu


def check_against_oracle(B, Hq, Hkv, Sq, Sk, D, causal, n_splits, seed, qk_std=1.0):
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, D, seed, qk_std=qk_std)
    scale = float(np.float32(D ** -0.5))
    o, lse = ops.attn_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, n_splits=n_splits)
    st, site = ops.debug_status()
    assert st == ops.ATTN_OK, site
    o_ref, lse_ref = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal, scale)
    return compare(o.cpu(), lse.cpu(), o_ref, lse_ref)


@pytest.mark.parametrize("shape,splits", [
    ((1, 4, 1, 300, 1000, 128, 1), 1),
    ((1, 4, 1, 300, 1000, 128, 1), 2),
    ((1, 4, 1, 300, 1000, 128, 1), 3),
    ((1, 4, 1, 300, 1000, 128, 1), 7),
    ((2, 2, 2, 129, 4000, 64, 0), 5),
    ((1, 8, 2, 512, 4096, 128, 1), 16),
    ((1, 2, 1, 64, 200, 128, 0), 5),      # more ranges than key tiles: empty ranges
    ((1, 2, 2, 600, 300, 64, 1), 3),      # Sq > Sk: fully masked rows
    ((1, 2, 1, 100, 2000, 128, 2), 4),    # top-left mask
], ids=lambda x: str(x))
def test_splitkv_matches_oracle(shape, splits):
    check_against_oracle(*shape, n_splits=splits, seed=sum(shape) + splits)


def test_splitkv_sharp_logits():
    check_against_oracle(1, 4, 1, 256, 3000, 128, 1, n_splits=6, seed=91, qk_std=3.0)


def test_splitkv_agrees_with_single_pass():
    q, k, v = [t.cuda() for t in draw(1, 8, 2, 384, 6000, 128, seed=17)]
    o1, l1 = ops.attn_fwd(q, k, v, causal=1)
    o2, l2 = ops.attn_fwd_splitkv(q, k, v, causal=1, n_splits=9)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 2 ** -6
    assert (l1 - l2).abs().max().item() <= 1e-4


def test_long_request_shape_on_sampled_rows():
    # a 512-query chunk against a 131072-key cache: 64 query blocks, far fewer than the SMs
    B, Hq, Hkv, Sq, Sk, D = 1, 32, 8, 512, 131072, 128
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, D, seed=33)
    splits = ops.splitkv_suggest(B, Hq, Sq, Sk, D, 1)
    assert splits > 1
    o, lse = ops.attn_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=1, n_splits=splits)
    rows = sample_rows(B, Hq, Sq, 6, seed=34)
    scale = float(np.float32(D ** -0.5))
    o_ref, lse_ref = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 1, scale, rows=rows)
    idx = torch.from_numpy(rows)
    compare(o.cpu().reshape(-1, D)[idx], lse.cpu().reshape(-1)[idx], o_ref, lse_ref)


def test_suggest_is_one_when_the_gpu_is_full():
    assert ops.splitkv_suggest(4, 16, 2048, 2048, 128, 1) == 1
    assert ops.splitkv_suggest(1, 1, 256, 100000, 128, 0) > 1


def test_workspace_checks():
    q, k, v = [t.cuda() for t in draw(1, 2, 1, 128, 1000, 64, seed=5)]
    o = torch.empty_like(q)
    lse = torch.empty((1, 2, 128), device="cuda")
    need = ops.splitkv_workspace_size(1, 2, 128, 64, 4)
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    st = ops.load().attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                     1, 2, 1, 128, 1000, 64, 0, 0.125, 4, small.data_ptr(), need - 16, None)
    assert st == ops.ATTN_ERR_INVALID_ARG
    st = ops.load().attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                     1, 2, 1, 128, 1000, 64, 0, 0.125, 4, None, need, None)
    assert st == ops.ATTN_ERR_NULL_PTR


def test_suggested_split_of_an_equal_item_workload_matches_the_oracle():
    # 512 equal work items on the GPU's SMs leave the last wave partly filled; the suggestion splits the keys
    # (the chunked-prefill shape at D = 64: 8 x 32 query heads, 512 rows, 16384 keys, bottom-right causal)
    B, Hq, Hkv, Sq, Sk, D = 8, 32, 8, 512, 16384, 64
    splits = ops.splitkv_suggest(B, Hq, Sq, Sk, D, 1)
    assert splits > 1
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, D, seed=35)
    o, lse = ops.attn_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=1, n_splits=splits)
    rows = sample_rows(B, Hq, Sq, 3, seed=36)
    scale = float(np.float32(D ** -0.5))
    o_ref, lse_ref = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 1, scale, rows=rows)
    idx = torch.from_numpy(rows)
    compare(o.cpu().reshape(-1, D)[idx], lse.cpu().reshape(-1)[idx], o_ref, lse_ref)


def test_one_split_is_the_plain_forward_bit_for_bit():
    q, k, v = [t.cuda() for t in draw(2, 8, 2, 700, 1500, 128, seed=37)]
    o1, l1 = ops.attn_fwd(q, k, v, causal=1)
    ws = torch.full((ops.splitkv_workspace_size(2, 8, 700, 128, 1),), 7, dtype=torch.uint8, device="cuda")
    o2, l2 = ops.attn_fwd_splitkv(q, k, v, causal=1, n_splits=1, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert bool((ws == 7).all())  # one range needs no partials
