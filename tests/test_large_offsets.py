"""Parity past 2^31 elements: forward and backward calls whose Q, O, dO and dQ each
hold more than 2^31 bf16 values (4.3 GB), so every offset into them beyond 4 GiB
must be formed in 64 bits (tensor-map coordinates, row pointers, the LSE index).

The shape: one kv head of 300 keys shared by 129 query heads of 131073 rows each
(G = 129, ragged in both lengths), no mask, D = 128.  Rows sampled over the whole
range, the last rows of the last head included, are checked against the oracle.
With no mask each row sees every key of the one kv head, so the sampled rows form
a problem of their own: n query heads of one row each over the same K and V, whose
forward and whose dQ the oracle computes exactly as it would inside the full call
(a row's O, LSE and dQ depend only on that row, K, V and its dO).  dK and dV sum
over all 16.9 million rows and are checked for finiteness only.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_06_gb300 import ops
from attention_forward_06_gb300.inputs import bf16_bits, draw, draw_on_device
from parity_util import compare
from test_backward import check

pytestmark = pytest.mark.gpu

B, HQ, HKV, SQ, SK, D = 1, 129, 1, 131073, 300, 128


def sampled_rows(n_random: int, seed: int):
    rng = np.random.default_rng(seed)
    h = np.concatenate([[0, 0, HQ - 1, HQ - 1, HQ - 1], rng.integers(0, HQ, n_random)])
    i = np.concatenate([[0, SQ - 1, 0, SQ - 2, SQ - 1], rng.integers(0, SQ, n_random)])
    return h, i


def test_forward_and_backward_past_2_to_the_31_elements():
    assert B * HQ * SQ * D > 2 ** 31
    free, _ = torch.cuda.mem_get_info()
    if free < (24 << 30):
        pytest.skip("needs about 20 GB of free device memory")
    q = draw_on_device((B, HQ, SQ, D), seed=71)
    do = draw_on_device((B, HQ, SQ, D), seed=72)
    _, k, v = draw(1, 1, HKV, 1, SK, D, seed=73)
    scale = float(np.float32(D ** -0.5))
    kd, vd = k.cuda(), v.cuda()

    o, lse = ops.attn_fwd(q, kd, vd, causal=0, scale=scale)
    st, site = ops.debug_status()
    assert st == ops.ATTN_OK, f"kernel wait ran out at site {site}"
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
    dq, dk, dv = ops.attn_bwd(q, kd, vd, o, lse, do, causal=0, scale=scale)
    st, site = ops.bwd_debug_status()
    assert st == ops.ATTN_OK, f"backward wait ran out at site {site}"
    assert bool(torch.isfinite(dq).all()) and bool(torch.isfinite(dk).all()) and bool(torch.isfinite(dv).all())

    h, i = sampled_rows(59, seed=74)
    assert int(((h * SQ + i) * D).max()) >= 2 ** 31  # the last rows sit past 2^31 elements
    hi, ii = torch.as_tensor(h, device="cuda"), torch.as_tensor(i, device="cuda")
    n = len(h)

    def rows(t):  # [1, HQ, SQ, ...] -> the sampled rows as [1, n, 1, ...] on the CPU
        return t[0, hi, ii].reshape((1, n, 1) + tuple(t.shape[3:])).contiguous().cpu()

    q_rows, do_rows = rows(q), rows(do)
    o_ref, lse_ref = oracle.attention(bf16_bits(q_rows), bf16_bits(k), bf16_bits(v), 0, scale)
    compare(rows(o), rows(lse), o_ref, lse_ref)
    dq_ref, _, _ = oracle.backward(bf16_bits(q_rows), bf16_bits(k), bf16_bits(v), bf16_bits(do_rows), 0, scale)
    check("dq", rows(dq), dq_ref)
