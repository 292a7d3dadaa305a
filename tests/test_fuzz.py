"""Seeded random configurations through every entry point, against the fp64 oracle.

Each case draws batch, heads (grouped-query ratios 1 to 8), ragged lengths up to
600, D in {64, 128}, all three causal modes, a positive scale around 1/sqrt(D)
and a logit spread from soft to sharply peaked; it runs the plain forward, one of
the split-key, block-sparse or ordered forwards (chosen by the case), and on every
third case the backward (odd cases run the dense forward in the grouped item order), each compared with the oracle's result for the same
inputs (the ordered forward with a random permutation is plain attention; the
block-sparse one is compared with the oracle's block-mask path).
"""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_06_gb300 import ops
from attention_forward_06_gb300.inputs import bf16_bits, draw
from parity_util import compare, round_to_bf16

pytestmark = pytest.mark.gpu
N_CASES = 96


def case_params(i):
    rng = np.random.default_rng(1000 + i)
    G = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.integers(1, 3))
    B = int(rng.integers(1, 3))
    D = int(rng.choice([64, 128]))
    Sq = int(rng.integers(1, 601))
    Sk = int(rng.integers(1, 601))
    causal = int(rng.integers(0, 3))
    scale = float(np.float32(D ** -0.5 * rng.uniform(0.5, 2.0)))
    qk_std = float(rng.choice([0.5, 1.0, 3.0]))
    return dict(B=B, Hq=Hkv * G, Hkv=Hkv, Sq=Sq, Sk=Sk, D=D, causal=causal, scale=scale, qk_std=qk_std, seed=2000 + i)


def check_grad(name, g, ref):
    g = g.float().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), f"non-finite {name}"
    if not ref.size:
        return
    peak = np.abs(ref).max()
    excess = np.abs(g - ref) - np.abs(round_to_bf16(ref) - ref)
    assert excess.max() <= 1e-2 * peak + 1e-6, f"{name}: excess {excess.max():.3g} (max|ref| {peak:.3g})"
    norm = np.linalg.norm(ref)
    if norm > 0:
        assert np.linalg.norm(g - ref) / norm <= 1e-2, f"{name}: relative error"


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case(i, monkeypatch):
    c = case_params(i)
    # half the cases run the dense forward in the grouped item order (a kv head's items together), which the
    # library otherwise picks only for K and V larger than L2
    if i % 2:
        monkeypatch.setenv("ATTN_FWD_ITEM_ORDER", "grouped")
    B, Hq, Hkv, Sq, Sk, D, causal, scale = (c[k] for k in ("B", "Hq", "Hkv", "Sq", "Sk", "D", "causal", "scale"))
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, D, c["seed"], qk_std=c["qk_std"])
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    qb, kb, vb = bf16_bits(q), bf16_bits(k), bf16_bits(v)
    o_ref, lse_ref = oracle.attention(qb, kb, vb, causal, scale)

    o, lse = ops.attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    st, site = ops.debug_status()
    assert st == ops.ATTN_OK, f"forward wait ran out at site {site}"
    compare(o, lse, o_ref, lse_ref)

    rng = np.random.default_rng(3000 + i)
    kind = i % 3
    if kind == 0:
        n_splits = int(rng.integers(1, 6))
        o2, l2 = ops.attn_fwd_splitkv(qd, kd, vd, causal=causal, scale=scale, n_splits=n_splits)
        ref2 = (o_ref, lse_ref)
    elif kind == 1:
        Hm = int(rng.choice([1, Hq]))
        blocks = torch.from_numpy(rng.random((B, Hm, -(-Sq // 128), -(-Sk // 128))) < 0.6)
        words = ops.pack_block_mask(blocks).cuda()
        o2, l2 = ops.attn_fwd_blocksparse(qd, kd, vd, words, causal=causal, scale=scale)
        ref2 = oracle.attention(qb, kb, vb, causal, scale, block_mask=words.cpu().numpy().view(np.uint32))
    else:
        Ho = int(rng.choice([1, Hq]))
        shp = (B, Ho, -(-Sq // 256), -(-Sk // 128))
        order = np.empty(shp, np.int32)
        for idx in np.ndindex(*shp[:3]):
            order[idx] = rng.permutation(shp[3])
        o2, l2 = ops.attn_fwd_ordered(qd, kd, vd, torch.from_numpy(order).cuda(), causal=causal, scale=scale)
        ref2 = (o_ref, lse_ref)
    st, site = ops.debug_status()
    assert st == ops.ATTN_OK, f"forward wait ran out at site {site}"
    compare(o2, l2, *ref2)

    if i % 3 == 0:
        do = draw(B, Hq, Hkv, Sq, Sk, D, c["seed"] + 1)[0]
        dq, dk, dv = ops.attn_bwd(qd, kd, vd, o, lse, do.cuda(), causal=causal, scale=scale)
        st, site = ops.bwd_debug_status()
        assert st == ops.ATTN_OK, f"backward wait ran out at site {site}"
        rq, rk, rv = oracle.backward(qb, kb, vb, bf16_bits(do), causal, scale)
        check_grad("dq", dq.cpu(), rq)
        check_grad("dk", dk.cpu(), rk)
        check_grad("dv", dv.cpu(), rv)
