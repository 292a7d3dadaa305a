"""Parity of the ordered forward (attn_fwd_ordered, through the C ABI): the key
tiles of every 256-row query block visited in a given order.  With every tile
listed the result is attention itself, so it is compared with the fp64 oracle's
plain attention (random permutations, reversed order, a score-ranked order on
sharply peaked rows, orders wider than one 32-entry window, shared and per-head
orders, all three causal modes, rows without keys); the identity order must
reproduce the dense kernel bit for bit; a row that leaves tiles out (or holds
entries out of range) is block-sparse attention and is compared with the
oracle's block-mask path.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_06_gb300 import ops
from attention_forward_06_gb300.inputs import bf16_bits, draw
from parity_util import compare

pytestmark = pytest.mark.gpu
ROWS, KEYS = 256, 128


def shape_of(B, Ho, Sq, Sk):
    return (B, Ho, -(-Sq // ROWS), -(-Sk // KEYS))


def run(q, k, v, order, causal, scale):
    t = torch.from_numpy(np.ascontiguousarray(order, dtype=np.int32)).cuda()
    o, lse = ops.attn_fwd_ordered(q.cuda(), k.cuda(), v.cuda(), t, causal=causal, scale=scale)
    st, site = ops.debug_status()
    assert st == ops.ATTN_OK, f"kernel wait ran out at site {site}"
    return o.cpu(), lse.cpu()


def permutations(B, Ho, Sq, Sk, seed):
    rng = np.random.default_rng(seed)
    shp = shape_of(B, Ho, Sq, Sk)
    out = np.empty(shp, np.int32)
    for idx in np.ndindex(*shp[:3]):
        out[idx] = rng.permutation(shp[3])
    return out


CASES = [
    # B, Hq, Hkv, Sq, Sk, D, causal, order heads
    (1, 4, 2, 300, 700, 128, 1, 1),
    (2, 4, 4, 513, 513, 64, 0, 4),
    (1, 2, 1, 1000, 129, 128, 1, 2),      # Sq > Sk bottom-right: rows without keys
    (1, 8, 2, 256, 2048, 128, 2, 8),
    (1, 2, 2, 640, 5000, 64, 0, 1),       # 40 key tiles: two 32-entry windows per row
    (1, 3, 1, 777, 4500, 128, 1, 3),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_random_orders_match_oracle(case):
    B, Hq, Hkv, Sq, Sk, D, causal, Ho = case
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, D, seed=sum(case))
    scale = float(np.float32(D ** -0.5))
    o, lse = run(q, k, v, permutations(B, Ho, Sq, Sk, seed=Sq * 7 + Sk), causal, scale)
    o_ref, lse_ref = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal, scale)
    compare(o, lse, o_ref, lse_ref)


def test_identity_order_equals_dense_kernel_bitwise():
    for (B, Hq, Hkv, Sq, Sk, D) in ((2, 4, 2, 700, 900, 128), (1, 2, 1, 513, 4500, 64)):
        q, k, v = draw(B, Hq, Hkv, Sq, Sk, D, seed=Sq + D)
        shp = shape_of(B, 1, Sq, Sk)
        ident = np.broadcast_to(np.arange(shp[3], dtype=np.int32), shp)
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        for causal in (0, 1, 2):
            o1, l1 = ops.attn_fwd(qd, kd, vd, causal=causal)
            o2, l2 = run(q, k, v, ident, causal, D ** -0.5)
            assert torch.equal(o1.cpu(), o2) and torch.equal(l1.cpu(), l2), (B, Sq, Sk, D, causal)


def test_reversed_and_score_ranked_orders_on_sharp_rows():
    # Q, K ~ N(0, 3^2): sharply peaked rows, so the first tile visited decides the running max
    B, Hq, Hkv, Sq, Sk, D = 1, 4, 1, 512, 2048, 128
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, D, seed=77, qk_std=3.0)
    scale = float(np.float32(D ** -0.5))
    o_ref, lse_ref = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 1, scale)
    shp = shape_of(B, Hq, Sq, Sk)
    rev = np.broadcast_to(np.arange(shp[3] - 1, -1, -1, dtype=np.int32), shp)
    compare(*run(q, k, v, rev, 1, scale), o_ref, lse_ref)
    # score-ranked: block means of Q rows and K keys, best key tile first (a training-free proxy)
    qf, kf = q.float(), k.float()
    qm = qf.reshape(B, Hq, shp[2], ROWS, D).mean(3)                      # [B, Hq, blocks, D]
    km = kf.reshape(B, Hkv, shp[3], KEYS, D).mean(3).repeat_interleave(Hq // Hkv, 1)
    score = torch.einsum("bhqd,bhkd->bhqk", qm, km)
    ranked = torch.argsort(score, dim=-1, descending=True).to(torch.int32).numpy()
    compare(*run(q, k, v, ranked, 1, scale), o_ref, lse_ref)


def test_rows_leaving_tiles_out_give_block_sparse_attention():
    B, Hq, Hkv, Sq, Sk, D = 1, 4, 2, 600, 3000, 128
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, D, seed=91)
    scale = float(np.float32(D ** -0.5))
    rng = np.random.default_rng(5)
    shp = shape_of(B, Hq, Sq, Sk)
    order = np.full(shp, -1, np.int32)
    blocks = np.zeros((B, Hq, -(-Sq // KEYS), shp[3]), bool)   # the oracle's 128 x 128 block mask
    for b, h, u in np.ndindex(*shp[:3]):
        keep = rng.permutation(shp[3])[: rng.integers(1, shp[3] + 1)]
        row = np.concatenate([keep, [-5, shp[3], shp[3] + 100]])   # entries out of range are passed over
        rng.shuffle(row)
        order[b, h, u, : len(row)] = row[: shp[3]]
        listed = [e for e in order[b, h, u] if 0 <= e < shp[3]]
        for qb in (2 * u, 2 * u + 1):
            if qb < blocks.shape[2]:
                blocks[b, h, qb, listed] = True
    words = np.zeros(blocks.shape[:3] + ((shp[3] + 31) // 32,), np.uint32)
    for kb in range(shp[3]):
        words[..., kb // 32] |= blocks[..., kb].astype(np.uint32) << np.uint32(kb % 32)
    o, lse = run(q, k, v, order, 1, scale)
    o_ref, lse_ref = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 1, scale, block_mask=words)
    compare(o, lse, o_ref, lse_ref)
