"""Parity of the block-sparse forward (attn_fwd_blocksparse, through the C ABI)
with the fp64 oracle's block-mask path, element by element on seeded inputs:
random masks over ragged shapes (query blocks that mark different key blocks
inside one 256-row work item, masks wider than one 32-bit word, shared and
per-head masks, all three causal modes), the all-ones mask (identical to the
dense kernel) and the empty mask (every row without keys).
"""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_06_gb300 import ops
from attention_forward_06_gb300.inputs import bf16_bits, draw, sample_rows
from parity_util import compare

pytestmark = pytest.mark.gpu
BLK = 128


def words_for(blocks: np.ndarray) -> np.ndarray:
    """bool [B, H, QB, KB] -> uint32 words [B, H, QB, ceil(KB/32)] (test-side packing)."""
    B, H, QB, KB = blocks.shape
    w = np.zeros((B, H, QB, (KB + 31) // 32), np.uint32)
    for kb in range(KB):
        w[..., kb // 32] |= blocks[..., kb].astype(np.uint32) << np.uint32(kb % 32)
    return w


def run(q, k, v, words, causal, scale):
    m = torch.from_numpy(words.view(np.int32)).cuda()
    o, lse = ops.attn_fwd_blocksparse(q.cuda(), k.cuda(), v.cuda(), m, causal=causal, scale=scale)
    st, site = ops.debug_status()
    assert st == ops.ATTN_OK, f"kernel wait ran out at site {site}"
    return o.cpu(), lse.cpu()


CASES = [
    # B, Hq, Hkv, Sq, Sk, D, causal, mask heads, density
    (1, 4, 2, 300, 700, 128, 1, 1, 0.5),
    (2, 4, 4, 513, 513, 64, 0, 4, 0.4),
    (1, 2, 1, 1000, 129, 128, 1, 2, 0.6),      # Sq > Sk bottom-right: rows without keys
    (1, 8, 2, 256, 2048, 128, 2, 8, 0.3),
    (1, 2, 2, 640, 5000, 64, 0, 1, 0.5),       # 40 key blocks: two words per mask row
    (1, 3, 1, 777, 4500, 128, 1, 3, 0.15),     # sparse, ragged everywhere
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_random_masks_match_oracle(case):
    B, Hq, Hkv, Sq, Sk, D, causal, Hm, density = case
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, D, seed=sum(case[:7]))
    rng = np.random.default_rng(Sq + Sk)
    blocks = rng.random((B, Hm, -(-Sq // BLK), -(-Sk // BLK))) < density
    words = words_for(blocks)
    scale = float(np.float32(D ** -0.5))
    o, lse = run(q, k, v, words, causal, scale)
    o_ref, lse_ref = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal, scale, block_mask=words)
    compare(o, lse, o_ref, lse_ref)


def test_query_blocks_of_one_item_mark_different_key_blocks():
    # rows 0-127 and 128-255 form one work item; they mark disjoint key blocks
    Sq, Sk, D = 256, 1024, 128
    q, k, v = draw(1, 2, 1, Sq, Sk, D, seed=21)
    blocks = np.zeros((1, 1, 2, 8), bool)
    blocks[0, 0, 0, [0, 3, 5]] = True
    blocks[0, 0, 1, [1, 2, 7]] = True
    words = words_for(blocks)
    o, lse = run(q, k, v, words, 0, 0.088)
    o_ref, lse_ref = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 0, 0.088, block_mask=words)
    compare(o, lse, o_ref, lse_ref)


def test_all_ones_mask_equals_dense_kernel_bitwise():
    q, k, v = draw(2, 4, 2, 700, 900, 128, seed=23)
    words = words_for(np.ones((2, 1, 6, 8), bool))
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    for causal in (0, 1, 2):
        o1, l1 = ops.attn_fwd(qd, kd, vd, causal=causal)
        o2, l2 = ops.attn_fwd_blocksparse(qd, kd, vd, torch.from_numpy(words.view(np.int32)).cuda(), causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_empty_mask_gives_zero_rows():
    q, k, v = draw(1, 2, 2, 300, 400, 64, seed=25)
    words = words_for(np.zeros((1, 1, 3, 4), bool))
    o, lse = run(q, k, v, words, 0, 0.125)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_long_sparse_on_sampled_rows():
    # 16k x 16k causal with a quarter of the blocks marked (diagonal blocks always kept)
    B, Hq, Hkv, S, D = 1, 8, 2, 16384, 128
    q, k, v = draw(B, Hq, Hkv, S, S, D, seed=27)
    rng = np.random.default_rng(27)
    blocks = rng.random((B, Hq, S // BLK, S // BLK)) < 0.25
    idx = np.arange(S // BLK)
    blocks[:, :, idx, idx] = True
    words = words_for(blocks)
    scale = float(np.float32(D ** -0.5))
    o, lse = run(q, k, v, words, 1, scale)
    rows = sample_rows(B, Hq, S, 16, seed=28)
    o_ref, lse_ref = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 1, scale, rows=rows, block_mask=words)
    compare(o.reshape(-1, D)[torch.from_numpy(rows)], lse.reshape(-1)[torch.from_numpy(rows)], o_ref, lse_ref)


def test_pack_block_mask_matches_test_packing():
    rng = np.random.default_rng(29)
    blocks = rng.random((2, 3, 5, 70)) < 0.5
    ref = words_for(blocks)
    got = ops.pack_block_mask(torch.from_numpy(blocks).cuda()).cpu().numpy().view(np.uint32)
    assert np.array_equal(ref, got)
