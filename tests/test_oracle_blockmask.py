"""Pins for the oracle's bit-packed block mask (CPU only).

Definition pinned: the keys a query row may attend to are the causally allowed
ones that also fall in a key block its query block's mask row marks -- one bit
per (query block, key block), 32 blocks per 32-bit word (page "AdaSplash-2:
Faster Differentiable Sparse Attention", technical summary section 2, bit-packed
block masking).  The expansion of the words into an element mask below is
written independently of the oracle (numpy bit arithmetic), and the attention
over that element mask is taken from torch's fp64 scaled_dot_product_attention,
a library routine; so a wrong word or bit order, a wrong head or block index, or
the mask applied with OR instead of AND to the causal limit fails here.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_06_gb300.inputs import bf16_bits, draw


def words_per_row(Sk, bk):
    return ((Sk + bk - 1) // bk + 31) // 32


def random_mask(B, Hm, Sq, Sk, bq, bk, density, seed):
    rng = np.random.default_rng(seed)
    QB, KB = -(-Sq // bq), -(-Sk // bk)
    bitsel = rng.random((B, Hm, QB, KB)) < density
    w = np.zeros((B, Hm, QB, words_per_row(Sk, bk)), np.uint32)
    for kb in range(KB):
        w[..., kb // 32] |= (bitsel[..., kb].astype(np.uint32) << np.uint32(kb % 32))
    return w, bitsel


def element_mask(words, b, h, Sq, Sk, bq, bk, causal):
    """Boolean [Sq, Sk]: causally allowed AND in a marked block (independent of the oracle)."""
    hm = 0 if words.shape[1] == 1 else h
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    kb = j // bk
    w = words[b, hm][i // bq, kb // 32]
    inblock = ((w >> (kb % 32).astype(np.uint32)) & 1).astype(bool)
    if causal == 0:
        allowed = np.ones((Sq, Sk), bool)
    elif causal == 1:
        allowed = j <= i + (Sk - Sq)
    else:
        allowed = j <= i
    return inblock & allowed


def sdpa_masked(q, k, v, emask, scale):
    """torch fp64 attention over an element mask; rows without any key: O = 0, LSE = -inf."""
    qd, kd, vd = q.double(), k.double(), v.double()
    s = (qd @ kd.transpose(-1, -2)) * scale
    s = s.masked_fill(~torch.from_numpy(emask), float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    dead = torch.isinf(lse) & (lse < 0)
    o = torch.nn.functional.scaled_dot_product_attention(qd[None, None], kd[None, None], vd[None, None],
                                                         attn_mask=torch.from_numpy(emask)[None, None],
                                                         scale=scale)[0, 0]
    o = torch.where(dead[:, None], torch.zeros_like(o), o)
    return o.numpy(), lse.numpy()


@pytest.mark.parametrize("causal", [0, 1, 2])
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,bq,bk,Hm,density", [
    (1, 2, 1, 70, 90, 16, 16, 16, 1, 0.5),
    (2, 4, 2, 65, 130, 8, 32, 8, 4, 0.4),     # more than 32 key blocks: two words per row
    (1, 3, 3, 40, 300, 8, 8, 8, 3, 0.2),      # ten words per row, sparse
])
def test_block_mask_against_library_attention(causal, B, Hq, Hkv, Sq, Sk, D, bq, bk, Hm, density):
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, D, seed=Sq + Sk + causal)
    scale = float(np.float32(D ** -0.5))
    words, _ = random_mask(B, Hm, Sq, Sk, bq, bk, density, seed=Sk + causal)
    o, lse = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal, scale, block_mask=words,
                              block=(bq, bk))
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            em = element_mask(words, b, h, Sq, Sk, bq, bk, causal)
            o_ref, l_ref = sdpa_masked(q[b, h], k[b, h // G], v[b, h // G], em, scale)
            np.testing.assert_allclose(o[b, h], o_ref, rtol=0, atol=1e-12)
            np.testing.assert_array_equal(np.isneginf(lse[b, h]), np.isneginf(l_ref))
            live = ~np.isneginf(l_ref)
            np.testing.assert_allclose(lse[b, h][live], l_ref[live], rtol=0, atol=1e-12)


def test_all_ones_mask_equals_unmasked():
    q, k, v = draw(2, 4, 2, 300, 500, 32, seed=3)
    scale = 0.2
    words = np.full((2, 1, 3, words_per_row(500, 128)), 0xFFFFFFFF, np.uint32)
    for causal in (0, 1, 2):
        o1, l1 = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal, scale)
        o2, l2 = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal, scale, block_mask=words)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_block_diagonal_mask_equals_independent_segments():
    # query block t sees only key block t: attention decomposes into independent segments
    S, D, blk = 96, 16, 32
    q, k, v = draw(1, 1, 1, S, S, D, seed=5)
    words = np.zeros((1, 1, S // blk, 1), np.uint32)
    for t in range(S // blk):
        words[0, 0, t, 0] = np.uint32(1 << t)
    o, lse = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 0, 0.25, block_mask=words, block=(blk, blk))
    for t in range(S // blk):
        sl = slice(t * blk, (t + 1) * blk)
        o_seg, l_seg = oracle.attention(bf16_bits(q[:, :, sl]), bf16_bits(k[:, :, sl]), bf16_bits(v[:, :, sl]), 0, 0.25)
        np.testing.assert_allclose(o[0, 0, sl], o_seg[0, 0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[0, 0, sl], l_seg[0, 0], rtol=0, atol=1e-13)


def test_empty_mask_row_gives_zero_and_minus_infinity():
    q, k, v = draw(1, 2, 2, 64, 64, 16, seed=7)
    words = np.full((1, 2, 2, 1), 0xFFFFFFFF, np.uint32)
    words[0, 1, 1, 0] = 0  # head 1, second query block: no key block
    o, lse = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 0, 0.25, block_mask=words, block=(32, 32))
    assert np.all(o[0, 1, 32:] == 0.0) and np.all(np.isneginf(lse[0, 1, 32:]))
    assert np.all(np.isfinite(lse[0, 0])) and np.all(np.isfinite(lse[0, 1, :32]))


def test_bits_past_the_last_key_block_are_ignored():
    q, k, v = draw(1, 1, 1, 40, 40, 8, seed=9)
    base = np.array([[[[0b101]]]], np.uint32)       # 40 keys in blocks of 16: blocks 0, 1, 2; marks 0 and 2
    padded = base | np.uint32(0xFFFFFFF8)             # bits 3..31 name no key block
    o1, l1 = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 0, 0.3, block_mask=base, block=(64, 16))
    o2, l2 = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 0, 0.3, block_mask=padded, block=(64, 16))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_shared_mask_equals_the_same_mask_per_head():
    q, k, v = draw(2, 4, 1, 100, 200, 16, seed=11)
    shared, _ = random_mask(2, 1, 100, 200, 32, 32, 0.5, seed=12)
    per_head = np.repeat(shared, 4, axis=1)
    o1, l1 = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 1, 0.25, block_mask=shared, block=(32, 32))
    o2, l2 = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 1, 0.25, block_mask=per_head, block=(32, 32))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_mask_and_causal_limit_combine_as_and_not_or():
    # a mask that marks only key blocks above the diagonal leaves a causal run with no key at all
    S, blk = 64, 16
    q, k, v = draw(1, 1, 1, S, S, 8, seed=13)
    words = np.zeros((1, 1, S // blk, 1), np.uint32)
    for t in range(S // blk - 1):
        words[0, 0, t, 0] = np.uint32(1 << (t + 1))  # query block t marks key block t+1 only
    o, lse = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 2, 0.3, block_mask=words, block=(blk, blk))
    assert np.all(np.isneginf(lse[0, 0])) and np.all(o == 0.0)


def test_bad_block_mask_shapes_are_rejected():
    q, k, v = draw(1, 2, 1, 64, 64, 8, seed=15)
    with pytest.raises(ValueError):
        oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 0, 0.3,
                         block_mask=np.zeros((1, 3, 1, 1), np.uint32))  # heads must be 1 or Hq
    with pytest.raises(ValueError):
        oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 0, 0.3,
                         block_mask=np.zeros((1, 1, 2, 1), np.uint32))  # 64 rows are one block of 128
