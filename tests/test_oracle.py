"""Pins for the fp64 oracle (CPU only; no GPU, no CUDA library).

Each test fixes the oracle to something other than itself: a hand-derived worked
example, a closed form, an invariant of the definition, a library routine, or
50-digit arithmetic.  The set is chosen so that a plausible slip in the oracle --
a dropped normaliser, a wrong sign, a transposed operand, a wrong kv-head index,
an off-by-one in the causal limit -- fails at least one of them.

Definition pinned: softmax attention with its closed-form log-sum-exp normaliser
(page "AdaSplash-2: Faster Differentiable Sparse Attention", technical summary
section 1), O = softmax(scale * Q K^T + mask) V, LSE = ln sum exp(scale * q.k).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from attention_forward_06_gb300.inputs import bf16_bits, draw, from_values, sample_rows

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form.json")


def bits(values):
    return bf16_bits(from_values(values))


def decode(b):
    """bf16 bit patterns -> float64 (via torch, independent of the oracle's decoder)."""
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).double().numpy()


def allowed_mask(Sq, Sk, causal):
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    if causal == 0:
        return np.ones((Sq, Sk), bool)
    if causal == 1:
        return j <= i + (Sk - Sq)
    return j <= i


# ---------------------------------------------------------------- worked examples
def closed_form_o(text):
    from fractions import Fraction
    return float(Fraction(text))


def closed_form_lse(text):
    """'-inf', '0', 'ln n' or 'k ln 2'."""
    text = text.strip()
    if text == "-inf":
        return -math.inf
    parts = text.split()
    if parts == ["0"]:
        return 0.0
    if len(parts) == 2 and parts[0] == "ln":
        return math.log(int(parts[1]))
    if len(parts) == 3 and parts[1] == "ln":
        return int(parts[0]) * math.log(int(parts[2]))
    raise ValueError(text)


def test_golden_closed_forms():
    spec = json.load(open(GOLDEN))
    scale, tol = spec["scale"], spec["tolerance"]
    assert np.float32(scale) == np.float32(math.log(2.0))
    for case in spec["cases"]:
        q = bits(case["q"])[None]
        k = bits(case["k"])[None]
        v = bits(case["v"])[None]
        o, lse = oracle.attention(q, k, v, case["causal"], scale)
        exp_o = np.vectorize(closed_form_o, otypes=[np.float64])(np.array(case["o"]))[None]
        exp_lse = np.vectorize(closed_form_lse, otypes=[np.float64])(np.array(case["lse"]))[None]
        np.testing.assert_allclose(o, exp_o, rtol=0, atol=tol, err_msg=case["name"])
        finite = np.isfinite(exp_lse)
        np.testing.assert_allclose(lse[finite], exp_lse[finite], rtol=0, atol=tol, err_msg=case["name"])
        assert np.all(np.isneginf(lse[~finite])), case["name"]


# ---------------------------------------------------------------- normalisation
@pytest.mark.parametrize("causal", [0, 1, 2])
@pytest.mark.parametrize("Sq,Sk", [(7, 7), (5, 13), (13, 5), (1, 1), (16, 31)])
def test_probabilities_rows_sum_to_one(causal, Sq, Sk):
    q, k, v = draw(1, 1, 1, Sq, Sk, 8, seed=11 + Sq * 31 + Sk)
    p, o, lse = oracle.probabilities(bf16_bits(q[0, 0]), bf16_bits(k[0, 0]), bf16_bits(v[0, 0]), causal, 0.3)
    allowed = allowed_mask(Sq, Sk, causal)
    has_key = allowed.any(axis=1)
    np.testing.assert_allclose(p.sum(axis=1)[has_key], 1.0, rtol=0, atol=1e-12)
    assert np.all(p[~allowed] == 0.0)
    assert np.all(p[allowed] > 0.0)
    # O is exactly the P-weighted sum of V rows
    np.testing.assert_allclose(o, p @ decode(bf16_bits(v[0, 0])), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("causal", [0, 1, 2])
def test_identical_keys_give_mean_of_allowed_values(causal):
    Sq, Sk, D = 9, 12, 16
    q, _, v = draw(1, 1, 1, Sq, Sk, D, seed=3)
    krow = draw(1, 1, 1, 1, 1, D, seed=4)[1][0, 0, 0]
    k = krow.expand(1, 1, Sk, D).contiguous()
    scale = 0.25
    o, lse = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal, scale)
    qd, kd, vd = decode(bf16_bits(q))[0, 0], decode(bf16_bits(krow)), decode(bf16_bits(v))[0, 0]
    allowed = allowed_mask(Sq, Sk, causal)
    for i in range(Sq):
        n = allowed[i].sum()
        if n == 0:
            assert np.all(o[0, 0, i] == 0) and np.isneginf(lse[0, 0, i])
            continue
        np.testing.assert_allclose(o[0, 0, i], vd[allowed[i]].mean(axis=0), rtol=0, atol=1e-12)
        s = float(np.float32(scale)) * float(qd[i] @ kd)
        np.testing.assert_allclose(lse[0, 0, i], s + math.log(n), rtol=0, atol=1e-12)


def test_one_hot_dominant_logit_returns_that_value_row():
    # q_i = 32 e0, k_{j*} = 32 e0, every other key 0: logit gap 1024*scale >= 90.
    Sq, Sk, D = 4, 40, 64
    scale = float(np.float32(1 / math.sqrt(D)))
    for jstar in (0, 17, Sk - 1):
        q = np.zeros((Sq, D), np.float32); q[:, 0] = 32.0
        k = np.zeros((Sk, D), np.float32); k[jstar, 0] = 32.0
        v = draw(1, 1, 1, 1, Sk, D, seed=5 + jstar)[2]
        o, lse = oracle.attention(bits(q)[None, None], bits(k)[None, None], bf16_bits(v), 0, scale)
        vd = decode(bf16_bits(v))[0, 0]
        for i in range(Sq):
            np.testing.assert_allclose(o[0, 0, i], vd[jstar], rtol=0, atol=1e-30)
            gap = 1024.0 * scale
            expect = gap + math.log1p((Sk - 1) * math.exp(-gap))
            np.testing.assert_allclose(lse[0, 0, i], expect, rtol=0, atol=1e-12)


def test_causal_row_zero_returns_first_value_row():
    q, k, v = draw(2, 3, 3, 33, 33, 32, seed=6)
    scale = 0.17
    for causal in (1, 2):
        o, lse = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal, scale)
        qd, kd, vd = decode(bf16_bits(q)), decode(bf16_bits(k)), decode(bf16_bits(v))
        np.testing.assert_allclose(o[:, :, 0], vd[:, :, 0], rtol=0, atol=1e-14)
        s00 = float(np.float32(scale)) * np.einsum("bhd,bhd->bh", qd[:, :, 0], kd[:, :, 0])
        np.testing.assert_allclose(lse[:, :, 0], s00, rtol=0, atol=1e-12)


def test_bottom_right_row_zero_sees_sk_minus_sq_plus_one_keys():
    Sq, Sk, D = 6, 20, 16
    q, k, v = draw(1, 1, 1, Sq, Sk, D, seed=7)
    o1, l1 = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 1, 0.2)
    # changing value rows beyond the limit of row 0 leaves row 0 alone, and changes row 0
    # when the last allowed row (Sk - Sq) changes
    v2 = v.clone(); v2[0, 0, Sk - Sq + 1:] = 3.0
    o2, _ = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v2), 1, 0.2)
    np.testing.assert_array_equal(o1[0, 0, 0], o2[0, 0, 0])
    v3 = v.clone(); v3[0, 0, Sk - Sq] += 1.0
    o3, _ = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v3), 1, 0.2)
    assert np.abs(o3[0, 0, 0] - o1[0, 0, 0]).max() > 1e-6
    # identical keys: row i sees exactly Sk - Sq + 1 + i keys
    kk = k[:, :, :1].expand(1, 1, Sk, D).contiguous()
    _, lse = oracle.attention(bf16_bits(q), bf16_bits(kk), bf16_bits(v), 1, 0.2)
    s = float(np.float32(0.2)) * (decode(bf16_bits(q))[0, 0] @ decode(bf16_bits(kk))[0, 0, 0])
    np.testing.assert_allclose(lse[0, 0], s + np.log(Sk - Sq + 1 + np.arange(Sq)), rtol=0, atol=1e-12)


def test_fully_masked_rows_are_zero_with_minus_infinite_lse():
    Sq, Sk = 10, 4
    q, k, v = draw(1, 2, 1, Sq, Sk, 8, seed=8)
    o, lse = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 1, 0.3)
    dead = Sq - Sk  # rows 0 .. Sq-Sk-1 have no key at bottom-right alignment
    assert np.all(o[:, :, :dead] == 0.0)
    assert np.all(np.isneginf(lse[:, :, :dead]))
    assert np.all(np.isfinite(lse[:, :, dead:]))


# ---------------------------------------------------------------- high precision
def test_lse_matches_50_digit_log_sum_exp():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    Sq, Sk, D = 5, 9, 8
    q, k, v = draw(1, 1, 1, Sq, Sk, D, seed=9, qk_std=2.0)
    scale = 0.35
    o, lse = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 1, scale)
    qd, kd, vd = decode(bf16_bits(q))[0, 0], decode(bf16_bits(k))[0, 0], decode(bf16_bits(v))[0, 0]
    sc = mpmath.mpf(float(np.float32(scale)))
    for i in range(Sq):
        n = i + Sk - Sq + 1
        logits = [sc * mpmath.fsum(mpmath.mpf(float(qd[i, d])) * mpmath.mpf(float(kd[j, d])) for d in range(D))
                  for j in range(n)]
        z = mpmath.fsum(mpmath.exp(x) for x in logits)
        assert abs(float(mpmath.log(z)) - lse[0, 0, i]) < 1e-12
        for d in range(D):
            od = mpmath.fsum(mpmath.exp(logits[j]) * mpmath.mpf(float(vd[j, d])) for j in range(n)) / z
            assert abs(float(od) - o[0, 0, i, d]) < 1e-12


# ---------------------------------------------------------------- library routines
@pytest.mark.parametrize("causal", [0, 1, 2])
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D", [
    (1, 1, 1, 17, 17, 16), (2, 4, 2, 13, 29, 32), (1, 8, 2, 32, 20, 64), (2, 2, 1, 1, 64, 8)])
def test_brute_force_against_torch_sdpa_fp64(causal, B, Hq, Hkv, Sq, Sk, D):
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, D, seed=10 + Sq + Sk + D)
    scale = float(np.float32(1 / math.sqrt(D)))
    o, lse = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal, scale)
    allowed = torch.from_numpy(allowed_mask(Sq, Sk, causal))
    live = allowed.any(dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.double(), k.double(), v.double(), attn_mask=allowed, scale=scale, enable_gqa=(Hq != Hkv))
    np.testing.assert_allclose(o[:, :, live.numpy()], ref[:, :, live].numpy(), rtol=0, atol=1e-12)
    G = Hq // Hkv
    logits = torch.einsum("bhid,bhjd->bhij", q.double(), k.double().repeat_interleave(G, dim=1)) * scale
    ref_lse = torch.logsumexp(logits.masked_fill(~allowed, -math.inf), dim=-1)
    np.testing.assert_allclose(lse[:, :, live.numpy()], ref_lse[:, :, live].numpy(), rtol=0, atol=1e-12)


def test_brute_force_against_numpy_softmax_matrix():
    Sq, Sk, D = 24, 40, 32
    q, k, v = draw(1, 1, 1, Sq, Sk, D, seed=12, qk_std=2.5)
    scale = 0.125
    p, o, lse = oracle.probabilities(bf16_bits(q[0, 0]), bf16_bits(k[0, 0]), bf16_bits(v[0, 0]), 1, scale)
    qd, kd, vd = decode(bf16_bits(q))[0, 0], decode(bf16_bits(k))[0, 0], decode(bf16_bits(v))[0, 0]
    s = np.where(allowed_mask(Sq, Sk, 1), float(np.float32(scale)) * qd @ kd.T, -np.inf)
    e = np.exp(s - s.max(axis=1, keepdims=True))
    pm = e / e.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(p, pm, rtol=0, atol=1e-13)
    np.testing.assert_allclose(o, pm @ vd, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- structural identities
def test_gqa_equals_mha_with_repeated_kv_heads():
    B, Hq, Hkv, Sq, Sk, D = 2, 8, 2, 19, 23, 16
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, D, seed=13)
    G = Hq // Hkv
    o1, l1 = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 1, 0.25)
    kr, vr = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
    o2, l2 = oracle.attention(bf16_bits(q), bf16_bits(kr), bf16_bits(vr), 1, 0.25)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    # and the head map is contiguous groups: head h reads kv head h // G, not h % Hkv
    o3, _ = oracle.attention(bf16_bits(q), bf16_bits(k.repeat(1, G, 1, 1)), bf16_bits(v.repeat(1, G, 1, 1)), 1, 0.25)
    assert np.abs(o3 - o1).max() > 1e-3


def test_bottom_right_equals_tail_of_square_causal_run():
    Sq, Sk, D = 16, 48, 16
    q, k, v = draw(1, 2, 2, Sk, Sk, D, seed=14)
    o_full, l_full = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 1, 0.2)
    qt = q[:, :, Sk - Sq:].contiguous()
    o_c, l_c = oracle.attention(bf16_bits(qt), bf16_bits(k), bf16_bits(v), 1, 0.2)
    np.testing.assert_array_equal(o_c, o_full[:, :, Sk - Sq:])
    np.testing.assert_array_equal(l_c, l_full[:, :, Sk - Sq:])


def test_split_keys_and_merge_by_lse_equals_full():
    Sq, Sk, D = 11, 30, 16
    q, k, v = draw(1, 1, 1, Sq, Sk, D, seed=15)
    o, lse = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 0, 0.3)
    h = 13
    parts = [oracle.attention(bf16_bits(q), bf16_bits(k[:, :, a:b].contiguous()),
                              bf16_bits(v[:, :, a:b].contiguous()), 0, 0.3) for a, b in ((0, h), (h, Sk))]
    lse_m = np.logaddexp(parts[0][1], parts[1][1])
    o_m = sum(np.exp(lp - lse_m)[..., None] * op for op, lp in parts)
    np.testing.assert_allclose(lse_m, lse, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o_m, o, rtol=0, atol=1e-12)


def test_value_linearity():
    Sq, Sk, D = 8, 21, 16
    q, k, _ = draw(1, 1, 1, Sq, Sk, D, seed=16)
    rng = np.random.default_rng(0)
    v1 = rng.integers(-8, 9, size=(1, 1, Sk, D)).astype(np.float32)
    v2 = rng.integers(-8, 9, size=(1, 1, Sk, D)).astype(np.float32)
    comb = 3 * v1 - 2 * v2  # integers below 256: exact in bf16
    oa, _ = oracle.attention(bf16_bits(q), bf16_bits(k), bits(v1), 1, 0.4)
    ob, _ = oracle.attention(bf16_bits(q), bf16_bits(k), bits(v2), 1, 0.4)
    oc, _ = oracle.attention(bf16_bits(q), bf16_bits(k), bits(comb), 1, 0.4)
    np.testing.assert_allclose(oc, 3 * oa - 2 * ob, rtol=0, atol=1e-12)


def test_joint_key_value_permutation_invariance_without_mask():
    Sq, Sk, D = 9, 25, 16
    q, k, v = draw(1, 1, 1, Sq, Sk, D, seed=17)
    perm = torch.from_numpy(np.random.default_rng(1).permutation(Sk))
    o1, l1 = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 0, 0.3)
    o2, l2 = oracle.attention(bf16_bits(q), bf16_bits(k[:, :, perm].contiguous()),
                              bf16_bits(v[:, :, perm].contiguous()), 0, 0.3)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-13)
    # with a causal mask the order matters
    o3, _ = oracle.attention(bf16_bits(q), bf16_bits(k[:, :, perm].contiguous()),
                             bf16_bits(v[:, :, perm].contiguous()), 1, 0.3)
    o4, _ = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 1, 0.3)
    assert np.abs(o3 - o4).max() > 1e-3


def test_key_shift_leaves_output_and_shifts_lse_by_scaled_query_sum():
    Sq, Sk, D = 7, 19, 16
    rng = np.random.default_rng(2)
    q = rng.integers(-16, 17, size=(1, 1, Sq, D)).astype(np.float32) / 8
    k = rng.integers(-16, 17, size=(1, 1, Sk, D)).astype(np.float32) / 8
    v = draw(1, 1, 1, 1, Sk, D, seed=18)[2]
    c = 1.0  # k + c stays exact in bf16
    scale = 0.25
    o1, l1 = oracle.attention(bits(q), bits(k), bf16_bits(v), 1, scale)
    o2, l2 = oracle.attention(bits(q), bits(k + c), bf16_bits(v), 1, scale)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1 + scale * c * q.sum(axis=-1), rtol=0, atol=1e-12)


def test_scale_is_applied_inside_the_exponent():
    # doubling q is the same as doubling scale; a scale left out (or applied to O) fails this
    Sq, Sk, D = 6, 10, 8
    q, k, v = draw(1, 1, 1, Sq, Sk, D, seed=19)
    o1, l1 = oracle.attention(bf16_bits(q * 2), bf16_bits(k), bf16_bits(v), 0, 0.25)
    o2, l2 = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 0, 0.5)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


# ---------------------------------------------------------------- modes and edges
def test_row_subset_matches_full_rows():
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 40, 40, 16
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, D, seed=20)
    o, lse = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 1, 0.25)
    rows = sample_rows(B, Hq, Sq, 6, seed=21)
    assert len(np.unique(rows)) == len(rows)
    for bh in range(B * Hq):  # rows 0 and Sq-1 of every head are present
        assert bh * Sq in rows and bh * Sq + Sq - 1 in rows
    os_, ls_ = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 1, 0.25, rows=rows)
    np.testing.assert_array_equal(os_, o.reshape(-1, D)[rows])
    np.testing.assert_array_equal(ls_, lse.reshape(-1)[rows])


def test_empty_inputs():
    q, k, v = draw(1, 1, 1, 0, 5, 8, seed=22)
    o, lse = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 0, 0.3)
    assert o.shape == (1, 1, 0, 8) and lse.shape == (1, 1, 0)
    q, k, v = draw(1, 1, 1, 3, 0, 8, seed=23)
    o, lse = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 0, 0.3)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_bad_arguments_are_rejected():
    q, k, v = draw(1, 3, 2, 4, 4, 8, seed=24)
    with pytest.raises(ValueError):
        oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 0, 0.3)  # Hq % Hkv != 0
    q, k, v = draw(1, 2, 2, 4, 4, 8, seed=24)
    with pytest.raises(ValueError):
        oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 3, 0.3)
    with pytest.raises(ValueError):
        oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 0, 0.3, rows=[999])
