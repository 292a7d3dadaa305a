"""Pins for the oracle's backward (CPU only).

Definition pinned: the gradients of the forward's O = softmax(scale Q K^T + mask) V
with respect to Q, K and V for an upstream gradient dO (the loss sum(O * dO)), the
forward being the closed-form-normalised softmax attention of page "AdaSplash-2:
Faster Differentiable Sparse Attention" (technical summary section 1).  The pins
use torch's fp64 autograd through scaled_dot_product_attention (a library
routine), central finite differences of an independent numpy forward, and closed
forms of the softmax Jacobian (every row's dS sums to zero, so sum_j dK_j = 0;
sum_j P_ij = 1, so sum_j dV_j = sum_i dO_i); a dropped term, a wrong sign, a
missing scale or a wrong head map in the oracle fails one of them.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_06_gb300.inputs import bf16_bits, draw, from_values


def allowed(Sq, Sk, causal):
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    if causal == 0:
        return np.ones((Sq, Sk), bool)
    return j <= i + (Sk - Sq) if causal == 1 else j <= i


def torch_grads(q, k, v, do, causal, scale):
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    G = Hq // Hkv
    qd, kd, vd = (t.double().requires_grad_(True) for t in (q, k, v))
    mask = torch.from_numpy(allowed(Sq, Sk, causal))
    o = torch.nn.functional.scaled_dot_product_attention(qd, kd.repeat_interleave(G, 1), vd.repeat_interleave(G, 1),
                                                         attn_mask=mask, scale=scale)
    (o * do.double()).sum().backward()
    return qd.grad.numpy(), kd.grad.numpy(), vd.grad.numpy()


@pytest.mark.parametrize("causal", [0, 1, 2])
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D", [(1, 1, 1, 17, 17, 8), (2, 4, 2, 33, 50, 16), (1, 6, 3, 40, 40, 8)])
def test_against_torch_autograd(causal, B, Hq, Hkv, Sq, Sk, D):
    if causal == 2 and Sq > Sk:
        pytest.skip("rows without keys make torch's attention NaN; covered separately")
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, D, seed=Sq + Sk + causal)
    do = draw(B, Hq, Hkv, Sq, Sk, D, seed=99 + causal)[0]
    scale = float(np.float32(D ** -0.5))
    dq, dk, dv = oracle.backward(bf16_bits(q), bf16_bits(k), bf16_bits(v), bf16_bits(do), causal, scale)
    tq, tk, tv = torch_grads(q, k, v, do, causal, scale)
    for a, b in ((dq, tq), (dk, tk), (dv, tv)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)


def numpy_loss(q, k, v, do, causal, scale):
    """sum(O * dO) from an explicit fp64 softmax (independent of the oracle and of torch)."""
    G = q.shape[1] // k.shape[1]
    total = 0.0
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            s = scale * q[b, h] @ k[b, h // G].T
            s = np.where(allowed(q.shape[2], k.shape[2], causal), s, -np.inf)
            p = np.exp(s - s.max(1, keepdims=True))
            p /= p.sum(1, keepdims=True)
            total += float(((p @ v[b, h // G]) * do[b, h]).sum())
    return total


def test_central_differences_of_an_independent_forward():
    B, Hq, Hkv, Sq, Sk, D, causal = 1, 2, 1, 12, 15, 8, 1
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, D, seed=3)
    do = draw(B, Hq, Hkv, Sq, Sk, D, seed=4)[0]
    scale = 0.35
    dq, dk, dv = oracle.backward(bf16_bits(q), bf16_bits(k), bf16_bits(v), bf16_bits(do), causal, scale)
    arrs = [t.double().numpy().copy() for t in (q, k, v)]
    dod = do.double().numpy()
    rng = np.random.default_rng(5)
    eps = 1e-6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        for _ in range(6):
            idx = tuple(rng.integers(0, n) for n in arrs[which].shape)
            plus = [a.copy() for a in arrs]
            minus = [a.copy() for a in arrs]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            fd = (numpy_loss(*plus, dod, causal, scale) - numpy_loss(*minus, dod, causal, scale)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (which, idx, fd, grad[idx])


@pytest.mark.parametrize("causal", [0, 1, 2])
def test_key_gradients_sum_to_zero_and_value_gradients_to_the_output_gradient(causal):
    B, Hq, Hkv, S, D = 2, 4, 2, 48, 16
    q, k, v = draw(B, Hq, Hkv, S, S, D, seed=7 + causal)
    do = draw(B, Hq, Hkv, S, S, D, seed=8)[0]
    dq, dk, dv = oracle.backward(bf16_bits(q), bf16_bits(k), bf16_bits(v), bf16_bits(do), causal, 0.25)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-11)
    G = Hq // Hkv
    dod = do.double().numpy().reshape(B, Hkv, G, S, D).sum(axis=(2, 3))
    np.testing.assert_allclose(dv.sum(axis=2), dod, atol=1e-11)


def test_query_gradient_ignores_a_common_key_shift():
    # integer-valued keys so that k + 1 is exact in bf16; without a mask every row sees every key
    rng = np.random.default_rng(9)
    S, D = 20, 8
    q = from_values(rng.normal(0, 0.3, (1, 1, S, D)))
    k = from_values(rng.integers(-3, 4, (1, 1, S, D)).astype(np.float64))
    k1 = from_values(k.double().numpy() + 1.0)
    v = from_values(rng.normal(0, 1, (1, 1, S, D)))
    do = from_values(rng.normal(0, 1, (1, 1, S, D)))
    dq0 = oracle.backward(bf16_bits(q), bf16_bits(k), bf16_bits(v), bf16_bits(do), 0, 0.3)[0]
    dq1 = oracle.backward(bf16_bits(q), bf16_bits(k1), bf16_bits(v), bf16_bits(do), 0, 0.3)[0]
    np.testing.assert_allclose(dq0, dq1, rtol=0, atol=1e-12)


def test_grouped_heads_sum_the_gradients_of_their_query_heads():
    B, Hq, Hkv, S, D = 1, 4, 1, 30, 8
    q, k, v = draw(B, Hq, Hkv, S, S, D, seed=11)
    do = draw(B, Hq, Hkv, S, S, D, seed=12)[0]
    dq, dk, dv = oracle.backward(bf16_bits(q), bf16_bits(k), bf16_bits(v), bf16_bits(do), 1, 0.3)
    kr, vr = k.repeat_interleave(Hq, 1), v.repeat_interleave(Hq, 1)
    dq2, dk2, dv2 = oracle.backward(bf16_bits(q), bf16_bits(kr), bf16_bits(vr), bf16_bits(do), 1, 0.3)
    np.testing.assert_allclose(dq, dq2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk, dk2.sum(axis=1, keepdims=True), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, dv2.sum(axis=1, keepdims=True), rtol=0, atol=1e-12)


def test_rows_without_keys_have_no_gradient():
    # bottom-right with Sq > Sk: the first Sq - Sk rows see no key
    q, k, v = draw(1, 2, 1, 40, 25, 8, seed=13)
    do = draw(1, 2, 1, 40, 25, 8, seed=14)[0]
    dq, dk, dv = oracle.backward(bf16_bits(q), bf16_bits(k), bf16_bits(v), bf16_bits(do), 1, 0.3)
    assert np.all(dq[:, :, :15] == 0.0)
    q2, do2 = q[:, :, 15:].contiguous(), do[:, :, 15:].contiguous()
    dq2, dk2, dv2 = oracle.backward(bf16_bits(q2), bf16_bits(k), bf16_bits(v), bf16_bits(do2), 1, 0.3)
    np.testing.assert_allclose(dq[:, :, 15:], dq2, atol=1e-13)
    np.testing.assert_allclose(dk, dk2, atol=1e-13)
    np.testing.assert_allclose(dv, dv2, atol=1e-13)
