"""Parity of the backward (attn_bwd, through the C ABI) with the fp64 oracle's
backward, element by element on seeded inputs, over ragged shapes, the three
causal modes, grouped heads, D = 64 and 128, rows without keys and keys no row
sees, and the training-prefill workload at full size.

Tolerance (derived from the arithmetic; the task states none for gradients):
the kernels round P and dS to bf16 before the products that use them (relative
error 2^-9 per term), form D_i from the bf16 O, and round each gradient to bf16
once.  An element may therefore miss its exact value by the bf16 rounding of
the exact value plus a few 2^-9-relative terms of the gradient's scale; the test
allows |g - ref| <= |bf16(ref) - ref| + 1e-2 * max|ref| + 1e-6 per tensor (the
1e-6 covers gradients whose exact value vanishes, e.g. dQ of a row with one key,
where D_i from the bf16 O leaves residues near 1e-8), and also requires the
relative 2-norm error ||g - ref|| / ||ref|| <= 1e-2 where ||ref|| > 0.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_06_gb300 import ops
from attention_forward_06_gb300.inputs import WORKLOADS, bf16_bits, draw
from parity_util import round_to_bf16

pytestmark = pytest.mark.gpu


def run(q, k, v, do, causal, scale):
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = ops.attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = ops.attn_bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    st, site = ops.bwd_debug_status()
    assert st == ops.ATTN_OK, f"backward wait ran out at site {site}"
    return dq.cpu(), dk.cpu(), dv.cpu()


def check(name, g, ref):
    g = g.float().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), f"non-finite {name}"
    if not ref.size:
        return
    scale = np.abs(ref).max()
    excess = np.abs(g - ref) - np.abs(round_to_bf16(ref) - ref)
    worst = np.unravel_index(np.argmax(excess), ref.shape)
    assert excess.max() <= 1e-2 * scale + 1e-6, (
        f"{name}: excess {excess.max():.3g} at {worst} (gpu {g[worst]} ref {ref[worst]}, max|ref| {scale:.3g})")
    norm = np.linalg.norm(ref)
    if norm > 0:
        rel = np.linalg.norm(g - ref) / norm
        assert rel <= 1e-2, f"{name}: relative 2-norm error {rel:.3g}"


def full_check(B, Hq, Hkv, Sq, Sk, D, causal, seed, qk_std=1.0):
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, D, seed, qk_std=qk_std)
    do = draw(B, Hq, Hkv, Sq, Sk, D, seed + 1)[0]
    scale = float(np.float32(D ** -0.5))
    dq, dk, dv = run(q, k, v, do, causal, scale)
    rq, rk, rv = oracle.backward(bf16_bits(q), bf16_bits(k), bf16_bits(v), bf16_bits(do), causal, scale)
    check("dq", dq, rq)
    check("dk", dk, rk)
    check("dv", dv, rv)


SHAPES = [
    # B, Hq, Hkv, Sq, Sk, D, causal
    (1, 1, 1, 128, 128, 128, 0),
    (1, 2, 2, 300, 300, 128, 1),      # ragged, causal
    (2, 4, 1, 129, 700, 64, 0),       # G = 4, ragged both ways
    (1, 4, 2, 1000, 129, 128, 1),     # Sq > Sk bottom-right: rows without keys
    (1, 2, 1, 200, 900, 64, 2),       # top-left, Sq < Sk: keys no row sees
    (1, 3, 3, 513, 513, 128, 1),
    (2, 8, 2, 256, 384, 128, 0),
    (1, 2, 1, 1, 1, 128, 0),          # one row, one key
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes_match_oracle(shape):
    full_check(*shape, seed=sum(shape))


def test_sharp_logits():
    full_check(1, 2, 1, 384, 640, 128, 1, seed=41, qk_std=3.0)


def test_train_workload_full_oracle():
    w = WORKLOADS["train"]
    full_check(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.causal, w.seed)


def test_empty_sequences_zero_the_gradients_that_exist():
    q, k, v = [t.cuda() for t in draw(1, 2, 1, 64, 64, 128, seed=43)]
    lse = torch.zeros((1, 2, 0), device="cuda")
    dq, dk, dv = ops.attn_bwd(q[:, :, :0].contiguous(), k, v, q[:, :, :0].contiguous(), lse,
                              q[:, :, :0].contiguous(), causal=0, dk=torch.full_like(k, 7.0),
                              dv=torch.full_like(v, 7.0))
    torch.cuda.synchronize()
    assert torch.all(dk == 0) and torch.all(dv == 0)


def test_deterministic_bitwise():
    q, k, v = [t.cuda() for t in draw(2, 4, 2, 500, 700, 128, seed=45)]
    do = draw(2, 4, 2, 500, 700, 128, seed=46)[0].cuda()
    o, lse = ops.attn_fwd(q, k, v, causal=1)
    a = ops.attn_bwd(q, k, v, o, lse, do, causal=1)
    b = ops.attn_bwd(q, k, v, o, lse, do, causal=1)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_back_to_back_calls_on_two_streams():
    """The three backward kernels overlap one another (programmatic dependent launch):
    many calls in a row, alternating two streams and two shapes, each read right after
    its stream's work, must all reproduce the first result of their shape bit for bit."""
    shapes = [(2, 4, 2, 500, 700, 128, 1), (1, 8, 8, 1024, 1024, 64, 0)]
    data = []
    for (B, Hq, Hkv, Sq, Sk, D, causal) in shapes:
        q, k, v = [t.cuda() for t in draw(B, Hq, Hkv, Sq, Sk, D, seed=Sq + D)]
        do = draw(B, Hq, Hkv, Sq, Sk, D, seed=Sq + D + 1)[0].cuda()
        o, lse = ops.attn_fwd(q, k, v, causal=causal)
        data.append((q, k, v, o, lse, do, causal))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    first = {}
    for i in range(24):
        s = streams[i % 2]
        q, k, v, o, lse, do, causal = data[(i // 2) % 2]
        with torch.cuda.stream(s):
            got = ops.attn_bwd(q, k, v, o, lse, do, causal=causal, stream=s)
            host = [t.cpu() for t in got]  # synchronous copies on the same stream
        st, site = ops.bwd_debug_status(s)
        assert st == ops.ATTN_OK, f"backward wait ran out at site {site}"
        key = (i // 2) % 2
        if key not in first:
            first[key] = host
        else:
            assert all(torch.equal(x, y) for x, y in zip(first[key], host)), i
