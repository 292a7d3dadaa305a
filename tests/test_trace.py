"""The forward kernel's timeline build (-DATTN_TRACE, include/attn_fwd_trace.h):
the traced library computes the same results as the default one bit for bit,
and its events are consistent -- per role in time order, and as many of each
kind as the work requires (items published, K and V loads, P.V products, S
tiles read by each softmax warpgroup)."""
import ctypes

import numpy as np
import pytest
import torch

from attention_forward_06_gb300 import _lib, build, trace
from attention_forward_06_gb300.inputs import draw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    build.build()
    return _lib.load("attn_fwd"), _lib.load("attn_fwd_trace")


def key_tiles(B, Hq, Sq, Sk, causal):
    """Key tiles each 256-row work item visits (causal 1: bottom-right aligned)."""
    total, items = 0, 0
    for q0 in range(0, Sq, 256):
        last = min(q0 + 256, Sq) - 1
        end = min(Sk, last + (Sk - Sq) + 1) if causal else Sk
        total += max(0, -(-end // 128)) * B * Hq
        items += B * Hq
    return total, items


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal", [
    (2, 16, 4, 2304, 2304, 128, 1),   # 288 items on at most 152 CTAs: several items per CTA
    (1, 8, 2, 700, 1500, 64, 1),      # bottom-right, ragged, D = 64
])
def test_traced_build_matches_and_its_events_are_consistent(libs, B, Hq, Hkv, Sq, Sk, D, causal):
    plain, traced = libs
    q, k, v = [t.cuda() for t in draw(B, Hq, Hkv, Sq, Sk, D, seed=Sq + D)]
    scale = float(np.float32(D ** -0.5))
    stream = torch.cuda.current_stream().cuda_stream
    outs = []
    trace.read(traced)  # start from empty counts
    for lib in (plain, traced):
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, Sq), device="cuda")
        assert lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Sq, Sk,
                            D, causal, ctypes.c_float(scale), stream) == 0
        outs.append((o, lse))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    site = ctypes.c_int(0)
    assert traced.attn_fwd_debug_status(stream, ctypes.byref(site)) == 0, site.value

    counts, recs = trace.read(traced)
    assert counts.max() <= recs.shape[2], "a role overflowed its event buffer"
    ctas = [c for c in range(counts.shape[0]) if counts[c, trace.PRODUCER] > 0]
    tiles, n_items = key_tiles(B, Hq, Sq, Sk, causal)
    assert len(ctas) == min(152, n_items) or len(ctas) <= n_items
    published = k_loads = v_loads = pv = 0
    for c in ctas:
        for role in range(counts.shape[1]):
            t = trace.events(counts, recs, c, role)["t"].astype(np.int64)
            assert np.all(np.diff(t) >= 0), f"CTA {c} role {role}: events out of time order"
        prod = trace.events(counts, recs, c, trace.PRODUCER)
        published += int(((prod["code"] == 1) & (prod["arg"] != 0xFFFFFFFF)).sum())
        k_loads += int((prod["code"] == 2).sum())
        v_loads += int((prod["code"] == 3).sum())
        iss = trace.events(counts, recs, c, trace.ISSUER)
        pv_c = int((iss["code"] == 11).sum())
        pv += pv_c
        assert (iss["code"] == 13).sum() == 1
        for role in (trace.SOFTMAX0, trace.SOFTMAX1):  # one S read and one hand-off per key tile
            sm = trace.events(counts, recs, c, role)
            assert (sm["code"] == 20).sum() == pv_c // 2 == (sm["code"] == 21).sum()
    assert published == n_items
    assert k_loads == v_loads == tiles
    assert pv == 2 * tiles
    s = trace.summarize(counts, recs)
    assert s["span_us"] > 0 and s["step_us"] > 0 and s["softmax_us"] > 0


# ---------------------------------------------------------------------------- backward
from attention_forward_06_gb300 import ops, trace_bwd  # noqa: E402


@pytest.fixture(scope="module")
def bwd_libs():
    build.build()
    return _lib.load("attn_bwd"), _lib.load("attn_bwd_trace")


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal", [
    (2, 8, 8, 1536, 1536, 128, 1),   # G = 1, more dQ and dK/dV items than CTAs
    (1, 8, 2, 700, 1300, 64, 1),     # G = 4, bottom-right, ragged, D = 64
])
def test_traced_backward_matches_and_its_events_are_consistent(bwd_libs, B, Hq, Hkv, Sq, Sk, D, causal):
    plain, traced = bwd_libs
    q, k, v = [t.cuda() for t in draw(B, Hq, Hkv, Sq, Sk, D, seed=Sk + D)]
    scale = float(np.float32(D ** -0.5))
    o, lse = ops.attn_fwd(q, k, v, causal=causal, scale=scale)
    dout = torch.randn(q.shape, generator=torch.Generator().manual_seed(Sq)).to(torch.bfloat16).cuda()
    ws = torch.empty(ops.bwd_workspace_size(B, Hq, Sq), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    trace_bwd.read(traced)  # start from empty counts
    grads = []
    for lib in (plain, traced):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        assert lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, Sq, Sk, D, causal,
                            ctypes.c_float(scale), ws.data_ptr(), ws.numel(), stream) == 0
        grads.append((dq, dk, dv))
    torch.cuda.synchronize()
    for a, b in zip(*grads):
        assert torch.equal(a, b)
    site = ctypes.c_int(0)
    assert traced.attn_bwd_debug_status(stream, ctypes.byref(site)) == 0, site.value

    counts, recs = trace_bwd.read(traced)
    assert counts.max() <= recs.shape[3], "a role overflowed its event buffer"
    diag = Sk - Sq
    n_qt, n_kt, G = -(-Sq // 128), -(-Sk // 128), Hq // Hkv
    # dK/dV: one item per (batch, kv head, key tile) with query tiles; a step per (query head, query tile)
    first_qt = [max(0, (j * 128 - diag) // 128) for j in range(n_kt)]
    dkdv_items = B * Hkv * sum(1 for j in range(n_kt) if n_qt - first_qt[j] > 0)
    dkdv_steps = B * Hkv * G * sum(max(0, n_qt - first_qt[j]) for j in range(n_kt))
    # dQ: one item per (batch, query head, query tile) with keys; a step per key tile
    kt = [max(0, -(-min(Sk, min(i * 128 + 128, Sq) - 1 + diag + 1) // 128)) for i in range(n_qt)]
    dq_items = B * Hq * sum(1 for n in kt if n > 0)
    dq_steps = B * Hq * sum(kt)
    for kernel, n_items, n_steps in ((trace_bwd.DKDV, dkdv_items, dkdv_steps), (trace_bwd.DQ, dq_items, dq_steps)):
        ctas = [c for c in range(counts.shape[1]) if counts[kernel, c, trace_bwd.PRODUCER] > 0]
        assert ctas
        heads = accs = 0
        for c in ctas:
            for role in range(counts.shape[2]):
                t = trace_bwd.events(counts, recs, kernel, c, role)["t"].astype(np.int64)
                assert np.all(np.diff(t) >= 0), f"kernel {kernel} CTA {c} role {role}: events out of time order"
            iss = trace_bwd.events(counts, recs, kernel, c, trace_bwd.ISSUER)
            heads += int((iss["code"] == 10).sum())
            accs += int((iss["code"] == 11).sum())
            assert (iss["code"] == 13).sum() == 1
            for role in (trace_bwd.COMPUTE0, trace_bwd.COMPUTE1):  # one S read and one hand-off per step
                ev = trace_bwd.events(counts, recs, kernel, c, role)
                assert (ev["code"] == 20).sum() == (ev["code"] == 21).sum() == (iss["code"] == 11).sum()
                assert (ev["code"] == 23).sum() == (ev["code"] == 24).sum() == (iss["code"] == 10).sum()
        assert heads == n_items
        assert accs == n_steps
        s = trace_bwd.summarize(counts, recs, kernel)
        assert s["span_us"] > 0 and s["step_us"] > 0 and s["epilogue_us"] > 0 and 0 <= s["item_share"] < 1
