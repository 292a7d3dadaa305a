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
