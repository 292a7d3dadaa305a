"""The entry points inside a captured CUDA graph.

Every call is asynchronous on its stream, allocates nothing and bakes its
arguments (pointers, sizes, tensor maps) into the launch, so a sequence of calls
can be captured once and replayed on new data copied into the same buffers.
The first call of each entry point on a device does its one-time set-up (device
query, kernel attributes); it is made before the capture, as with any library.
The test captures the forward, the split-key forward (two kernels) and the
backward (three kernels, chained by programmatic dependent launch) in one graph,
replays it on two input sets in turn, and requires every output to equal, bit for
bit, the same calls made eagerly on the same inputs.
"""
import numpy as np
import pytest
import torch

from attention_forward_06_gb300 import ops
from attention_forward_06_gb300.inputs import draw

pytestmark = pytest.mark.gpu

B, HQ, HKV, SQ, SK, D, CAUSAL = 2, 8, 2, 700, 900, 128, 1
SCALE = float(np.float32(D ** -0.5))


def inputs(seed):
    q, k, v = draw(B, HQ, HKV, SQ, SK, D, seed)
    do = draw(B, HQ, HKV, SQ, SK, D, seed + 1)[0]
    return [t.cuda() for t in (q, k, v, do)]


def calls(q, k, v, do):
    o, lse = ops.attn_fwd(q, k, v, causal=CAUSAL, scale=SCALE)
    o2, lse2 = ops.attn_fwd_splitkv(q, k, v, causal=CAUSAL, scale=SCALE, n_splits=3)
    dq, dk, dv = ops.attn_bwd(q, k, v, o, lse, do, causal=CAUSAL, scale=SCALE)
    return o, lse, o2, lse2, dq, dk, dv


def test_forward_splitkv_and_backward_replay_in_a_cuda_graph():
    a, b = inputs(41), inputs(43)
    ref = {"a": [t.clone() for t in calls(*a)], "b": [t.clone() for t in calls(*b)]}
    torch.cuda.synchronize()
    static = [t.clone() for t in a]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out = calls(*static)
    for name, src in (("b", b), ("a", a), ("b", b)):
        for dst, s in zip(static, src):
            dst.copy_(s)
        graph.replay()
        torch.cuda.synchronize()
        st, site = ops.debug_status()
        assert st == ops.ATTN_OK, f"forward wait ran out at site {site}"
        st, site = ops.bwd_debug_status()
        assert st == ops.ATTN_OK, f"backward wait ran out at site {site}"
        for i, (got, want) in enumerate(zip(out, ref[name])):
            assert torch.equal(got, want), f"output {i} of the replay on input set {name} differs from the eager call"


def test_graph_replays_next_to_direct_launches_on_another_stream():
    """A recorded launch keeps the schedule counter it was given at capture; direct
    launches draw from a separate set, so a replay running next to many direct
    launches on another stream (every direct counter taken in turn) shares none."""
    a = inputs(51)
    q, k, v = a[:3]
    o_ref, lse_ref = ops.attn_fwd(q, k, v, causal=CAUSAL, scale=SCALE)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    o_g = torch.full_like(q, float("nan"))
    lse_g = torch.full(q.shape[:3], float("nan"), device=q.device)
    with torch.cuda.graph(graph):
        ops.attn_fwd(q, k, v, causal=CAUSAL, scale=SCALE, o=o_g, lse=lse_g)
    other = torch.cuda.Stream()
    direct = []
    for rep in range(3):
        o_g.fill_(float("nan"))
        lse_g.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()  # on the current stream
        with torch.cuda.stream(other):
            for _ in range(70):  # more than the 64 direct counters
                o = torch.full_like(q, float("nan"))
                lse = torch.full(q.shape[:3], float("nan"), device=q.device)
                ops.attn_fwd(q, k, v, causal=CAUSAL, scale=SCALE, o=o, lse=lse, stream=other)
                direct.append((o, lse))
        torch.cuda.synchronize()
        st, site = ops.debug_status()
        assert st == ops.ATTN_OK, f"forward wait ran out at site {site}"
        assert torch.equal(o_g, o_ref) and torch.equal(lse_g, lse_ref), f"replay {rep}"
    for o, lse in direct:
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
