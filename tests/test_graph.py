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
