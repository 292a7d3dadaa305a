"""Failure handling on the GPU without a fault: every wait in the kernels is
bounded, and a wait that runs out (or sees the abort flag another role raised)
is reported as a status the host reads, leaving the CUDA context usable.  The
wait is made to run out on a barrier that nothing arrives on; no trap, no
assert, no bad address, no endless loop.
"""
import numpy as np
import pytest
import torch

from attention_forward_06_gb300 import _lib, ops
from attention_forward_06_gb300.inputs import draw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def probe():
    from attention_forward_06_gb300 import build
    build.build()
    return _lib.load("attn_probe")


def run_wait(probe, timeout_ns, abort_after_ns):
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    rc = probe.attn_probe_wait_timeout(timeout_ns, abort_after_ns, status.data_ptr(), waited.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    return status.item(), waited.item()


def test_bounded_wait_times_out_and_reports(probe):
    st, waited = run_wait(probe, 50_000_000, 0)  # 50 ms on a barrier nobody arrives on
    assert st == 1
    assert 50_000_000 <= waited < 2_000_000_000


def test_bounded_wait_sees_abort_flag(probe):
    st, waited = run_wait(probe, 1_000_000_000, 20_000_000)  # another warp aborts after 20 ms
    assert st == 2
    assert 20_000_000 <= waited < 1_000_000_000


def test_context_usable_after_timeouts(probe):
    run_wait(probe, 10_000_000, 0)
    q, k, v = [t.cuda() for t in draw(1, 2, 1, 300, 300, 128, seed=3)]
    o, lse = ops.attn_fwd(q, k, v, causal=1)
    st, site = ops.debug_status()
    assert st == ops.ATTN_OK and site == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_invalid_probe_arguments_are_rejected(probe):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    assert probe.attn_probe_wait_timeout(0, 0, status.data_ptr(), waited.data_ptr(), None) == 1
    assert probe.attn_probe_wait_timeout(3_000_000_000, 0, status.data_ptr(), waited.data_ptr(), None) == 1
    assert probe.attn_probe_wait_timeout(1000, 0, None, waited.data_ptr(), None) == 2
