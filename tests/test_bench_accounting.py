"""The benchmark's work accounting, which sets the headline metric, against brute
force on small shapes (CPU only).

bench.py counts the algorithmic work as 4*D FLOP per unmasked (query row, key)
pair, summed over every (batch, head); the conventional count is 4*B*Hq*Sq*Sk*D,
halved under a causal mask; the minimal HBM traffic is Q, K, V, O (bf16) and LSE
(fp32) once.  Each helper is checked here against an explicit element mask or
the tensors' byte sizes, and the documented relations between the two FLOP
conventions are checked on the benchmark workloads themselves.
"""
import numpy as np
import pytest

import bench
from attention_forward_06_gb300.inputs import WORKLOADS, Workload


def element_mask(Sq, Sk, causal):
    """bool [Sq, Sk]: key j visible to row i (0 none, 1 bottom-right j <= i + Sk - Sq, 2 top-left j <= i)."""
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    if causal == 0:
        return np.ones((Sq, Sk), bool)
    return j <= (i + (Sk - Sq) if causal == 1 else i)


SHAPES = [(1, 1, 1, 5, 5, 64, 0), (2, 4, 2, 7, 13, 64, 1), (1, 2, 1, 13, 7, 128, 1), (1, 3, 3, 9, 4, 64, 2),
          (2, 2, 1, 4, 9, 128, 2), (1, 1, 1, 300, 300, 64, 1), (1, 2, 2, 0, 5, 64, 1), (1, 1, 1, 6, 0, 64, 1)]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal", SHAPES)
def test_pair_and_flop_counts_match_brute_force(B, Hq, Hkv, Sq, Sk, D, causal):
    w = Workload("t", B, Hq, Hkv, Sq, Sk, D, causal, seed=0)
    pairs = int(element_mask(Sq, Sk, causal).sum())
    assert bench.allowed_pairs(w) == pairs
    assert bench.alg_flops(w) == 4.0 * D * B * Hq * pairs
    assert bench.conv_flops(w) == 4.0 * B * Hq * Sq * Sk * D * (0.5 if causal else 1.0)
    q_bytes = B * Hq * Sq * D * 2
    kv_bytes = B * Hkv * Sk * D * 2
    assert bench.min_hbm_bytes(w) == q_bytes * 2 + kv_bytes * 2 + B * Hq * Sq * 4  # Q, O, K, V, LSE


@pytest.mark.parametrize("Sq,Sk,causal", [(300, 300, 1), (130, 700, 1), (700, 130, 1), (256, 512, 0), (200, 390, 2)])
def test_row_flops_match_brute_force(Sq, Sk, causal):
    w = Workload("t", 2, 3, 1, Sq, Sk, 64, causal, seed=0)
    visible = element_mask(Sq, Sk, causal).sum(axis=1)
    rows = np.random.default_rng(7).integers(0, w.B * w.Hq * Sq, 40)
    assert bench.row_flops(w, rows) == 4.0 * w.D * float(visible[rows % Sq].sum())
    every = np.arange(w.B * w.Hq * Sq)
    assert bench.row_flops(w, every) == bench.alg_flops(w)


@pytest.mark.parametrize("Sq,Sk,causal,Hm", [(300, 300, 1, 1), (256, 640, 1, 3), (640, 256, 1, 1), (384, 384, 0, 3),
                                             (200, 450, 2, 1)])
def test_blocksparse_pairs_match_brute_force(Sq, Sk, causal, Hm):
    B, Hq, blk = 2, 3, 128
    w = Workload("t", B, Hq, 1, Sq, Sk, 64, causal, seed=0)
    QB, KB = -(-Sq // blk), -(-Sk // blk)
    blocks = np.random.default_rng(Sq + Sk).random((B, Hm, QB, KB)) < 0.4
    base = element_mask(Sq, Sk, causal)
    total = 0
    for b in range(B):
        for h in range(Hq):
            marked = blocks[b, 0 if Hm == 1 else h]
            elem = np.repeat(np.repeat(marked, blk, axis=0), blk, axis=1)[:Sq, :Sk]
            total += int((base & elem).sum())
    assert bench.blocksparse_pairs(w, blocks) == total


def test_flop_conventions_on_the_benchmark_workloads():
    # square causal shapes: the two conventions agree to 0.05 %
    for name in ("train", "gqa", "long"):
        w = WORKLOADS[name]
        assert abs(bench.alg_flops(w) / bench.conv_flops(w) - 1.0) < 5e-4
    # bottom-right chunks over a long context see almost every key: per head the pairs are
    # Sq (Sk - Sq) + Sq (Sq + 1) / 2 against the conventional Sq Sk / 2, a ratio of 1.969 here
    for name in ("chunked128", "chunked64"):
        w = WORKLOADS[name]
        ratio = 2.0 * (w.Sk - w.Sq) / w.Sk + (w.Sq + 1) / w.Sk
        assert bench.alg_flops(w) / bench.conv_flops(w) == pytest.approx(ratio, rel=1e-12)
        assert ratio == pytest.approx(1.9688, abs=1e-4)
    # the minimal bytes of every workload, as the scope table lists them (MB)
    for name, mb in (("tiny", 0.07), ("train", 134.7), ("gqa", 337.6), ("chunked128", 604.5), ("chunked64", 302.5),
                     ("long", 1350.6)):
        assert bench.min_hbm_bytes(WORKLOADS[name]) / 1e6 == pytest.approx(mb, abs=0.05)
    assert bench.alg_flops(WORKLOADS["tiny"]) == bench.conv_flops(WORKLOADS["tiny"])


def test_traffic_record_key_ignores_comments_and_tracks_code(tmp_path):
    """The DRAM traffic record is keyed to the kernel's code: editing a comment keeps the key, editing code
    changes it."""
    src = tmp_path / "k.cu"
    src.write_text("// a comment\nint f(int x) {\n  return x + 1;  // trailing\n}\n/* block\n comment */\n")
    base = bench.kernel_code_sha256([str(src)])
    src.write_text("// another comment\n\nint f(int x) {\n  return x + 1;  // changed\n}\n")
    assert bench.kernel_code_sha256([str(src)]) == base
    src.write_text("int f(int x) {\n  return x + 2;\n}\n")
    assert bench.kernel_code_sha256([str(src)]) != base


def test_committed_traffic_record_is_for_the_current_kernel():
    """Every performance workload has a DRAM traffic record taken on the kernel code as it stands, so the
    benchmark line carries measured traffic (a kernel change without a new capture fails here)."""
    for name in bench.PERF_WORKLOADS:
        assert bench.traffic_for(name), f"no current traffic record for {name}"
