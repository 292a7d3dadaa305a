"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, element by
element on the same seeded inputs: small shapes that span several tiles and
ragged tails, the edge cases (fully masked rows, one row, one key, no keys,
grouped heads), and every benchmark workload at full size: every row of tiny, train, gqa and both
chunked shapes, and 256 seeded rows per head of the long-context one.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_06_gb300 import ops
from attention_forward_06_gb300.inputs import WORKLOADS, bf16_bits, draw, draw_workload, sample_rows
from parity_util import compare

pytestmark = pytest.mark.gpu


def run_gpu(q, k, v, causal, scale):
    o, lse = ops.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    st, site = ops.debug_status()
    assert st == ops.ATTN_OK, f"kernel wait ran out at site {site}"
    return o.cpu(), lse.cpu()


def full_check(B, Hq, Hkv, Sq, Sk, D, causal, seed, qk_std=1.0, label=None):
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, D, seed, qk_std=qk_std)
    scale = float(np.float32(D ** -0.5))
    o, lse = run_gpu(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal, scale)
    return compare(o, lse, o_ref, lse_ref, label=label)


SHAPES = [
    # B, Hq, Hkv, Sq, Sk, D, causal
    (1, 1, 1, 128, 128, 64, 0),       # one tile each
    (1, 2, 2, 300, 300, 128, 1),      # two query blocks, ragged
    (2, 4, 1, 129, 1000, 128, 0),     # ragged both ways, G = 4
    (1, 8, 2, 1000, 129, 64, 1),      # Sq > Sk bottom-right: fully masked rows
    (1, 2, 1, 1, 1, 128, 0),          # one row, one key
    (1, 2, 1, 1, 257, 64, 1),         # one query row against three key tiles
    (1, 1, 1, 257, 1, 128, 1),        # one key
    (1, 4, 4, 127, 127, 64, 2),       # top-left, Sq = Sk
    (1, 2, 1, 200, 700, 128, 2),      # top-left, Sq < Sk
    (1, 2, 1, 700, 200, 64, 2),       # top-left, Sq > Sk
    (1, 3, 3, 513, 513, 128, 1),      # three query blocks
    (2, 8, 8, 256, 384, 64, 0),
    (1, 8, 1, 256, 256, 128, 1),      # G = 8
    (1, 2, 2, 100, 0, 128, 1),        # no keys at all
    (1, 1, 1, 640, 1920, 128, 1),     # bottom-right, many tiles, ragged none
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes_match_oracle(shape):
    B, Hq, Hkv, Sq, Sk, D, causal = shape
    full_check(B, Hq, Hkv, Sq, Sk, D, causal, seed=sum(shape))


def test_tiny_workload_matches_oracle():
    w = WORKLOADS["tiny"]
    stats = full_check(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.causal, w.seed, label="tiny (all rows)")
    assert stats["max_abs_dO"] <= 1e-2


def test_sharp_logits_online_rescale():
    # logits with standard deviation ~9 (Q, K entries N(0, 3^2)): the running max moves a lot
    full_check(1, 4, 1, 512, 1536, 128, 1, seed=77, qk_std=3.0)
    full_check(1, 2, 2, 384, 384, 64, 0, seed=78, qk_std=3.0)


@pytest.mark.parametrize("Sq,Sk,D,causal,boost", [
    (256, 512, 128, 0, 20.0),    # a later key tile ~70 log2 units above the first: P mass beyond 2^64 (row max path)
    (384, 384, 64, 1, 100.0),    # first pass overflows to inf; the boosted tile is the diagonal (masked) one
    (300, 700, 128, 1, 11.0),    # bottom-right, ragged: masses between 2^16 and 2^64 (power-of-two rescale path)
    (256, 512, 64, 0, 16.0),     # rows of one warp on both paths at once
])
def test_lazy_max_second_pass(Sq, Sk, D, causal, boost):
    # The kernel takes a tile's exponentials against a reference value set 8 above
    # the first tile's row max; when a later tile's P mass passes fp16's range it
    # moves the reference up (by a power of two, or to the tile's row max for a mass
    # beyond 2^64) and stores that tile's P again.  Keys 256-383 (the third key tile)
    # are scaled so that this later tile dominates.
    q, k, v = draw(1, 4, 2, Sq, Sk, D, seed=int(boost) + Sq)
    k = k.clone()
    k[:, :, 256:384] = (k[:, :, 256:384].float() * boost).to(torch.bfloat16)
    scale = float(np.float32(D ** -0.5))
    o, lse = run_gpu(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal, scale)
    compare(o, lse, o_ref, lse_ref)


def test_train_workload_full_oracle():
    w = WORKLOADS["train"]
    q, k, v = draw_workload(w)
    o, lse = run_gpu(q, k, v, w.causal, w.scale)
    o_ref, lse_ref = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), w.causal, w.scale)
    compare(o, lse, o_ref, lse_ref, label="train (all rows)")


@pytest.mark.parametrize("name", ["gqa", "chunked128", "chunked64"])
def test_full_size_workloads_every_row(name):
    # the whole workload against the oracle: every row of every head
    w = WORKLOADS[name]
    q, k, v = draw_workload(w)
    o, lse = run_gpu(q, k, v, w.causal, w.scale)
    o_ref, lse_ref = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), w.causal, w.scale)
    compare(o, lse, o_ref, lse_ref, label=f"{name} (all rows)")


def test_long_context_on_256_rows_per_head():
    # 256 seeded rows per head (rows 0 and Sq - 1 always among them), 8192 rows in all
    w = WORKLOADS["long"]
    q, k, v = draw_workload(w)
    o, lse = run_gpu(q, k, v, w.causal, w.scale)
    rows = sample_rows(w.B, w.Hq, w.Sq, 256, seed=w.seed + 1000)
    assert rows.size == w.B * w.Hq * 256
    o_ref, lse_ref = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), w.causal, w.scale, rows=rows)
    o_rows = o.reshape(-1, w.D)[torch.from_numpy(rows)]
    lse_rows = lse.reshape(-1)[torch.from_numpy(rows)]
    compare(o_rows, lse_rows, o_ref, lse_ref, label="long (256 rows per head)")


def test_deterministic_bitwise():
    q, k, v = draw(2, 8, 2, 700, 900, 128, seed=5)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = ops.attn_fwd(qd, kd, vd, causal=1)
    o2, l2 = ops.attn_fwd(qd, kd, vd, causal=1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_gqa_equals_mha_with_repeated_heads():
    q, k, v = draw(1, 8, 2, 384, 512, 128, seed=6)
    G = 4
    o1, l1 = run_gpu(q, k, v, 1, 0.088)
    o2, l2 = run_gpu(q, k.repeat_interleave(G, 1), v.repeat_interleave(G, 1), 1, 0.088)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_chunked_equals_tail_of_full_causal():
    Sq, Sk = 384, 1280
    q, k, v = draw(1, 4, 2, Sk, Sk, 128, seed=8)
    o_full, l_full = run_gpu(q, k, v, 1, 0.088)
    o_c, l_c = run_gpu(q[:, :, Sk - Sq:].contiguous(), k, v, 1, 0.088)
    assert torch.equal(o_c, o_full[:, :, Sk - Sq:]) and torch.equal(l_c, l_full[:, :, Sk - Sq:])


def test_one_hot_rows_return_value_rows():
    # q_i = 32 e0 and k_j* = 32 e0, all other keys 0: O_i = V[j*] exactly representable
    Sq, Sk, D = 256, 640, 128
    q = torch.zeros(1, 1, Sq, D); q[..., 0] = 32
    k = torch.zeros(1, 1, Sk, D); k[0, 0, 333, 0] = 32
    v = draw(1, 1, 1, 1, Sk, D, seed=9)[2]
    o, lse = run_gpu(q.to(torch.bfloat16), k.to(torch.bfloat16), v, 0, float(np.float32(D ** -0.5)))
    assert torch.equal(o[0, 0], v[0, 0, 333].expand(Sq, D))


def test_outputs_written_through_given_buffers_and_stream():
    q, k, v = [t.cuda() for t in draw(1, 2, 1, 200, 300, 64, seed=10)]
    o = torch.full_like(q, float("nan"))
    lse = torch.full((1, 2, 200), float("nan"), device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ops.attn_fwd(q, k, v, causal=0, o=o, lse=lse, stream=s)
    s.synchronize()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def test_wrong_dtype_is_rejected_by_binding():
    q, k, v = [t.cuda() for t in draw(1, 1, 1, 16, 16, 64, seed=11)]
    with pytest.raises(ValueError):
        ops.attn_fwd(q.float(), k, v)


def test_schedule_counters_across_many_launches():
    """Each launch claims work items from one of a set of device counters, and the
    launch's last claim returns its counter to zero.  Many launches in a row, on two
    streams and with item counts below and above the SM count, mixing the plain,
    split-key and block-sparse entry points, must each reproduce the first result
    bit for bit (a counter left non-zero would skip items and leave NaN behind)."""
    dev = torch.device("cuda")
    cases = []
    for (B, Hq, Hkv, Sq, Sk, D, causal) in [(2, 16, 4, 2048, 2048, 128, 1), (1, 4, 4, 1000, 1000, 64, 0),
                                            (1, 2, 1, 300, 4000, 128, 1)]:
        q, k, v = (t.to(dev) for t in draw(B, Hq, Hkv, Sq, Sk, D, seed=Sq + Sk))
        cases.append((q, k, v, causal))
    mask_q, mask_k, mask_v, _ = cases[0]
    gen = torch.Generator().manual_seed(7)
    blocks = (torch.rand(2, 1, 16, 16, generator=gen) < 0.4) | torch.eye(16, dtype=torch.bool)
    mask = ops.pack_block_mask(blocks).to(dev)

    def call(i, stream):
        q, k, v, causal = cases[i % 3]
        kind = (i // 3) % 3
        o = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:3], float("nan"), device=dev)
        if kind == 0:
            ops.attn_fwd(q, k, v, causal=causal, o=o, lse=lse, stream=stream)
        elif kind == 1:
            ops.attn_fwd_splitkv(q, k, v, causal=causal, n_splits=3, o=o, lse=lse, stream=stream)
        else:
            q, k, v, causal = mask_q, mask_k, mask_v, 1
            o = torch.full_like(q, float("nan"))
            lse = torch.full(q.shape[:3], float("nan"), device=dev)
            ops.attn_fwd_blocksparse(q, k, v, mask, causal=causal, o=o, lse=lse, stream=stream)
        return (i % 3, kind), o, lse

    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    first = {}
    results = []
    for i in range(150):
        s = streams[i % 2]
        with torch.cuda.stream(s):
            results.append(call(i, s))
        if i % 10 == 9:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    st, site = ops.debug_status()
    assert st == ops.ATTN_OK, f"kernel wait ran out at site {site}"
    for key, o, lse in results:
        if key not in first:
            first[key] = (o, lse)
            assert not torch.isnan(o.float()).any() and not torch.isnan(lse).any(), key
        else:
            assert torch.equal(o, first[key][0]) and torch.equal(lse, first[key][1]), key


def test_tiny_v_values_round_to_fp16_subnormals_within_tolerance():
    # V is converted to fp16 for the P.V product: magnitudes below 2^-14 fall on fp16's subnormal grid
    # (absolute error below 2^-25), far inside the tolerance; values of every binade down to 2^-30
    q, k, _ = draw(1, 2, 1, 256, 384, 128, seed=21)
    g = torch.Generator().manual_seed(22)
    mag = torch.exp2(-torch.randint(10, 31, (1, 1, 384, 128), generator=g).float())
    sign = torch.where(torch.rand(1, 1, 384, 128, generator=g) < 0.5, -1.0, 1.0)
    v = (sign * mag * (1 + torch.rand(1, 1, 384, 128, generator=g))).to(torch.bfloat16)
    scale = float(np.float32(128 ** -0.5))
    o, lse = run_gpu(q, k, v, 1, scale)
    o_ref, lse_ref = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 1, scale)
    compare(o, lse, o_ref, lse_ref)
    assert float(np.abs(o.float().numpy() - o_ref).max()) < 1e-6


def test_v_beyond_fp16_range_is_clamped_and_leaves_other_rows_exact():
    # The documented limit of the fp16 P.V product: a V entry beyond 65504 is clamped to 65504.  The rows
    # that give its key weight come out wrong but finite; every other row -- including the rows of the same
    # work items for which the key is masked (their P = 0 multiplies it in the same product) -- is exact.
    Sq = Sk = 256
    q, k, v = draw(1, 1, 1, Sq, Sk, 128, seed=23)
    v = v.clone()
    v[0, 0, 200, 5] = 1.0e5  # a bf16 value above fp16's largest finite 65504
    scale = float(np.float32(128 ** -0.5))
    o, lse = run_gpu(q, k, v, 1, scale)  # causal: rows 0..199 never see key 200
    o_ref, lse_ref = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), 1, scale)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    compare(o[:, :, :200], lse[:, :, :200], o_ref[:, :, :200], lse_ref[:, :, :200])
    # the other columns of the rows that see the key are unaffected as well
    keep = [c for c in range(128) if c != 5]
    compare(o[:, :, 200:, keep].contiguous(), lse[:, :, 200:], o_ref[:, :, 200:, keep], lse_ref[:, :, 200:])


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal", [
    (2, 8, 2, 512, 3000, 128, 1),   # chunked-prefill shape: 8 items per kv head
    (1, 4, 4, 700, 700, 64, 2),     # ragged, no grouping of heads (G = 1)
    (3, 6, 2, 300, 1000, 128, 0),   # non-causal, G = 3
])
def test_item_orders_give_identical_results(B, Hq, Hkv, Sq, Sk, D, causal, monkeypatch):
    """The grouped item order (a kv head's items handed out together) computes every output element exactly as
    the heads-fastest order does; both match the oracle."""
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, D, seed=Sq + Sk)
    scale = float(np.float32(D ** -0.5))
    outs = {}
    for order in ("heads", "grouped"):
        monkeypatch.setenv("ATTN_FWD_ITEM_ORDER", order)
        outs[order] = run_gpu(q, k, v, causal, scale)
    assert torch.equal(outs["heads"][0], outs["grouped"][0]) and torch.equal(outs["heads"][1], outs["grouped"][1])
    o_ref, lse_ref = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal, scale)
    compare(*outs["grouped"], o_ref, lse_ref, label=f"order {B}x{Hq}x{Hkv}x{Sq}x{Sk}x{D}x{causal}")
    # the block-sparse and ordered forwards have the grouped order too
    rng = np.random.default_rng(Sq + Sk)
    blocks = torch.from_numpy(rng.random((B, Hq, -(-Sq // 128), -(-Sk // 128))) < 0.5)
    words = ops.pack_block_mask(blocks).cuda()
    tile_order = torch.from_numpy(np.stack([rng.permutation(-(-Sk // 128)) for _ in range(B * -(-Sq // 256))])
                                  .reshape(B, 1, -(-Sq // 256), -(-Sk // 128)).astype(np.int32)).cuda()
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    for call in (lambda: ops.attn_fwd_blocksparse(qd, kd, vd, words, causal=causal, scale=scale),
                 lambda: ops.attn_fwd_ordered(qd, kd, vd, tile_order, causal=causal, scale=scale)):
        res = {}
        for order in ("heads", "grouped"):
            monkeypatch.setenv("ATTN_FWD_ITEM_ORDER", order)
            res[order] = call()
        torch.cuda.synchronize()
        assert torch.equal(res["heads"][0], res["grouped"][0]) and torch.equal(res["heads"][1], res["grouped"][1])
