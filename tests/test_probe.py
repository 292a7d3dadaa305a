"""Primitive checks of the attention kernel's building blocks on the GPU:
TMA swizzled tile loads, the SS-form QK^T MMA with its descriptors, and the
TS-form P.V MMA with P in tensor memory and V as an MN-major operand.  Each is
compared with a CPU matmul of the same bf16 values.
"""
import numpy as np
import pytest
import torch

from attention_forward_06_gb300 import _lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def probe():
    from attention_forward_06_gb300 import build
    build.build()
    return _lib.load("attn_probe")


def swizzled_offset(r, c, rows):
    """Byte offset of element (r, c) of a [rows][D] bf16 tile loaded as 64-column boxes with
    the 128-byte swizzle: box cb = c // 64 holds rows at a 128-byte pitch, and the 16-byte
    chunk index inside a row is XORed with (row mod 8)."""
    cb, cc = divmod(c, 64)
    chunk, within = divmod(cc, 8)
    return cb * rows * 128 + r * 128 + ((chunk ^ (r % 8)) * 16) + within * 2


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("q_rows,k_rows", [(128, 128), (100, 77), (1, 128)])
def test_ss_mma_and_tma_swizzle(probe, D, q_rows, k_rows):
    g = torch.Generator().manual_seed(D + q_rows)
    q = torch.randn(q_rows, D, generator=g).to(torch.bfloat16)
    k = torch.randn(k_rows, D, generator=g).to(torch.bfloat16)
    qd, kd = q.cuda(), k.cuda()
    s = torch.full((128, 128), float("nan"), device="cuda")
    dump = torch.zeros(128 * D, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.attn_probe_mma_ss(qd.data_ptr(), q_rows, kd.data_ptr(), k_rows, D, s.data_ptr(), dump.data_ptr(),
                                 status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert status.item() == 0
    # TMA: shared-memory image is the 128-byte swizzle of Q, zero past the last row
    qpad = torch.zeros(128, D, dtype=torch.bfloat16)
    qpad[:q_rows] = q
    img = dump.cpu().numpy().view(np.uint16)
    qbits = qpad.view(torch.int16).numpy().view(np.uint16)
    expect = np.zeros(128 * D, np.uint16)
    r, c = np.meshgrid(np.arange(128), np.arange(D), indexing="ij")
    expect[swizzled_offset(r, c, 128) // 2] = qbits[r, c]
    np.testing.assert_array_equal(img, expect)
    # MMA: S = Q K^T in fp32
    kpad = torch.zeros(128, D, dtype=torch.bfloat16)
    kpad[:k_rows] = k
    ref = qpad.float() @ kpad.float().T
    torch.testing.assert_close(s.cpu(), ref, rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("D", [64, 128])
def test_ts_mma_p_from_tensor_memory(probe, D):
    g = torch.Generator().manual_seed(7 + D)
    p = torch.rand(128, 128, generator=g).to(torch.bfloat16)  # asymmetric, so a swapped pair shows
    v = torch.randn(128, D, generator=g).to(torch.bfloat16)
    ref = p.float() @ v.float()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pd, vd = p.cuda(), v.cuda()

    def run(lbo, sbo):
        o = torch.full((128, D), float("nan"), device="cuda")
        status.zero_()
        rc = probe.attn_probe_mma_ts(pd.data_ptr(), vd.data_ptr(), D, lbo, sbo, o.data_ptr(), status.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
        assert rc == 0
        torch.cuda.synchronize()
        assert status.item() == 0
        return o.cpu()

    # MN-major V: leading offset = stride between 64-column chunks (128 rows x 128 B),
    # stride offset = stride between 8-row groups (1024 B)
    o = run(128 * 128, 1024)
    err = (o - ref).abs().max().item()
    if not err < 1e-3:
        alt = (run(1024, 128 * 128) - ref).abs().max().item()
        pytest.fail(f"P.V mismatch: max err {err} (with leading/stride offsets swapped: {alt})")


def test_bf16_mma_rate_per_sm(probe):
    """The dense bf16 tensor-core rate of one SM, measured with back-to-back 128 x N x 16 MMAs on every SM: the
    per-SM figure behind the benchmark's hardware-derived peak (8192 FLOP per clock)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rates = {}
    for N in (128, 256):
        cycles = torch.zeros(sms, dtype=torch.int64, device="cuda")
        nanos = torch.zeros(sms, dtype=torch.int64, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        n_mma = 4096
        assert probe.attn_probe_mma_rate(n_mma, N, sms, cycles.data_ptr(), nanos.data_ptr(), status.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream) == 0
        torch.cuda.synchronize()
        assert status.item() == 0
        c = cycles.cpu().double().numpy()
        rates[N] = float(np.median(2 * 128 * N * 16 * n_mma / c))
        ghz = float(np.median(c / nanos.cpu().double().numpy()))
        print(f"N={N}: {rates[N]:.0f} bf16 FLOP per clock per SM at {ghz:.2f} GHz "
              f"({rates[N] * sms * ghz * 1e9 / 1e12:.0f} TFLOP/s over {sms} SMs)")
    assert 0.9 * 8192 <= rates[256] <= 1.05 * 8192
    assert rates[128] <= 1.05 * 8192


def test_ex2_rate_per_sm(probe):
    """ex2.approx results per clock of one SM (the softmax's exponent unit), every SM busy."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cycles = torch.zeros(sms, dtype=torch.int64, device="cuda")
    sink = torch.zeros(sms * 512, dtype=torch.float32, device="cuda")
    iters = 4096
    assert probe.attn_probe_ex2_rate(iters, sms, cycles.data_ptr(), sink.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    rate = float(np.median(512 * 8 * iters / cycles.cpu().double().numpy()))
    print(f"{rate:.1f} ex2.approx per clock per SM")
    assert torch.isfinite(sink).all()
    assert 8 <= rate <= 128
