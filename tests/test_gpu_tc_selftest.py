"""tcgen05 descriptor self-test: one MMA chain through the C ABI against a float64
matmul of the same bf16 operands (K-major and MN-major B operands)."""
import pytest
import torch

from sparse_attention_diffusion_gb300 import mcs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    return torch.device("cuda")


def _operands(seed, dev):
    g = torch.Generator().manual_seed(seed)
    a = torch.randn(128, 64, generator=g).to(torch.bfloat16)
    b = torch.randn(128, 64, generator=g).to(torch.bfloat16)
    return a, b


def test_kmajor_b(dev):
    a, b = _operands(0, dev)
    d = torch.zeros(128, 128, dtype=torch.float32, device=dev)
    mcs.mcs_selftest_tc_mma(a.to(dev), b.to(dev), d, 0)
    mcs.mcs_check_status()
    ref = a.double() @ b.double().T
    assert torch.allclose(d.cpu().double(), ref, atol=1e-3, rtol=1e-4)


def test_mnmajor_b(dev):
    a, b = _operands(1, dev)
    bt = b.T.contiguous()                   # [64 (K) x 128 (N)], N contiguous
    d = torch.zeros(128, 128, dtype=torch.float32, device=dev)
    mcs.mcs_selftest_tc_mma(a.to(dev), bt.to(dev), d, 1, 16384, 1024)
    mcs.mcs_check_status()
    ref = a.double() @ bt.double()
    assert torch.allclose(d.cpu().double(), ref, atol=1e-3, rtol=1e-4)


def test_a_operand_from_tensor_memory(dev):
    a, b = _operands(2, dev)
    d = torch.zeros(128, 128, dtype=torch.float32, device=dev)
    mcs.mcs_selftest_tc_mma(a.to(dev), b.to(dev), d, 2)
    mcs.mcs_check_status()
    ref = a.double() @ b.double().T
    assert torch.allclose(d.cpu().double(), ref, atol=1e-3, rtol=1e-4)


def test_tma_gather4_rows(dev):
    g = torch.Generator().manual_seed(3)
    src = torch.randn(1000, 128, generator=g).to(torch.bfloat16)
    rows = torch.randint(0, 1000, (128,), generator=g, dtype=torch.int32)
    rows[5] = 1000          # out of range -> zeros
    rows[77] = 5000
    out = torch.empty(128, 128, dtype=torch.bfloat16, device=dev)
    mcs.mcs_selftest_tma_gather(src.to(dev), rows.to(dev), out)
    mcs.mcs_check_status()
    want = torch.zeros(128, 128, dtype=torch.bfloat16)
    ok = rows < 1000
    want[ok] = src[rows[ok].long()]
    assert torch.equal(out.cpu(), want)


def test_ex2_rate(dev):
    """The exponential-rate diagnostic: one CTA per SM, each reporting its SM
    clock cycles and exponential count; the rate is positive, finite and of the
    order an SM's special-function units allow (a few to a few tens per clock)."""
    n = torch.cuda.get_device_properties(dev).multi_processor_count
    out = torch.zeros((n, 2), dtype=torch.int64, device=dev)
    mcs.mcs_selftest_ex2_rate(1 << 12, out)
    mcs.mcs_check_status()
    cyc, cnt = out[:, 0].cpu(), out[:, 1].cpu()
    assert bool((cyc > 0).all()) and bool((cnt == 1024 * 8 * (1 << 12)).all())
    rate = mcs.ex2_per_clock_per_sm(1 << 12)
    print(f"ex2.approx.ftz.f32 per SM clock: {rate:.2f}")
    assert 2.0 < rate < 256.0
