"""Unit self-tests of the tcgen05 building blocks of the prefill kernel."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from attention_forward_blackwell_gb300 import build
    build.build()


def test_tmem_noop_roundtrip_is_bit_exact():
    from attention_forward_blackwell_gb300 import binding
    g = torch.Generator(device="cuda").manual_seed(5)
    x = torch.randn(128, 64, device="cuda", generator=g) * 1e3
    x[0, :4] = torch.tensor([float("inf"), -float("inf"), 1e-40, -0.0])
    y = binding.selftest_tmem_roundtrip(x)
    torch.cuda.synchronize()
    assert torch.equal(x.view(torch.int32), y.view(torch.int32))


@pytest.mark.parametrize("kdim", [64, 128, 256])
def test_score_mma_tile(kdim):
    from attention_forward_blackwell_gb300 import binding
    g = torch.Generator(device="cuda").manual_seed(kdim)
    a = torch.randn(128, kdim, device="cuda", generator=g).bfloat16()
    b = torch.randn(128, kdim, device="cuda", generator=g).bfloat16()
    d = binding.selftest_mma_tile(a, b, 0)
    ref = a.double() @ b.double().T
    torch.cuda.synchronize()
    err = (d.double() - ref).abs().max().item()
    print("score tile kdim", kdim, "max err", err)
    assert err < 1e-3 * kdim ** 0.5


def test_value_mma_tile():
    from attention_forward_blackwell_gb300 import binding
    g = torch.Generator(device="cuda").manual_seed(9)
    p = torch.rand(128, 128, device="cuda", generator=g).bfloat16()
    v = torch.randn(128, 128, device="cuda", generator=g).bfloat16()
    d = binding.selftest_mma_tile(p, v, 1)
    ref = p.double() @ v.double()
    torch.cuda.synchronize()
    err = (d.double() - ref).abs().max().item()
    print("value tile max err", err)
    assert err < 1e-2


def test_polynomial_exp2_against_exact():
    """The FMA-pipe exp2 used for part of the softmax: relative error below
    1e-4 against the exact 2^x wherever the result is a normal float
    (x in [-125, 126]), and tiny positive normal values further down (inputs
    are clamped at -125)."""
    import numpy as np
    from attention_forward_blackwell_gb300 import binding
    xs = np.concatenate([np.linspace(-125, 126, 400001), np.arange(-125, 127, 1.0),
                         np.arange(-125, 126, 1.0) + 0.5]).astype(np.float32)
    y = binding.selftest_exp2_poly(torch.from_numpy(xs).cuda()).cpu().numpy().astype(np.float64)
    rel = np.abs(y / np.exp2(xs.astype(np.float64)) - 1)
    print("poly exp2 max rel err", rel.max())
    assert rel.max() < 1e-4
    low = binding.selftest_exp2_poly(torch.tensor([-126.0, -127.0, -500.0, -float("inf")],
                                                  device="cuda")).cpu().numpy()
    assert np.all(low > 0) and np.all(low < 2.0 ** -124)
