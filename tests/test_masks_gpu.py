"""Sliding-window mask and attention sinks ("2026-05-28_STATUS.md" items D3,
D4, D5c) on the GPU against the fp64 oracle (same readings: oracle.c)."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_parity import THREADS, check_device_error, compare, free_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from attention_forward_blackwell_gb300 import build
    build.build()
    yield
    free_cuda()


def _oracle(x, scale, causal, window, sinks, rows=None):
    from attention_forward_blackwell_gb300 import inputs
    lens = None if x.seqlens_k is None else x.seqlens_k.cpu().tolist()
    sk = None if sinks is None else sinks.cpu().double().numpy()
    return oracle.attention_fwd(inputs.bf16_bits(x.q), inputs.bf16_bits(x.k),
                                inputs.bf16_bits(x.v), scale=scale, causal=causal,
                                seqlens_k=lens, rows=rows, threads=THREADS,
                                window=window, sinks=sk)


def _sinks(hq, seed, on):
    if not on:
        return None
    g = torch.Generator().manual_seed(seed)
    return (2.0 * torch.randn(hq, generator=g)).float().cuda()


PREFILL = [
    # B, Hq, Hkv, Sq, Sk, d, causal, window, sinks, lengths
    (1, 2, 1, 300, 300, 64, True, 1, False, None),
    (1, 2, 1, 300, 300, 64, True, 100, True, None),
    (1, 2, 2, 600, 600, 128, True, 128, False, None),
    (1, 2, 2, 600, 600, 128, True, 257, True, None),
    (1, 2, 2, 600, 600, 128, False, 300, True, None),
    (2, 2, 2, 400, 700, 96, True, 200, True, [700, 350]),
    (1, 4, 2, 300, 500, 256, True, 129, True, None),
    (1, 4, 2, 300, 500, 256, False, 64, False, None),
    (1, 2, 2, 333, 200, 128, True, 50, True, None),       # Sq > Sk: leading rows see no key
    (1, 2, 2, 1000, 1000, 128, False, 0, True, None),     # sinks only (256-key kernel)
    (1, 2, 1, 1000, 1500, 96, False, 0, True, [1433]),    # sinks only (256-key kernel), d = 96
    (1, 1, 1, 16384, 16384, 64, False, 0, True, None),    # sinks through the split-block merge
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,d,causal,window,sinks_on,lengths", PREFILL,
                         ids=[f"b{c[0]}h{c[1]}q{c[3]}k{c[4]}d{c[5]}{'c' if c[6] else 'n'}"
                              f"w{c[7]}{'s' if c[8] else ''}" for c in PREFILL])
def test_prefill_window_and_sinks(B, Hq, Hkv, Sq, Sk, d, causal, window, sinks_on, lengths):
    from attention_forward_blackwell_gb300 import binding, inputs
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=700 + Sq + window, device="cuda",
                           lengths=lengths)
    if lengths is not None:
        inputs.poison_beyond_lengths(x.k, x.seqlens_k)
        inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    sinks = _sinks(Hq, 31 + Sq, sinks_on)
    scale = 1.0 / math.sqrt(d)
    o, lse = binding.prefill(x.q, x.k, x.v, scale=scale, causal=causal, seqlens_k=x.seqlens_k,
                             window=window, sinks=sinks)
    torch.cuda.synchronize()
    check_device_error()
    rows = None
    if B * Hq * Sq > 4096:   # large case: sampled rows
        rng = np.random.default_rng(Sq)
        rows = np.unique(np.concatenate([np.arange(300), rng.integers(0, B * Hq * Sq, 200),
                                         np.arange(B * Hq * Sq - 300, B * Hq * Sq)]))
    ro, rl = _oracle(x, scale, causal, window, sinks, rows)
    if rows is None:
        compare(o, lse, ro, rl, f"prefill window={window} sinks={sinks_on}")
    else:
        idx = torch.from_numpy(rows).cuda()
        compare(o.view(-1, d)[idx], lse.view(-1)[idx], ro, rl,
                f"prefill window={window} sinks={sinks_on} (sampled)")
    free_cuda()


@pytest.mark.parametrize("d", [64, 128])
def test_prefill_minus_inf_sinks_and_wide_window_are_identities(d):
    """sinks = -inf give exactly the plain result (the same kernel, no block
    split changes the rounding); a window wider than every row's keys gives
    the plain result exactly where the same kernel runs both (head_dim 64),
    and within the parity tolerance of it otherwise (head_dim 128: windowed
    launches run the two-tile kernel, plain ones the 256-key kernel)."""
    from attention_forward_blackwell_gb300 import binding, inputs
    x = inputs.make_inputs(1, 2, 2, 700, 700, d, tag=720, device="cuda")
    o0, l0 = binding.prefill(x.q, x.k, x.v, causal=True)
    neg = torch.full((2,), float("-inf"), device="cuda")
    o1, l1 = binding.prefill(x.q, x.k, x.v, causal=True, sinks=neg)
    o2, l2 = binding.prefill(x.q, x.k, x.v, causal=True, window=100000)
    torch.cuda.synchronize()
    check_device_error()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    if d == 64:
        assert torch.equal(o0, o2) and torch.equal(l0, l2)
    else:
        ro, rl = _oracle(x, 1.0 / math.sqrt(d), True, 0, None)
        compare(o2, l2, ro, rl, "window 100000")
        compare(o0, l0, ro, rl, "no window")


DECODE = [
    # B, Hq, Hkv, Sq, d, causal, window, sinks
    (8, 8, 2, 1, 128, False, 1, False),
    (8, 8, 2, 1, 128, False, 64, True),
    (8, 8, 2, 1, 128, False, 1000, True),
    (8, 8, 2, 1, 64, False, 0, True),
    (4, 16, 4, 4, 128, True, 300, True),
    (4, 4, 1, 1, 256, False, 513, False),
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,d,causal,window,sinks_on", DECODE,
                         ids=[f"b{c[0]}h{c[1]}x{c[2]}q{c[3]}d{c[4]}w{c[6]}{'s' if c[7] else ''}"
                              for c in DECODE])
def test_decode_window_and_sinks(B, Hq, Hkv, Sq, d, causal, window, sinks_on):
    from attention_forward_blackwell_gb300 import binding, inputs
    Sk = 5000
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=740 + window, device="cuda",
                           lengths=(1, Sk))
    inputs.poison_beyond_lengths(x.k, x.seqlens_k)
    inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    sinks = _sinks(Hq, 41 + window, sinks_on)
    scale = 1.0 / math.sqrt(d)
    o, lse = binding.decode(x.q, x.k, x.v, scale=scale, causal=causal, seqlens_k=x.seqlens_k,
                            window=window, sinks=sinks)
    torch.cuda.synchronize()
    check_device_error()
    ro, rl = _oracle(x, scale, causal, window, sinks)
    compare(o, lse, ro, rl, f"decode window={window} sinks={sinks_on}")


def test_no_keys_with_sinks_gives_sink_lse():
    """Sk = 0, or every key outside the window: O = 0 and LSE = sinks[h]."""
    from attention_forward_blackwell_gb300 import binding
    q = torch.randn(2, 3, 4, 64, device="cuda").bfloat16()
    k = torch.empty(2, 3, 0, 64, device="cuda", dtype=torch.bfloat16)
    sinks = torch.tensor([0.5, -1.0, 2.0], device="cuda")
    for fn in (binding.prefill, binding.decode):
        o, lse = fn(q, k, k, sinks=sinks)
        torch.cuda.synchronize()
        assert torch.all(o == 0)
        assert torch.equal(lse, sinks.view(1, 3, 1).expand(2, 3, 4).contiguous())
