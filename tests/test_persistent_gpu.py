"""Head dimension 256 runs one persistent CTA per SM over many units: tensor
memory, the K/V ring, the score buffers and every barrier carry over from one
unit to the next.  These cases give each CTA several units of different
lengths, including units without keys (written without any signal), ragged
last value tiles (the partial-tile barrier's parity runs on across units),
windows, sinks and paged caches, and compare every row with the fp64 oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_parity import THREADS, check_device_error, compare, free_cuda, oracle_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from attention_forward_blackwell_gb300 import build
    build.build()
    yield
    free_cuda()


def _units(B, Hq, Sq):
    return B * Hq * math.ceil(Sq / 128)


def _no_split(B, Hq, Sq, Sk, causal):
    from attention_forward_blackwell_gb300 import binding
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    n_full, n_tail, split = binding.debug_prefill_plan(B, Hq, Sq, Sk, 256, causal, n_sms)
    return n_tail == 0 and split == 1 and n_full == _units(B, Hq, Sq)


CASES = [
    # B, Hq, Hkv, Sq, Sk, causal, lengths
    (8, 16, 2, 512, 1000, False, [1000, 0, 129, 1, 777, 1000, 0, 300]),
    (8, 16, 2, 512, 1000, True, [1000, 0, 129, 1, 777, 1000, 0, 300]),
    (6, 16, 4, 640, 640, True, None),
    (2, 64, 8, 1024, 1024, True, None),
    (3, 32, 32, 512, 2050, False, [2050, 1, 1500]),
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,causal,lengths", CASES,
                         ids=[f"b{c[0]}h{c[1]}q{c[3]}k{c[4]}{'c' if c[5] else 'n'}"
                              f"{'L' if c[6] else ''}" for c in CASES])
def test_persistent_units_every_row(B, Hq, Hkv, Sq, Sk, causal, lengths):
    from attention_forward_blackwell_gb300 import binding, inputs
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert _units(B, Hq, Sq) > 2 * n_sms, "each CTA should walk several units"
    assert _no_split(B, Hq, Sq, Sk, causal)
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, 256, tag=1700 + Sq + Sk, device="cuda",
                           lengths=lengths)
    if lengths is not None:
        inputs.poison_beyond_lengths(x.k, x.seqlens_k)
        inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    scale = 1.0 / math.sqrt(256)
    o, lse = binding.prefill(x.q, x.k, x.v, scale=scale, causal=causal, seqlens_k=x.seqlens_k)
    torch.cuda.synchronize()
    check_device_error()
    ro, rl = oracle_for(x, scale, causal)
    compare(o, lse, ro, rl, f"persistent d256 B={B} Hq={Hq} Sq={Sq} Sk={Sk} causal={causal}")
    # repeated launches give the same bits (no state leaks between launches)
    o2, l2 = binding.prefill(x.q, x.k, x.v, scale=scale, causal=causal, seqlens_k=x.seqlens_k)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, l2)
    free_cuda()


def test_persistent_window_and_sinks():
    from attention_forward_blackwell_gb300 import binding, inputs
    B, Hq, Hkv, Sq, Sk, window = 4, 16, 4, 1024, 1024, 200
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, 256, tag=1750, device="cuda",
                           lengths=[1024, 700, 5, 1000])
    g = torch.Generator().manual_seed(1751)
    sinks = (2.0 * torch.randn(Hq, generator=g)).float().cuda()
    scale = 1.0 / math.sqrt(256)
    for causal in (True, False):
        assert _no_split(B, Hq, Sq, Sk, True)   # windowed units are never split
        o, lse = binding.prefill(x.q, x.k, x.v, scale=scale, causal=causal,
                                 seqlens_k=x.seqlens_k, window=window, sinks=sinks)
        torch.cuda.synchronize()
        check_device_error()
        ro, rl = oracle.attention_fwd(inputs.bf16_bits(x.q), inputs.bf16_bits(x.k),
                                      inputs.bf16_bits(x.v), scale=scale, causal=causal,
                                      seqlens_k=x.seqlens_k.cpu().tolist(), threads=THREADS,
                                      window=window, sinks=sinks.cpu().double().numpy())
        compare(o, lse, ro, rl, f"persistent d256 window={window} sinks causal={causal}")
    free_cuda()


def test_persistent_paged_matches_contiguous():
    from attention_forward_blackwell_gb300 import binding, inputs
    from gpu_parity import to_pages
    B, Hq, Hkv, Sq, Sk, P = 6, 16, 2, 512, 1024, 256
    lens = [1024, 0, 300, 1024, 129, 777]
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, 256, tag=1760, device="cuda", lengths=lens)
    kc, vc, table, _ = to_pages(x.k, x.v, lens, P, seed=1761)
    scale = 1.0 / math.sqrt(256)
    for causal in (True, False):
        assert _no_split(B, Hq, Sq, Sk, causal)
        o, lse = binding.prefill_paged(x.q, kc, vc, table, x.seqlens_k, scale=scale,
                                       causal=causal)
        o2, l2 = binding.prefill(x.q, x.k, x.v, scale=scale, causal=causal,
                                 seqlens_k=x.seqlens_k)
        torch.cuda.synchronize()
        check_device_error()
        assert torch.equal(o, o2) and torch.equal(lse, l2)
        rows = np.arange(0, B * Hq * Sq, 7, dtype=np.int64)
        ro, rl = oracle_for(x, scale, causal, rows=rows)
        compare(o.reshape(-1, 256)[torch.from_numpy(rows).cuda()],
                lse.reshape(-1)[torch.from_numpy(rows).cuda()], ro, rl,
                f"persistent d256 paged causal={causal}")
    free_cuda()
