"""GQA head packing in the 256-key prefill kernel against the fp64 oracle.

With short queries (sq <= 64) and hq / hkv = G > 1, one 128-row tile holds
P query heads of a kv group x 128 / P query positions, all reading the same
K/V tiles ("b200-flash-attention4-planner" E.7: explicit head mapping and
reuse).  These cases cover every P (2, 4, 8) and rows-per-head (16, 32, 64),
query lengths that fill a head's rows or leave them ragged, the causal mask
(bottom-right aligned per row position, rows that see no key), per-sequence
key lengths with NaN padding and empty sequences, attention sinks (a per-row
head), many units per CTA, and repeated launches.
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


def _pack(B, Hq, Hkv, Sq, Sk, d, causal):
    from attention_forward_blackwell_gb300 import binding
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    return binding.debug_prefill_plan_gqa(B, Hq, Hkv, Sq, Sk, d, causal, n_sms).pack


CASES = [
    # B, Hq, Hkv, Sq, Sk, d, lengths, expected heads per tile
    (2, 8, 1, 1, 700, 128, None, 8),              # 8 heads x 16 rows, one query each
    (1, 16, 2, 16, 3000, 96, None, 8),            # full 16-row heads
    (3, 8, 2, 5, 1300, 128, [1300, 0, 257], 4),   # G = 4: 4 heads x 32 rows; an empty sequence
    (2, 8, 1, 17, 999, 128, [600, 999], 4),       # 17 rows: 32 per head
    (1, 32, 4, 32, 2048, 128, None, 4),
    (2, 4, 2, 40, 513, 96, None, 2),              # 64 rows per head, ragged
    (1, 12, 2, 64, 1500, 128, [1111], 2),         # G = 6: two heads per tile
    (2, 8, 4, 3, 256, 128, None, 2),              # G = 2
    (1, 8, 1, 1, 1, 128, None, 8),                # one key
    (2, 16, 2, 64, 64, 96, None, 2),              # short square: the causal triangle
    (1, 8, 1, 16, 257, 128, [257], 8),            # a last key block of one key
    (2, 8, 2, 30, 20, 128, [20, 7], 4),           # Sq > Sk: causal rows without keys
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,d,lengths,pack", CASES,
                         ids=[f"b{c[0]}h{c[1]}x{c[2]}q{c[3]}k{c[4]}d{c[5]}" for c in CASES])
def test_packed_every_element(B, Hq, Hkv, Sq, Sk, d, lengths, pack, causal):
    from attention_forward_blackwell_gb300 import binding, inputs
    assert _pack(B, Hq, Hkv, Sq, Sk, d, causal) == pack
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=4100 + Sq + Sk, device="cuda",
                           lengths=lengths)
    if lengths is not None:
        inputs.poison_beyond_lengths(x.k, x.seqlens_k)
        inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    scale = 1.0 / math.sqrt(d)
    o, lse = binding.prefill(x.q, x.k, x.v, scale=scale, causal=causal, seqlens_k=x.seqlens_k)
    torch.cuda.synchronize()
    check_device_error()
    if lengths is not None:
        for b, L in enumerate(lengths):
            if L == 0:
                assert torch.all(o[b] == 0) and torch.all(torch.isneginf(lse[b]))
    ro, rl = oracle_for(x, scale, causal)
    compare(o, lse, ro, rl, f"packed {B, Hq, Hkv, Sq, Sk, d} P={pack} causal={causal}")
    free_cuda()


def test_packed_with_sinks():
    """The sink of each row's own head joins its normaliser."""
    from attention_forward_blackwell_gb300 import binding, inputs
    B, Hq, Hkv, Sq, Sk, d = 2, 16, 2, 12, 2500, 128
    assert _pack(B, Hq, Hkv, Sq, Sk, d, True) == 8
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=4200, device="cuda")
    g = torch.Generator().manual_seed(23)
    sinks = (2.0 * torch.randn(Hq, generator=g)).float().cuda()
    scale = 1.0 / math.sqrt(d)
    for causal in (False, True):
        o, lse = binding.prefill(x.q, x.k, x.v, scale=scale, causal=causal, sinks=sinks)
        torch.cuda.synchronize()
        check_device_error()
        ro, rl = oracle.attention_fwd(inputs.bf16_bits(x.q), inputs.bf16_bits(x.k),
                                      inputs.bf16_bits(x.v), scale=scale, causal=causal,
                                      threads=THREADS, sinks=sinks.cpu().double().numpy())
        compare(o, lse, ro, rl, f"packed with sinks causal={causal}")
    free_cuda()


def test_packed_many_units_and_repeats():
    """A chunked-prefill shape: 64 sequences x 4 kv groups of 8 heads, 16 new
    queries each over 4,096 keys -- 256 packed units (2,048 unpacked) walked
    by the persistent CTAs; sampled rows against the oracle, then bit-equal
    results over repeated launches."""
    from attention_forward_blackwell_gb300 import binding, inputs
    B, Hq, Hkv, Sq, Sk, d = 64, 32, 4, 16, 4096, 128
    assert _pack(B, Hq, Hkv, Sq, Sk, d, True) == 8
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=4300, device="cuda",
                           lengths=(1, Sk))
    inputs.poison_beyond_lengths(x.k, x.seqlens_k)
    inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    scale = 1.0 / math.sqrt(d)
    o, lse = binding.prefill(x.q, x.k, x.v, scale=scale, causal=True, seqlens_k=x.seqlens_k)
    torch.cuda.synchronize()
    check_device_error()
    rng = np.random.default_rng(5)
    total = B * Hq * Sq
    rows = np.unique(np.concatenate([np.arange(0, 2 * Hq * Sq), rng.integers(0, total, 1500),
                                     np.arange(total - Hq * Sq, total)]))
    ro, rl = oracle_for(x, scale, True, rows=rows)
    idx = torch.from_numpy(rows).cuda()
    compare(o.view(-1, d)[idx], lse.view(-1)[idx], ro, rl, "packed chunked prefill (sampled)")
    for _ in range(3):
        o2, l2 = binding.prefill(x.q, x.k, x.v, scale=scale, causal=True,
                                 seqlens_k=x.seqlens_k)
        torch.cuda.synchronize()
        assert torch.equal(o, o2) and torch.equal(lse, l2)
    check_device_error()
    free_cuda()


DECODE_ROUTED = [
    # B, Hq, Hkv, Sq, Sk, lengths, causal, sinks: R = (Hq / Hkv) * Sq >= 32
    # rows per kv head
    (8, 32, 4, 4, 3000, (1, 3000), True, False),        # 32 units x 32 rows
    (4, 64, 8, 16, 2048, None, False, True),            # 32 x 128
    (6, 16, 2, 16, 5000, [5000, 0, 1, 4999, 2500, 17], True, True),   # 12 x 128
    (12, 32, 2, 2, 700, None, False, False),            # G = 16: 48 x 32
    (1, 64, 8, 8, 9000, (1, 9000), False, True),        # one sequence: 8 units split along the keys
]


def _routed(B, Hq, Hkv, Sq, Sk, causal):
    """Whether fa_fwd_decode takes the packed prefill kernel (head_dim 128)."""
    return Hq // Hkv * Sq >= 32


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,lengths,causal,sinks_on", DECODE_ROUTED,
                         ids=[f"b{c[0]}h{c[1]}x{c[2]}q{c[3]}k{c[4]}" for c in DECODE_ROUTED])
def test_decode_with_many_rows_per_kv_head_runs_the_packed_kernel(B, Hq, Hkv, Sq, Sk, lengths,
                                                                   causal, sinks_on):
    """fa_fwd_decode / fa_fwd_decode_ex at head_dim 128 with >= 32 query rows
    per kv head give fa_fwd_prefill's result bit for bit (the same packed
    kernel ran) and match the oracle on every element."""
    from attention_forward_blackwell_gb300 import binding, inputs
    d = 128
    assert _routed(B, Hq, Hkv, Sq, Sk, causal)
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=4400 + Sq + Sk, device="cuda",
                           lengths=lengths)
    if lengths is not None:
        inputs.poison_beyond_lengths(x.k, x.seqlens_k)
        inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    sinks = None
    if sinks_on:
        g = torch.Generator().manual_seed(Sq + Sk)
        sinks = (2.0 * torch.randn(Hq, generator=g)).float().cuda()
    scale = 1.0 / math.sqrt(d)
    o, lse = binding.decode(x.q, x.k, x.v, scale=scale, causal=causal, seqlens_k=x.seqlens_k,
                            sinks=sinks)
    o2, l2 = binding.prefill(x.q, x.k, x.v, scale=scale, causal=causal, seqlens_k=x.seqlens_k,
                             sinks=sinks)
    torch.cuda.synchronize()
    check_device_error()
    assert torch.equal(o, o2) and torch.equal(lse, l2)
    lens = None if x.seqlens_k is None else x.seqlens_k.cpu().tolist()
    ro, rl = oracle.attention_fwd(inputs.bf16_bits(x.q), inputs.bf16_bits(x.k),
                                  inputs.bf16_bits(x.v), scale=scale, causal=causal,
                                  seqlens_k=lens, threads=THREADS,
                                  sinks=None if sinks is None else sinks.cpu().double().numpy())
    compare(o, lse, ro, rl, f"decode routed {B, Hq, Hkv, Sq, Sk} causal={causal} sinks={sinks_on}")
    # an explicit split count keeps the split-KV kernel (same values within
    # the parity tolerance, not the same bits)
    o3, l3 = binding.decode(x.q, x.k, x.v, scale=scale, causal=causal, seqlens_k=x.seqlens_k,
                            num_splits=3) if sinks is None else (o, lse)
    torch.cuda.synchronize()
    compare(o3, l3, ro, rl, "decode with 3 splits")
    free_cuda()
