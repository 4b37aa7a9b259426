"""The persistent 256-key prefill kernel (head_dim 96 and 128, dense, no
window, causal or not) against the fp64 oracle.

One CTA per SM walks units of 128 query rows; each score block is 256 keys
(one N = 256 score MMA per K-step), the two softmax warpgroups take 128 keys
each and exchange their block maxima, P has tensor-memory columns of its own
and the next block's score MMA runs during the softmax ("b200-flash-attention4-
planner" A1, E.3-E.8).  These shapes exercise: ragged query and key lengths
(a last block of 1 key, a value half with no valid key), per-sequence key
lengths with NaN padding and empty sequences (units written as O = 0,
LSE = -inf), one query row, one key, GQA, attention sinks, the causal mask
(bottom-right aligned, with rows that see no key when Sq > Sk), 24 seeded
random shapes (head_dim, GQA ratio, ragged lengths, causal), many units
per CTA (running barrier phases over the CTA's units, heaviest-first causal
units), repeated launches and a CUDA graph replay.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_parity import (THREADS, check_device_error, compare, free_cuda, oracle_for,
                        sample_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from attention_forward_blackwell_gb300 import build
    build.build()
    yield
    free_cuda()


def _assert_wide(B, Hq, Sq, Sk, d, causal=False):
    from attention_forward_blackwell_gb300 import binding
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = binding.debug_prefill_plan_ex(B, Hq, Sq, Sk, d, causal, n_sms)
    assert p.keys_per_block == 256 and p.rows_per_unit == 128 and p.persistent, p
    return p


def _run(x, scale, sinks=None, causal=False):
    from attention_forward_blackwell_gb300 import binding
    o, lse = binding.prefill(x.q, x.k, x.v, scale=scale, causal=causal, seqlens_k=x.seqlens_k,
                             sinks=sinks)
    torch.cuda.synchronize()
    check_device_error()
    return o, lse


FULL = [
    # B, Hq, Hkv, Sq, Sk, d, lengths: every output element against the oracle
    (1, 2, 1, 300, 1000, 96, None),            # GQA, ragged query and key tails
    (2, 3, 3, 129, 257, 128, None),            # a 1-row query tail, a last block of 1 key
    (1, 1, 1, 1000, 1, 128, None),             # one key
    (1, 2, 2, 1, 5000, 96, None),              # one query row
    (3, 2, 1, 200, 1300, 128, [1300, 0, 513]), # empty sequence; a value half with no key
    (2, 4, 2, 384, 768, 96, [700, 256]),       # a length of exactly one block
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,d,lengths", FULL,
                         ids=[f"b{c[0]}h{c[1]}x{c[2]}q{c[3]}k{c[4]}d{c[5]}" for c in FULL])
def test_every_element(B, Hq, Hkv, Sq, Sk, d, lengths, causal):
    from attention_forward_blackwell_gb300 import inputs
    _assert_wide(B, Hq, Sq, Sk, d, causal)
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=1500 + Sq + d, device="cuda",
                           lengths=lengths)
    if lengths is not None:
        inputs.poison_beyond_lengths(x.k, x.seqlens_k)
        inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(x, scale, causal=causal)
    if lengths is not None:
        for b, L in enumerate(lengths):
            if L == 0:
                assert torch.all(o[b] == 0) and torch.all(torch.isneginf(lse[b]))
    ro, rl = oracle_for(x, scale, causal)
    compare(o, lse, ro, rl, f"256-key kernel {B, Hq, Hkv, Sq, Sk, d} causal={causal}")
    free_cuda()


MANY = [
    # B, Hq, Hkv, S, d: more units than SMs, so every CTA walks 6-7 units
    (8, 16, 4, 1024, 128),
    (4, 16, 16, 2048, 96),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,S,d", MANY, ids=[f"b{c[0]}h{c[1]}s{c[3]}d{c[4]}" for c in MANY])
def test_many_units_per_cta(B, Hq, Hkv, S, d, causal):
    """Sampled rows (unit edges of a few heads plus random rows) against the
    oracle, and the first and last head in full."""
    from attention_forward_blackwell_gb300 import inputs
    p = _assert_wide(B, Hq, S, S, d, causal)
    assert p.n_full > 4 * torch.cuda.get_device_properties(0).multi_processor_count
    x = inputs.make_inputs(B, Hq, Hkv, S, S, d, tag=1600 + d, device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(x, scale, causal=causal)
    rows = np.unique(np.concatenate([sample_rows(B, Hq, S, n_random=400, seed=S + d),
                                     np.arange(S), np.arange(B * Hq * S - S, B * Hq * S)]))
    ro, rl = oracle_for(x, scale, causal, rows=rows)
    idx = torch.from_numpy(rows).cuda()
    compare(o.view(-1, d)[idx], lse.view(-1)[idx], ro, rl,
            f"many units {B, Hq, Hkv, S, d} causal={causal}")
    del x, o, lse
    free_cuda()


def test_sinks_over_many_units():
    """Attention sinks join each row's normaliser in the epilogue."""
    from attention_forward_blackwell_gb300 import inputs
    B, Hq, S, d = 2, 8, 2048, 96
    _assert_wide(B, Hq, S, S, d)
    x = inputs.make_inputs(B, Hq, Hq, S, S, d, tag=1700, device="cuda")
    g = torch.Generator().manual_seed(17)
    sinks = (2.0 * torch.randn(Hq, generator=g)).float().cuda()
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(x, scale, sinks=sinks)
    rows = sample_rows(B, Hq, S, n_random=300, seed=5)
    ro, rl = oracle.attention_fwd(inputs.bf16_bits(x.q), inputs.bf16_bits(x.k),
                                  inputs.bf16_bits(x.v), scale=scale, causal=False,
                                  seqlens_k=None, rows=rows, threads=THREADS,
                                  window=0, sinks=sinks.cpu().double().numpy())
    idx = torch.from_numpy(rows).cuda()
    compare(o.view(-1, d)[idx], lse.view(-1)[idx], ro, rl, "256-key kernel with sinks")
    free_cuda()


def test_repeated_launches_are_bit_equal():
    """Units are never split, so every launch gives the same bits."""
    from attention_forward_blackwell_gb300 import inputs
    x = inputs.make_inputs(2, 16, 4, 2048, 2048, 128, tag=1800, device="cuda")
    o1, l1 = _run(x, 0.088)
    for _ in range(5):
        o2, l2 = _run(x, 0.088)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    free_cuda()


def test_barrier_protocol_stress():
    """Back-to-back launches of one-block units (every unit boundary is also
    a block boundary): no wait may time out, every result equals the first."""
    from attention_forward_blackwell_gb300 import binding, inputs
    x = inputs.make_inputs(3, 8, 8, 300, 200, 128, tag=1850, device="cuda")
    o0, l0 = _run(x, 0.09)
    for _ in range(40):
        o, l = binding.prefill(x.q, x.k, x.v, scale=0.09)
    torch.cuda.synchronize()
    check_device_error()
    assert torch.equal(o, o0) and torch.equal(l, l0)


def test_replay_in_a_cuda_graph():
    from attention_forward_blackwell_gb300 import binding, inputs
    x = inputs.make_inputs(1, 4, 2, 1024, 3000, 96, tag=1900, device="cuda")
    o_ref, l_ref = binding.prefill(x.q, x.k, x.v)
    o = torch.empty_like(x.q)
    lse = torch.empty(1, 4, 1024, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):   # warm-up outside the capture
        binding.prefill(x.q, x.k, x.v, out=o, lse=lse)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.prefill(x.q, x.k, x.v, out=o, lse=lse)
    for _ in range(3):
        o.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        check_device_error()
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    free_cuda()


def _random_cases(n, seed):
    """Seeded random small shapes for the 256-key kernel: head_dim 96 / 128,
    causal or not, GQA ratio 1-4, Sq and Sk from 1 to 1,500 (ragged against
    the 128-row units and 256-key blocks), optional per-sequence key lengths
    with zeros."""
    import random
    rng = random.Random(seed)
    cases = []
    for _ in range(n):
        d = rng.choice([96, 128])
        hkv = rng.choice([1, 2])
        hq = hkv * rng.choice([1, 2, 4])
        B = rng.choice([1, 2, 3])
        sq = rng.randint(1, 1500)
        sk = rng.randint(1, 1500)
        lens = None
        if rng.random() < 0.4:
            lens = [rng.choice([0, rng.randint(1, sk), sk]) for _ in range(B)]
        cases.append((B, hq, hkv, sq, sk, d, rng.random() < 0.5, lens))
    return cases


RANDOM = _random_cases(24, seed=2026)


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,d,causal,lengths", RANDOM,
                         ids=[f"r{i}" for i in range(len(RANDOM))])
def test_random_shapes_every_element(B, Hq, Hkv, Sq, Sk, d, causal, lengths):
    from attention_forward_blackwell_gb300 import inputs
    _assert_wide(B, Hq, Sq, Sk, d, causal)
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=2000 + Sq + Sk, device="cuda",
                           lengths=lengths)
    if lengths is not None:
        inputs.poison_beyond_lengths(x.k, x.seqlens_k)
        inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(x, scale, causal=causal)
    ro, rl = oracle_for(x, scale, causal)
    compare(o, lse, ro, rl, f"random {B, Hq, Hkv, Sq, Sk, d} causal={causal} lengths={lengths}")
    free_cuda()


SPLIT = [
    # B, Hq, Hkv, Sq, Sk, d, lengths: at most half a wave of units, each cut
    # along the keys into pieces of >= 4 key blocks over several CTAs
    (1, 2, 2, 300, 5000, 128, None),               # 6 units x 5 pieces
    (1, 1, 1, 128, 65536, 96, None),               # one unit x 8 pieces
    (2, 2, 1, 200, 6000, 128, [6000, 1100]),       # later pieces of a short sequence: no key
    (1, 4, 2, 129, 4097, 96, None),                # ragged: a last block of one key
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,d,lengths", SPLIT,
                         ids=[f"b{c[0]}h{c[1]}q{c[3]}k{c[4]}d{c[5]}" for c in SPLIT])
def test_split_units_every_element(B, Hq, Hkv, Sq, Sk, d, lengths):
    """Pieces write unnormalised O, row max and row sum to scratch; the last
    to arrive merges them (rebasing each to the common max) and stores O and
    LSE."""
    from attention_forward_blackwell_gb300 import binding, inputs
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = _assert_wide(B, Hq, Sq, Sk, d)
    assert p.n_full == 0 and p.split > 1 and p.n_tail * p.split <= n_sms, p
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=2100 + Sq + Sk, device="cuda",
                           lengths=lengths)
    if lengths is not None:
        inputs.poison_beyond_lengths(x.k, x.seqlens_k)
        inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(x, scale)
    ro, rl = oracle_for(x, scale, False)
    compare(o, lse, ro, rl, f"split {B, Hq, Hkv, Sq, Sk, d} x{p.split} lengths={lengths}")
    free_cuda()


def test_split_units_with_sinks_packed_and_replayed():
    """Head-packed units split along the keys (4 units of 8 heads x 16
    queries, 8 pieces each), with sinks; bit-equal over repeated launches and
    a CUDA graph replay (the arrival counters reset themselves)."""
    from attention_forward_blackwell_gb300 import binding, inputs
    B, Hq, Hkv, Sq, Sk, d = 1, 32, 4, 16, 8192, 128
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = binding.debug_prefill_plan_gqa(B, Hq, Hkv, Sq, Sk, d, False, n_sms)
    assert p.pack == 8 and p.n_full == 0 and p.n_tail == 4 and p.split == 8, p
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=2200, device="cuda")
    g = torch.Generator().manual_seed(29)
    sinks = (2.0 * torch.randn(Hq, generator=g)).float().cuda()
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(x, scale, sinks=sinks)
    ro, rl = oracle.attention_fwd(inputs.bf16_bits(x.q), inputs.bf16_bits(x.k),
                                  inputs.bf16_bits(x.v), scale=scale, causal=False,
                                  threads=THREADS, sinks=sinks.cpu().double().numpy())
    compare(o, lse, ro, rl, "packed split with sinks")
    for _ in range(3):
        o2, l2 = _run(x, scale, sinks=sinks)
        assert torch.equal(o, o2) and torch.equal(lse, l2)
    o3 = torch.empty_like(o)
    l3 = torch.empty_like(lse)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        binding.prefill(x.q, x.k, x.v, scale=scale, sinks=sinks, out=o3, lse=l3)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        binding.prefill(x.q, x.k, x.v, scale=scale, sinks=sinks, out=o3, lse=l3)
    for _ in range(3):
        o3.zero_()
        l3.zero_()
        graph.replay()
        torch.cuda.synchronize()
        check_device_error()
        assert torch.equal(o3, o) and torch.equal(l3, lse)
    free_cuda()
