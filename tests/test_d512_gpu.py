"""Prefill at head_dim 512 (two CTAs per query tile, each computing the
scores and one 256-column half of O) against the fp64 oracle: dense,
causal, grouped heads, ragged tails, key lengths with poisoned padding,
sliding window and sinks, paged and packed key/value layouts, and sampled
rows of the 2 x 8 x 4096 x 4096 workload in its timed launch configuration."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_parity import THREADS, check_device_error, compare, free_cuda, oracle_for

pytestmark = pytest.mark.gpu

D = 512


@pytest.fixture(scope="module", autouse=True)
def built():
    from attention_forward_blackwell_gb300 import build
    build.build()
    yield
    free_cuda()


def _oracle(x, scale, causal, window=0, sinks=None, rows=None):
    from attention_forward_blackwell_gb300 import inputs
    lens = None if x.seqlens_k is None else x.seqlens_k.cpu().tolist()
    sk = None if sinks is None else sinks.cpu().double().numpy()
    return oracle.attention_fwd(inputs.bf16_bits(x.q), inputs.bf16_bits(x.k),
                                inputs.bf16_bits(x.v), scale=scale, causal=causal,
                                seqlens_k=lens, rows=rows, threads=THREADS,
                                window=window, sinks=sk)


DENSE = [
    # B, Hq, Hkv, Sq, Sk, causal, window, sinks, lengths
    (1, 1, 1, 128, 128, False, 0, False, None),          # one tile, one key block
    (1, 2, 2, 300, 300, False, 0, False, None),          # ragged query and key tails
    (1, 2, 2, 300, 300, True, 0, False, None),
    (2, 4, 2, 257, 700, True, 0, False, None),           # GQA 2:1, bottom-right causal
    (1, 4, 1, 200, 1100, False, 0, False, None),         # GQA 4:1, nine key blocks
    (2, 2, 2, 300, 640, False, 0, False, [640, 1]),      # key lengths, padding poisoned
    (3, 2, 1, 256, 512, True, 0, False, [512, 300, 0]),  # an entry without keys
    (1, 2, 2, 400, 400, True, 100, True, None),          # window + sinks
    (1, 2, 2, 333, 200, False, 64, True, None),          # Sq > Sk, window
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,causal,window,sinks_on,lengths", DENSE,
                         ids=[f"b{c[0]}h{c[1]}x{c[2]}q{c[3]}k{c[4]}{'c' if c[5] else 'n'}"
                              f"w{c[6]}{'s' if c[7] else ''}{'L' if c[8] else ''}"
                              for c in DENSE])
def test_prefill_d512(B, Hq, Hkv, Sq, Sk, causal, window, sinks_on, lengths):
    from attention_forward_blackwell_gb300 import binding, inputs
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, D, tag=5120 + Sq + Sk, device="cuda",
                           lengths=lengths)
    if lengths is not None:
        inputs.poison_beyond_lengths(x.k, x.seqlens_k)
        inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    sinks = None
    if sinks_on:
        g = torch.Generator().manual_seed(51 + Sq)
        sinks = (2.0 * torch.randn(Hq, generator=g)).float().cuda()
    scale = 1.0 / math.sqrt(D)
    # guard rows after the output: nothing may be written past it
    o_big = torch.full((B * Hq * Sq + 64, D), float("nan"), device="cuda", dtype=torch.bfloat16)
    out = o_big[:B * Hq * Sq].view(B, Hq, Sq, D)
    o, lse = binding.prefill(x.q, x.k, x.v, scale=scale, causal=causal, seqlens_k=x.seqlens_k,
                             window=window, sinks=sinks, out=out)
    torch.cuda.synchronize()
    check_device_error()
    assert torch.isnan(o_big[B * Hq * Sq:].float()).all()
    ro, rl = _oracle(x, scale, causal, window, sinks)
    compare(o, lse, ro, rl, f"d512 B={B} Hq={Hq} Sq={Sq} Sk={Sk}")
    free_cuda()


def test_prefill_d512_workload_sampled():
    """The 2 x 8 x 4096 x 4096 workload (non-causal and causal) in the launch
    configuration the benchmark times; tile edges and random rows against the
    oracle row by row."""
    from attention_forward_blackwell_gb300 import binding, inputs, workloads as W
    from gpu_parity import sample_rows
    for w in (W.PREFILL_D512, W.PREFILL_D512_CAUSAL):
        x = inputs.make_inputs(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, tag=w.tag, device="cuda")
        o, lse = binding.prefill(x.q, x.k, x.v, scale=w.scale, causal=w.causal)
        torch.cuda.synchronize()
        check_device_error()
        rows = sample_rows(w.B, w.Hq, w.Sq, n_random=160, seed=w.tag)
        ro, rl = oracle_for(x, w.scale, w.causal, rows=rows)
        idx = torch.from_numpy(rows).cuda()
        compare(o.view(-1, w.d)[idx], lse.view(-1)[idx], ro, rl, f"{w.name} (sampled)")
        del x, o, lse
        free_cuda()


def test_prefill_d512_paged_matches_contiguous():
    """Shuffled, NaN-poisoned pages of 128 keys: the oracle, and bit for bit
    the contiguous call on the same keys."""
    from attention_forward_blackwell_gb300 import binding, inputs
    from gpu_parity import to_pages
    B, Hq, Hkv, Sq, Sk = 2, 4, 2, 200, 640
    lengths = [640, 333]
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, D, tag=5200, device="cuda", lengths=lengths)
    kc, vc, table, _ = to_pages(x.k, x.v, lengths, 128, seed=5)
    scale = 1.0 / math.sqrt(D)
    o, lse = binding.prefill_paged(x.q, kc, vc, table, x.seqlens_k, scale=scale, causal=True)
    torch.cuda.synchronize()
    check_device_error()
    ro, rl = oracle_for(x, scale, True)
    compare(o, lse, ro, rl, "d512 paged")
    o2, l2 = binding.prefill(x.q, x.k, x.v, scale=scale, causal=True, seqlens_k=x.seqlens_k)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, l2)
    free_cuda()


def test_prefill_d512_packed_sequences():
    """Packed variable-length sequences (a tile past a sequence's end is
    stored row by row, at the CTA's column offset)."""
    from attention_forward_blackwell_gb300 import binding, inputs
    lens_q, lens_k = [1, 200, 77], [300, 200, 500]
    Hq, Hkv = 2, 1
    q = inputs.randn_bf16((sum(lens_q), Hq, D), 5301, "cuda")
    k = inputs.randn_bf16((sum(lens_k), Hkv, D), 5302, "cuda")
    v = inputs.randn_bf16((sum(lens_k), Hkv, D), 5303, "cuda")
    cq = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32, device="cuda")
    ck = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(D)
    total_q = q.shape[0]
    o_big = torch.full((total_q + 8, Hq, D), float("nan"), device="cuda", dtype=torch.bfloat16)
    o, lse = binding.prefill_varlen(q, k, v, cq, ck, max(lens_q), max(lens_k), scale=scale,
                                    causal=True, out=o_big[:total_q])
    torch.cuda.synchronize()
    check_device_error()
    assert torch.isnan(o_big[total_q:].float()).all()
    qs = np.concatenate([[0], np.cumsum(lens_q)])
    ks = np.concatenate([[0], np.cumsum(lens_k)])

    def seq(t, a, b):
        return t[a:b].permute(1, 0, 2).unsqueeze(0).contiguous()

    for b in range(len(lens_q)):
        qb, kb, vb = seq(q, qs[b], qs[b + 1]), seq(k, ks[b], ks[b + 1]), seq(v, ks[b], ks[b + 1])
        ro, rl = oracle.attention_fwd(inputs.bf16_bits(qb), inputs.bf16_bits(kb),
                                      inputs.bf16_bits(vb), scale=scale, causal=True,
                                      threads=THREADS)
        compare(seq(o, qs[b], qs[b + 1]), lse[:, qs[b]:qs[b + 1]].unsqueeze(0), ro, rl,
                f"d512 packed seq {b}")
    free_cuda()


def test_prefill_d512_halves_are_independent_of_each_other():
    """O's two column halves come from different CTAs with the same scores:
    V with its second half zeroed gives exactly the first half of O and zeros,
    and LSE (stored by the first CTA) does not depend on V."""
    from attention_forward_blackwell_gb300 import binding, inputs
    x = inputs.make_inputs(1, 2, 2, 300, 500, D, tag=5400, device="cuda")
    o, lse = binding.prefill(x.q, x.k, x.v, causal=True)
    v2 = x.v.clone()
    v2[..., D // 2:] = 0
    o2, lse2 = binding.prefill(x.q, x.k, v2, causal=True)
    torch.cuda.synchronize()
    check_device_error()
    assert torch.equal(o2[..., :D // 2], o[..., :D // 2])
    assert torch.all(o2[..., D // 2:] == 0)
    assert torch.equal(lse2, lse)


def test_prefill_d512_extreme_logits_one_hot_key():
    """K*8 and one key whose score is 60 above the rest for every query: the
    row's weight is all on that key (LSE > 55), and both column halves of O
    reproduce its value row; the rebase path runs whenever the max jumps."""
    from attention_forward_blackwell_gb300 import binding, inputs
    x = inputs.make_inputs(1, 2, 2, 300, 300, D, tag=5500, device="cuda", k_scale=8.0)
    x.q[..., 0] = 4.0
    x.k[..., 17, :] = 0.0
    x.k[..., 17, 0] = 60.0 * math.sqrt(D) / 4.0
    scale = 1.0 / math.sqrt(D)
    o, lse = binding.prefill(x.q, x.k, x.v, scale=scale)
    torch.cuda.synchronize()
    check_device_error()
    ro, rl = oracle_for(x, scale, False)
    compare(o, lse, ro, rl, "d512 extreme logits")
    assert float(lse.min()) > 55.0
    assert (o.float() - x.v[:, :, 17:18].float()).abs().max().item() < 2e-2


def test_prefill_d512_replays_in_a_cuda_graph():
    """Captured in a CUDA graph and replayed: every replay equals the eager
    result bit for bit."""
    from attention_forward_blackwell_gb300 import binding, inputs
    x = inputs.make_inputs(1, 4, 2, 700, 700, D, tag=5600, device="cuda")
    o_ref, l_ref = binding.prefill(x.q, x.k, x.v, causal=True)
    o = torch.empty_like(x.q)
    lse = torch.empty(1, 4, 700, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):   # warm-up outside the capture
        binding.prefill(x.q, x.k, x.v, causal=True, out=o, lse=lse)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.prefill(x.q, x.k, x.v, causal=True, out=o, lse=lse)
    for _ in range(3):
        o.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    check_device_error()
