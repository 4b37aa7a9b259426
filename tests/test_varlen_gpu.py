"""Prefill over packed variable-length sequences (fa_fwd_prefill_varlen)
against the fp64 oracle run on each sequence alone, and against the dense
kernel run on each sequence alone."""
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


def packed(lens_q, lens_k, Hq, Hkv, d, seed):
    from attention_forward_blackwell_gb300 import inputs
    q = inputs.randn_bf16((sum(lens_q), Hq, d), 5000 + seed, "cuda")
    k = inputs.randn_bf16((sum(lens_k), Hkv, d), 6000 + seed, "cuda")
    v = inputs.randn_bf16((sum(lens_k), Hkv, d), 7000 + seed, "cuda")
    cq = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32, device="cuda")
    ck = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32, device="cuda")
    return q, k, v, cq, ck


def seq(t, a, b):
    """[tokens, heads, d] rows a..b -> dense [1, heads, b - a, d]."""
    return t[a:b].permute(1, 0, 2).unsqueeze(0).contiguous()


CASES = [
    # Hq, Hkv, d, lens_q, lens_k, causal, window, sinks
    (4, 2, 128, [1, 128, 300, 513, 0, 77], [1, 128, 300, 513, 0, 77], True, 0, False),
    (4, 2, 128, [1, 128, 300, 513, 0, 77], [1, 128, 300, 513, 0, 77], False, 0, False),
    (2, 2, 64, [100, 256, 40], [600, 256, 1000], True, 0, False),     # key prefix longer
    (4, 1, 256, [129, 64, 300], [129, 64, 300], True, 0, False),      # GQA 4:1
    (2, 2, 96, [200, 333], [200, 333], True, 64, True),               # window + sinks
    (2, 1, 128, [90, 50, 260], [90, 0, 260], False, 0, True),          # a sequence without keys
    (2, 2, 128, [300, 40], [20, 500], False, 0, False),               # fewer keys than queries
]


@pytest.mark.parametrize("Hq,Hkv,d,lens_q,lens_k,causal,window,sinks_on", CASES,
                         ids=[f"h{c[0]}x{c[1]}d{c[2]}n{len(c[3])}{'c' if c[5] else 'n'}"
                              f"w{c[6]}{'s' if c[7] else ''}" for c in CASES])
def test_prefill_varlen(Hq, Hkv, d, lens_q, lens_k, causal, window, sinks_on):
    from attention_forward_blackwell_gb300 import binding, inputs
    q, k, v, cq, ck = packed(lens_q, lens_k, Hq, Hkv, d, seed=sum(lens_q) + d)
    sinks = None
    if sinks_on:
        g = torch.Generator().manual_seed(77)
        sinks = (2.0 * torch.randn(Hq, generator=g)).float().cuda()
    scale = 1.0 / math.sqrt(d)
    total_q = q.shape[0]
    # guard rows after the output: nothing may be written past total_q
    o_big = torch.full((total_q + 300, Hq, d), float("nan"), device="cuda", dtype=torch.bfloat16)
    out = o_big[:total_q]
    o, lse = binding.prefill_varlen(q, k, v, cq, ck, max(lens_q), max(lens_k), scale=scale,
                                    causal=causal, window=window, sinks=sinks, out=out)
    torch.cuda.synchronize()
    check_device_error()
    assert torch.isnan(o_big[total_q:].float()).all()
    qs = np.concatenate([[0], np.cumsum(lens_q)])
    ks = np.concatenate([[0], np.cumsum(lens_k)])
    sk_np = None if sinks is None else sinks.cpu().double().numpy()
    for b, (lq, lk) in enumerate(zip(lens_q, lens_k)):
        if lq == 0:
            continue
        o_b = seq(o, qs[b], qs[b + 1])
        l_b = lse[:, qs[b]:qs[b + 1]].unsqueeze(0)
        if lk == 0:
            assert torch.all(o_b == 0)
            want = (torch.full((1, Hq, lq), float("-inf"), device="cuda") if sinks is None
                    else sinks.view(1, Hq, 1).expand(1, Hq, lq))
            # (the sink passes through log2 units: equal up to rounding)
            assert torch.allclose(l_b, want, rtol=1e-6, atol=1e-6)
            continue
        qb, kb, vb = seq(q, qs[b], qs[b + 1]), seq(k, ks[b], ks[b + 1]), seq(v, ks[b], ks[b + 1])
        ro, rl = oracle.attention_fwd(inputs.bf16_bits(qb), inputs.bf16_bits(kb),
                                      inputs.bf16_bits(vb), scale=scale, causal=causal,
                                      threads=THREADS, window=window, sinks=sk_np)
        compare(o_b, l_b, ro, rl, f"varlen seq {b} (lq={lq}, lk={lk})")
        # the dense kernel on the sequence alone does the same arithmetic
        # (no key-axis split: causal, windowed or fewer than 16 key blocks;
        # not the 256-key kernel, which takes dense non-causal head_dim-96 /
        # 128 launches without a window)
        same_kernel = binding.debug_prefill_plan_ex(
            1, Hq, lq, lk, d, causal, 152, window=window).keys_per_block == 128
        if same_kernel and (causal or window > 0 or lk < 2048):
            o2, l2 = binding.prefill(qb, kb, vb, scale=scale, causal=causal, window=window,
                                     sinks=sinks)
            torch.cuda.synchronize()
            assert torch.equal(o_b, o2) and torch.equal(l_b, l2), f"seq {b} differs from dense"
    free_cuda()


def test_prefill_varlen_many_short_sequences():
    """64 sequences of 1..200 tokens: most query blocks of the grid lie past
    their sequence's end and must do nothing."""
    from attention_forward_blackwell_gb300 import binding, inputs
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(1, 201, size=64)]
    Hq, Hkv, d = 2, 1, 128
    q, k, v, cq, ck = packed(lens, lens, Hq, Hkv, d, seed=9)
    o, lse = binding.prefill_varlen(q, k, v, cq, ck, max(lens), max(lens), causal=True)
    torch.cuda.synchronize()
    check_device_error()
    qs = np.concatenate([[0], np.cumsum(lens)])
    scale = 1.0 / math.sqrt(d)
    for b in range(0, 64, 7):
        qb, kb, vb = (seq(t, qs[b], qs[b + 1]) for t in (q, k, v))
        ro, rl = oracle.attention_fwd(inputs.bf16_bits(qb), inputs.bf16_bits(kb),
                                      inputs.bf16_bits(vb), scale=scale, causal=True,
                                      threads=THREADS)
        compare(seq(o, qs[b], qs[b + 1]), lse[:, qs[b]:qs[b + 1]].unsqueeze(0), ro, rl,
                f"short seq {b}")


def test_prefill_varlen_offsets_clamped_and_args():
    """Offsets past the tensors are clamped on the device (no write outside
    o / lse); bad host arguments are rejected before any launch."""
    from attention_forward_blackwell_gb300 import binding
    Hq, d = 2, 64
    q, k, v, _, _ = packed([100, 100], [100, 100], Hq, Hq, d, seed=3)
    o_big = torch.full((200 + 64, Hq, d), float("nan"), device="cuda", dtype=torch.bfloat16)
    lse_big = torch.full((Hq * 200 + 64,), float("nan"), device="cuda")
    bad = torch.tensor([0, 150, 900], dtype=torch.int32, device="cuda")   # past total
    binding.prefill_varlen(q, k, v, bad, bad, 256, 256, out=o_big[:200],
                           lse=lse_big[:Hq * 200].view(Hq, 200))
    torch.cuda.synchronize()
    check_device_error()
    assert torch.isnan(o_big[200:].float()).all() and torch.isnan(lse_big[Hq * 200:]).all()
    good = torch.tensor([0, 100, 200], dtype=torch.int32, device="cuda")
    with pytest.raises(binding.FaError):   # max_seqlen_q = 0 with tokens present
        binding.prefill_varlen(q, k, v, good, good, 0, 100)


PAGED_CASES = [
    # Hq, Hkv, d, page_size, lens_q, lens_k, causal
    (4, 2, 128, 128, [100, 257, 1], [600, 257, 900], True),   # chunks of new tokens
    (2, 2, 64, 256, [300, 50], [300, 1000], False),
    (4, 1, 256, 128, [129, 64], [400, 64], True),
]


@pytest.mark.parametrize("Hq,Hkv,d,P,lens_q,lens_k,causal", PAGED_CASES,
                         ids=[f"h{c[0]}x{c[1]}d{c[2]}p{c[3]}{'c' if c[6] else 'n'}"
                              for c in PAGED_CASES])
def test_prefill_varlen_paged(Hq, Hkv, d, P, lens_q, lens_k, causal):
    """Packed queries over shuffled, NaN-poisoned pages: each sequence against
    the oracle, and bit for bit against the packed-key path on the same keys."""
    from attention_forward_blackwell_gb300 import binding, inputs
    from gpu_parity import to_pages
    q, k, v, cq, ck = packed(lens_q, lens_k, Hq, Hkv, d, seed=7 * P + d)
    B, Sk = len(lens_k), max(lens_k)
    ks = np.concatenate([[0], np.cumsum(lens_k)])
    kd = torch.zeros(B, Hkv, Sk, d, device="cuda", dtype=torch.bfloat16)
    vd = torch.zeros_like(kd)
    for b in range(B):
        kd[b, :, :lens_k[b]] = k[ks[b]:ks[b + 1]].permute(1, 0, 2)
        vd[b, :, :lens_k[b]] = v[ks[b]:ks[b + 1]].permute(1, 0, 2)
    kc, vc, table, _ = to_pages(kd, vd, lens_k, P, seed=P + d)
    lens_t = torch.tensor(lens_k, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = binding.prefill_varlen_paged(q, kc, vc, cq, max(lens_q), table, lens_t, scale=scale,
                                          causal=causal)
    torch.cuda.synchronize()
    check_device_error()
    o2, l2 = binding.prefill_varlen(q, k, v, cq, ck, max(lens_q), max(lens_k), scale=scale,
                                    causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, l2)
    qs = np.concatenate([[0], np.cumsum(lens_q)])
    for b in range(B):
        qb, kb, vb = seq(q, qs[b], qs[b + 1]), seq(k, ks[b], ks[b + 1]), seq(v, ks[b], ks[b + 1])
        ro, rl = oracle.attention_fwd(inputs.bf16_bits(qb), inputs.bf16_bits(kb),
                                      inputs.bf16_bits(vb), scale=scale, causal=causal,
                                      threads=THREADS)
        compare(seq(o, qs[b], qs[b + 1]), lse[:, qs[b]:qs[b + 1]].unsqueeze(0), ro, rl,
                f"varlen paged seq {b}")
    free_cuda()
