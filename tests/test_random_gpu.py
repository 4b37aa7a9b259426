"""Seeded random shapes through every entry point, element by element against
the fp64 oracle.

The hand-picked cases of the other files pin the edges one at a time; these
draw them in combination: head_dim 64 / 96 / 128 / 256 / 512 (each prefill
kernel family: two-tile, 256-key, persistent head_dim 256, head_dim 512),
GQA ratios 1-8, query and key lengths ragged against every tile size,
per-sequence key lengths with empty sequences and NaN padding, the causal
mask, sliding windows and attention sinks (the readings of "2026-05-28_STATUS.md"
D3, D4, D5c), paged caches, packed sequences, and decode with 1-16 query
rows, explicit split counts and arbitrary page sizes.  The draws are fixed
by the seeds, so a failure names its case.
"""
import math
import random

import numpy as np
import pytest
import torch

import oracle
from gpu_parity import THREADS, check_device_error, compare, free_cuda, to_pages

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from attention_forward_blackwell_gb300 import build
    build.build()
    yield
    free_cuda()


def _oracle(x, scale, causal, window=0, sinks=None, lens=None):
    from attention_forward_blackwell_gb300 import inputs
    if lens is None and x.seqlens_k is not None:
        lens = x.seqlens_k.cpu().tolist()
    sk = None if sinks is None else sinks.cpu().double().numpy()
    return oracle.attention_fwd(inputs.bf16_bits(x.q), inputs.bf16_bits(x.k),
                                inputs.bf16_bits(x.v), scale=scale, causal=causal,
                                seqlens_k=lens, threads=THREADS, window=window, sinks=sk)


def _sinks(hq, seed):
    g = torch.Generator().manual_seed(seed)
    return (2.0 * torch.randn(hq, generator=g)).float().cuda()


def _lengths(rng, B, sk):
    """None, or B key lengths in [0, sk] with the ends and zero likely."""
    if rng.random() < 0.5:
        return None
    return [rng.choice([0, sk, rng.randint(1, sk), rng.randint(1, sk)]) for _ in range(B)]


# --------------------------------------------------------------- prefill ----

def _prefill_cases(n, seed):
    rng = random.Random(seed)
    out = []
    for _ in range(n):
        d = rng.choice([64, 96, 128, 256, 512])
        hkv = rng.choice([1, 2])
        hq = hkv * rng.choice([1, 2, 4])
        B = rng.choice([1, 2])
        smax = 700 if d == 512 else 1500
        sq, sk = rng.randint(1, smax), rng.randint(1, smax)
        causal = rng.random() < 0.5
        window = rng.randint(1, sk) if rng.random() < 0.35 else 0
        sinks = rng.random() < 0.3
        out.append((B, hq, hkv, sq, sk, d, causal, window, sinks, _lengths(rng, B, sk)))
    return out


PREFILL = _prefill_cases(30, seed=31)


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,d,causal,window,sinks_on,lengths", PREFILL,
                         ids=[f"p{i}" for i in range(len(PREFILL))])
def test_random_prefill(B, Hq, Hkv, Sq, Sk, d, causal, window, sinks_on, lengths):
    from attention_forward_blackwell_gb300 import binding, inputs
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=3000 + Sq + Sk + d, device="cuda",
                           lengths=lengths)
    if lengths is not None:
        inputs.poison_beyond_lengths(x.k, x.seqlens_k)
        inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    sinks = _sinks(Hq, Sq + Sk) if sinks_on else None
    scale = 1.0 / math.sqrt(d)
    o, lse = binding.prefill(x.q, x.k, x.v, scale=scale, causal=causal, seqlens_k=x.seqlens_k,
                             window=window, sinks=sinks)
    torch.cuda.synchronize()
    check_device_error()
    ro, rl = _oracle(x, scale, causal, window, sinks)
    compare(o, lse, ro, rl, f"prefill {B, Hq, Hkv, Sq, Sk, d} causal={causal} "
                            f"window={window} sinks={sinks_on} lengths={lengths}")
    free_cuda()


# --------------------------------------------------------- paged prefill ----

def _paged_cases(n, seed):
    rng = random.Random(seed)
    out = []
    for _ in range(n):
        d = rng.choice([64, 96, 128, 256, 512])
        hkv = rng.choice([1, 2])
        hq = hkv * rng.choice([1, 2, 4])
        B = rng.choice([1, 2, 3])
        smax = 600 if d == 512 else 1300
        sq, sk = rng.randint(1, smax), rng.randint(1, smax)
        lens = [rng.choice([0, sk, rng.randint(1, sk)]) for _ in range(B)]
        out.append((B, hq, hkv, sq, sk, d, rng.choice([128, 256]), rng.random() < 0.5, lens))
    return out


PAGED = _paged_cases(14, seed=47)


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,d,P,causal,lengths", PAGED,
                         ids=[f"g{i}" for i in range(len(PAGED))])
def test_random_paged_prefill(B, Hq, Hkv, Sq, Sk, d, P, causal, lengths):
    from attention_forward_blackwell_gb300 import binding, inputs
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=3300 + Sq + d, device="cuda",
                           lengths=lengths)
    kc, vc, table, _ = to_pages(x.k, x.v, lengths, P, seed=Sk + P)
    scale = 1.0 / math.sqrt(d)
    o, lse = binding.prefill_paged(x.q, kc, vc, table, x.seqlens_k, scale=scale, causal=causal)
    torch.cuda.synchronize()
    check_device_error()
    ro, rl = _oracle(x, scale, causal)
    compare(o, lse, ro, rl, f"paged prefill {B, Hq, Hkv, Sq, Sk, d} P={P} causal={causal} "
                            f"lengths={lengths}")
    free_cuda()


# ------------------------------------------------------ packed sequences ----

def _varlen_cases(n, seed):
    rng = random.Random(seed)
    out = []
    for _ in range(n):
        d = rng.choice([64, 96, 128, 256])
        hkv = rng.choice([1, 2])
        hq = hkv * rng.choice([1, 2, 4])
        B = rng.randint(1, 5)
        lq = [rng.choice([0, rng.randint(1, 700), rng.randint(1, 130)]) for _ in range(B)]
        same = rng.random() < 0.5
        lk = list(lq) if same else [rng.choice([0, rng.randint(1, 900)]) for _ in range(B)]
        if sum(lq) == 0:
            lq[0] = 1
        causal = rng.random() < 0.5
        window = rng.randint(1, 400) if rng.random() < 0.3 else 0
        out.append((hq, hkv, d, lq, lk, causal, window, rng.random() < 0.3))
    return out


VARLEN = _varlen_cases(14, seed=59)


@pytest.mark.parametrize("Hq,Hkv,d,lens_q,lens_k,causal,window,sinks_on", VARLEN,
                         ids=[f"v{i}" for i in range(len(VARLEN))])
def test_random_varlen(Hq, Hkv, d, lens_q, lens_k, causal, window, sinks_on):
    from attention_forward_blackwell_gb300 import binding, inputs
    seed = sum(lens_q) + sum(lens_k) + d
    q = inputs.randn_bf16((sum(lens_q), Hq, d), 5000 + seed, "cuda")
    tk = max(1, sum(lens_k))
    k = inputs.randn_bf16((tk, Hkv, d), 6000 + seed, "cuda")
    v = inputs.randn_bf16((tk, Hkv, d), 7000 + seed, "cuda")
    qs = np.concatenate([[0], np.cumsum(lens_q)])
    ks = np.concatenate([[0], np.cumsum(lens_k)])
    cq = torch.tensor(qs, dtype=torch.int32, device="cuda")
    ck = torch.tensor(ks, dtype=torch.int32, device="cuda")
    sinks = _sinks(Hq, seed) if sinks_on else None
    scale = 1.0 / math.sqrt(d)
    o, lse = binding.prefill_varlen(q, k, v, cq, ck, max(lens_q), max(1, max(lens_k)),
                                    scale=scale, causal=causal, window=window, sinks=sinks)
    torch.cuda.synchronize()
    check_device_error()
    sk_np = None if sinks is None else sinks.cpu().double().numpy()

    def seq(t, a, b):
        return t[a:b].permute(1, 0, 2).unsqueeze(0).contiguous()

    for b, (lq, lk) in enumerate(zip(lens_q, lens_k)):
        if lq == 0:
            continue
        o_b = seq(o, qs[b], qs[b + 1])
        l_b = lse[:, qs[b]:qs[b + 1]].unsqueeze(0)
        if lk == 0:
            assert torch.all(o_b == 0)
            want = (torch.full((1, Hq, lq), float("-inf"), device="cuda") if sinks is None
                    else sinks.view(1, Hq, 1).expand(1, Hq, lq))
            assert torch.allclose(l_b, want, rtol=1e-6, atol=1e-6)
            continue
        ro, rl = oracle.attention_fwd(inputs.bf16_bits(seq(q, qs[b], qs[b + 1])),
                                      inputs.bf16_bits(seq(k, ks[b], ks[b + 1])),
                                      inputs.bf16_bits(seq(v, ks[b], ks[b + 1])), scale=scale,
                                      causal=causal, threads=THREADS, window=window, sinks=sk_np)
        compare(o_b, l_b, ro, rl, f"varlen {Hq, Hkv, d} seq {b} (lq={lq}, lk={lk}) "
                                  f"causal={causal} window={window} sinks={sinks_on}")
    free_cuda()


# ---------------------------------------------------------------- decode ----

def _decode_cases(n, seed):
    rng = random.Random(seed)
    out = []
    for _ in range(n):
        d = rng.choice([64, 128, 256])
        hkv = rng.choice([1, 2, 4])
        hq = hkv * rng.choice([1, 2, 4, 8])
        B = rng.randint(1, 8)
        sq = rng.choice([1, 1, 2, 4, rng.randint(1, 16)])
        sk = rng.randint(1, 5000)
        lens = [rng.choice([0, sk, rng.randint(1, sk), rng.randint(1, sk)]) for _ in range(B)]
        mode = rng.choice(["auto", "splits", "window", "paged"])
        extra = {"auto": 0, "splits": rng.randint(1, 24), "window": rng.randint(1, sk),
                 "paged": rng.choice([16, 37, 64, 128, 200])}[mode]
        out.append((B, hq, hkv, sq, sk, d, rng.random() < 0.5, lens, mode, extra))
    return out


DECODE = _decode_cases(28, seed=71)


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,d,causal,lengths,mode,extra", DECODE,
                         ids=[f"d{i}" for i in range(len(DECODE))])
def test_random_decode(B, Hq, Hkv, Sq, Sk, d, causal, lengths, mode, extra):
    from attention_forward_blackwell_gb300 import binding, inputs
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=3600 + Sk + d, device="cuda",
                           lengths=lengths)
    inputs.poison_beyond_lengths(x.k, x.seqlens_k)
    inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    scale = 1.0 / math.sqrt(d)
    window, sinks = 0, None
    if mode == "paged":
        kc, vc, table, _ = to_pages(x.k, x.v, lengths, extra, seed=Sk + extra)
        o, lse = binding.decode_paged(x.q, kc, vc, table, x.seqlens_k, scale=scale,
                                      causal=causal)
    elif mode == "window":
        window, sinks = extra, _sinks(Hq, Sk)
        o, lse = binding.decode(x.q, x.k, x.v, scale=scale, causal=causal,
                                seqlens_k=x.seqlens_k, window=window, sinks=sinks)
    else:
        o, lse = binding.decode(x.q, x.k, x.v, scale=scale, causal=causal,
                                seqlens_k=x.seqlens_k, num_splits=extra)
    torch.cuda.synchronize()
    check_device_error()
    ro, rl = _oracle(x, scale, causal, window, sinks)
    compare(o, lse, ro, rl, f"decode {B, Hq, Hkv, Sq, Sk, d} causal={causal} {mode}={extra} "
                            f"lengths={lengths}")
    free_cuda()
