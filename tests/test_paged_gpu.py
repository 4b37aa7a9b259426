"""Paged K/V caches (prefill and decode) against the fp64 oracle on the same
keys laid out contiguously, and against the contiguous kernels."""
import math

import numpy as np
import pytest
import torch

from gpu_parity import check_device_error, compare, free_cuda, oracle_for, to_pages

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from attention_forward_blackwell_gb300 import build
    build.build()
    yield
    free_cuda()


def _wide(B, Hq, Sq, Sk, d, causal):
    """A contiguous launch of this shape runs the 256-key kernel."""
    from attention_forward_blackwell_gb300 import binding
    return binding.debug_prefill_plan_ex(B, Hq, Sq, Sk, d, causal, 152).keys_per_block == 256


PREFILL = [
    # B, Hq, Hkv, Sq, Sk, d, page_size, causal, lengths
    (3, 4, 2, 300, 1024, 128, 128, False, [1024, 700, 129]),
    (3, 4, 2, 300, 1024, 128, 256, True, [1024, 700, 300]),
    (2, 2, 1, 257, 768, 64, 256, True, [768, 500]),
    (2, 4, 2, 200, 640, 256, 128, False, [640, 333]),
    (2, 2, 2, 300, 1152, 96, 384, True, [1152, 1000]),
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,d,P,causal,lengths", PREFILL,
                         ids=[f"b{c[0]}q{c[3]}k{c[4]}d{c[5]}p{c[6]}{'c' if c[7] else 'n'}"
                              for c in PREFILL])
def test_prefill_paged(B, Hq, Hkv, Sq, Sk, d, P, causal, lengths):
    from attention_forward_blackwell_gb300 import binding, inputs
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=800 + Sk + P, device="cuda",
                           lengths=lengths)
    kc, vc, table, _ = to_pages(x.k, x.v, lengths, P, seed=P + Sq)
    scale = 1.0 / math.sqrt(d)
    o, lse = binding.prefill_paged(x.q, kc, vc, table, x.seqlens_k, scale=scale, causal=causal)
    torch.cuda.synchronize()
    check_device_error()
    ro, rl = oracle_for(x, scale, causal)
    compare(o, lse, ro, rl, f"prefill paged P={P}")
    # contiguous K/V of the same (page-rounded) length: the same kernel gives
    # the same result bit for bit (the 256-key kernel, which takes the
    # contiguous non-causal head_dim-96/128 launches, is checked on its own)
    if Sk % P == 0 and not _wide(B, Hq, Sq, Sk, d, causal):
        o2, l2 = binding.prefill(x.q, x.k, x.v, scale=scale, causal=causal,
                                 seqlens_k=x.seqlens_k)
        torch.cuda.synchronize()
        assert torch.equal(o, o2) and torch.equal(lse, l2)
    free_cuda()


SPLIT_PAGED = [
    # B, Hq, Hkv, Sq, Sk, d, page_size, lengths: non-causal shapes with at
    # least 16 key blocks whose units do not fill a wave, so the plan cuts
    # them into pieces along the key axis (page lookups inside every piece)
    (2, 2, 1, 1024, 2560, 128, 256, [2560, 2300]),
    (2, 2, 1, 1024, 2560, 96, 256, [2560, 1800]),
    (1, 4, 2, 512, 2048, 256, 128, [2048]),
    (2, 2, 2, 1024, 3072, 64, 512, [3000, 2049]),
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,d,P,lengths", SPLIT_PAGED,
                         ids=[f"b{c[0]}q{c[3]}k{c[4]}d{c[5]}p{c[6]}" for c in SPLIT_PAGED])
def test_prefill_paged_split_units(B, Hq, Hkv, Sq, Sk, d, P, lengths):
    """Paged caches with the last wave split into pieces and merged on the
    device: every row against the oracle, and bit-equal to the same plan on
    contiguous K/V where the contiguous launch runs the same kernel (else
    that one against the oracle too)."""
    from attention_forward_blackwell_gb300 import binding, inputs
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert binding.debug_prefill_plan_ex(B, Hq, Sq, Sk, d, False, n_sms, paged=True).split > 1
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=850 + d, device="cuda", lengths=lengths)
    kc, vc, table, _ = to_pages(x.k, x.v, lengths, P, seed=P + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = binding.prefill_paged(x.q, kc, vc, table, x.seqlens_k, scale=scale)
    torch.cuda.synchronize()
    check_device_error()
    ro, rl = oracle_for(x, scale, False)
    compare(o, lse, ro, rl, f"prefill paged split P={P} d={d}")
    inputs.poison_beyond_lengths(x.k, x.seqlens_k)
    inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    o2, l2 = binding.prefill(x.q, x.k, x.v, scale=scale, seqlens_k=x.seqlens_k)
    torch.cuda.synchronize()
    check_device_error()
    if _wide(B, Hq, Sq, Sk, d, False):
        compare(o2, l2, ro, rl, f"prefill contiguous (256-key kernel) d={d}")
    else:
        assert torch.equal(o, o2) and torch.equal(lse, l2)
    free_cuda()


DECODE = [
    # B, Hq, Hkv, Sq, Sk, d, page_size
    (8, 8, 2, 1, 4096, 128, 16),
    (8, 8, 2, 1, 4096, 128, 64),
    (8, 8, 2, 1, 4096, 128, 128),
    (4, 16, 4, 4, 3000, 64, 1000),
    (4, 4, 1, 1, 2048, 256, 256),
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,d,P", DECODE,
                         ids=[f"b{c[0]}h{c[1]}q{c[3]}k{c[4]}d{c[5]}p{c[6]}" for c in DECODE])
def test_decode_paged(B, Hq, Hkv, Sq, Sk, d, P):
    from attention_forward_blackwell_gb300 import binding, inputs
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=900 + P, device="cuda", lengths=(1, Sk))
    lens = x.seqlens_k.cpu().tolist()
    kc, vc, table, _ = to_pages(x.k, x.v, lens, P, seed=P)
    scale = 1.0 / math.sqrt(d)
    causal = Sq > 1
    o, lse = binding.decode_paged(x.q, kc, vc, table, x.seqlens_k, scale=scale, causal=causal)
    torch.cuda.synchronize()
    check_device_error()
    ro, rl = oracle_for(x, scale, causal)
    compare(o, lse, ro, rl, f"decode paged P={P}")
    if Sk % P == 0:   # same split plan as the contiguous call: same result bit for bit
        o2, l2 = binding.decode(x.q, x.k, x.v, scale=scale, causal=causal,
                                seqlens_k=x.seqlens_k)
        torch.cuda.synchronize()
        assert torch.equal(o, o2) and torch.equal(lse, l2)


def test_paged_argument_checks():
    from attention_forward_blackwell_gb300 import binding
    q = torch.zeros(1, 1, 4, 64, device="cuda", dtype=torch.bfloat16)
    kc = torch.zeros(2, 1, 64, 64, device="cuda", dtype=torch.bfloat16)
    table = torch.zeros(1, 2, dtype=torch.int32, device="cuda")
    lens = torch.full((1,), 100, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.FaError):   # prefill tiles need pages of 128 keys
        binding.prefill_paged(q, kc, kc, table, lens)
    o, lse = binding.decode_paged(q, kc, kc, table, lens)   # decode takes any page size
    torch.cuda.synchronize()
    assert torch.isfinite(o).all()
