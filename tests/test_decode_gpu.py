"""Split-KV decode (split kernel + LSE combine) against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

from gpu_parity import check_device_error, compare, free_cuda, oracle_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from attention_forward_blackwell_gb300 import build
    build.build()
    yield
    free_cuda()


def _decode(x, scale, causal=False, splits=0):
    from attention_forward_blackwell_gb300 import binding
    o, lse = binding.decode(x.q, x.k, x.v, scale=scale, causal=causal, seqlens_k=x.seqlens_k,
                            num_splits=splits)
    torch.cuda.synchronize()
    check_device_error()
    return o, lse


@pytest.mark.parametrize("splits", [1, 2, 7, 0, 1000])
def test_split_counts_agree_with_oracle(splits):
    """Any split count gives the oracle's result (merge over disjoint key sets)."""
    from attention_forward_blackwell_gb300 import inputs
    x = inputs.make_inputs(3, 8, 2, 1, 700, 128, tag=500, device="cuda", lengths=[700, 1, 333])
    inputs.poison_beyond_lengths(x.k, x.seqlens_k)
    inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    o, lse = _decode(x, 128 ** -0.5, splits=splits)
    ro, rl = oracle_for(x, 128 ** -0.5, False)
    compare(o, lse, ro, rl, f"decode splits={splits}")


DECODE_SHAPES = [
    # B, Hq, Hkv, Sq, Sk, d, causal, lengths
    (2, 4, 4, 1, 513, 64, False, [513, 64]),
    (2, 16, 1, 1, 900, 128, False, None),          # MQA, 16 heads on one tile
    (1, 32, 2, 1, 400, 128, False, None),          # 16 heads per kv head
    (2, 8, 2, 4, 600, 128, True, [600, 5]),        # 4 queries per sequence, causal
    (1, 64, 2, 2, 300, 128, True, None),           # 64 rows per kv head -> 4 M tiles
    (2, 8, 1, 1, 777, 256, False, [777, 300]),
    (1, 4, 2, 16, 40, 64, True, None),             # more queries than keys for some rows
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,d,causal,lengths", DECODE_SHAPES)
def test_decode_shapes(B, Hq, Hkv, Sq, Sk, d, causal, lengths):
    from attention_forward_blackwell_gb300 import inputs
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=600 + Sk, device="cuda", lengths=lengths)
    if lengths is not None:
        inputs.poison_beyond_lengths(x.k, x.seqlens_k)
        inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    o, lse = _decode(x, 1 / math.sqrt(d), causal)
    ro, rl = oracle_for(x, 1 / math.sqrt(d), causal)
    compare(o, lse, ro, rl, f"decode {B,Hq,Hkv,Sq,Sk,d,causal}")


def test_decode_matches_prefill_at_one_query():
    from attention_forward_blackwell_gb300 import binding, inputs
    x = inputs.make_inputs(2, 8, 2, 1, 1000, 128, tag=700, device="cuda")
    od, ld = _decode(x, 0.088)
    op, lp = binding.prefill(x.q, x.k, x.v, scale=0.088)
    torch.cuda.synchronize()
    assert (od.float() - op.float()).abs().max().item() <= 2e-2
    assert (ld - lp).abs().max().item() <= 1e-3


def test_empty_sequences():
    from attention_forward_blackwell_gb300 import inputs
    x = inputs.make_inputs(3, 4, 2, 1, 256, 128, tag=701, device="cuda", lengths=[0, 256, 0])
    o, lse = _decode(x, 0.1)
    assert torch.all(o[0] == 0) and torch.all(o[2] == 0)
    assert torch.all(torch.isneginf(lse[0])) and torch.all(torch.isneginf(lse[2]))
    ro, rl = oracle_for(x, 0.1, False)
    compare(o, lse, ro, rl, "decode empty sequences")


def test_full_decode_configuration_all_rows():
    """The full decode workload (B=64, Hq=64, Hkv=8, d=128, L_b~U[1024,16384],
    KV padded to 16384 with NaN past each length): every output row against
    the oracle."""
    from attention_forward_blackwell_gb300 import inputs, workloads
    w = workloads.DECODE
    x = inputs.make_inputs(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, tag=w.tag, device="cuda",
                           lengths=w.lengths)
    inputs.poison_beyond_lengths(x.k, x.seqlens_k)
    inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    o, lse = _decode(x, w.scale)
    ro, rl = oracle_for(x, w.scale, False)
    compare(o, lse, ro, rl, "decode full config")
    del x
    free_cuda()


def test_decode_many_sequences_max_queries_sampled():
    """256 sequences, 16 queries each (the decode maximum), GQA 4, lengths
    U[1, 2000] with poisoned padding: sampled rows against the oracle."""
    from attention_forward_blackwell_gb300 import inputs
    B, Hq, Hkv, Sq, Sk, d = 256, 16, 4, 16, 2000, 128
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=640, device="cuda", lengths=(1, Sk))
    inputs.poison_beyond_lengths(x.k, x.seqlens_k)
    inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    o, lse = _decode(x, 1 / math.sqrt(d), True)
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([np.arange(64), rng.integers(0, B * Hq * Sq, 400),
                                     np.arange(B * Hq * Sq - 64, B * Hq * Sq)]))
    ro, rl = oracle_for(x, 1 / math.sqrt(d), True, rows=rows)
    idx = torch.from_numpy(rows).cuda()
    compare(o.view(-1, d)[idx], lse.view(-1)[idx], ro, rl, "decode B=256 Sq=16 (sampled)")
    free_cuda()


@pytest.mark.parametrize("B,Hq,Sq,lengths,causal", [
    (2, 8, 1, [1 << 20, 300001], False),   # 1,048,576 keys: ~1,700 splits merged
    (1, 2, 16, [1 << 20], True),           # the most queries decode takes, causal
])
def test_decode_million_keys(B, Hq, Sq, lengths, causal):
    """A key range of 2^20 (padding past shorter lengths poisoned with NaN):
    every output row against the oracle."""
    from attention_forward_blackwell_gb300 import binding, inputs
    d, Sk = 128, 1 << 20
    x = inputs.make_inputs(B, Hq, 1, Sq, Sk, d, tag=1400 + Sq, device="cuda", lengths=lengths)
    inputs.poison_beyond_lengths(x.k, x.seqlens_k)
    inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    scale = 1.0 / math.sqrt(d)
    o, lse = binding.decode(x.q, x.k, x.v, scale=scale, causal=causal, seqlens_k=x.seqlens_k)
    torch.cuda.synchronize()
    check_device_error()
    ro, rl = oracle_for(x, scale, causal)
    compare(o, lse, ro, rl, f"decode 2^20 keys B={B} Sq={Sq}")
    del x, o, lse
    free_cuda()
