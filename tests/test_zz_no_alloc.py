"""fa_fwd_decode_noalloc: the decode entry point for callers that cannot
allocate device memory while they run (its split partials live in a fixed
array inside the library instead of a per-call workspace).  Its results must
match the fp64 oracle and fa_fwd_decode, call after call.

This file is collected last on purpose: a run that stops at the first failure
has run every other test before reaching it.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from gpu_parity import compare, oracle_for

pytestmark = pytest.mark.gpu

TOL_O = 2e-2
TOL_LSE = 1e-3
SCRATCH_FLOATS = (16 << 20) // 4     # FA_DECODE_NOALLOC_SCRATCH_BYTES / sizeof(float)


def _call_noalloc(lib, x, out, lse, scale, causal=False):
    B, Hq, Sq, d = x.q.shape
    _, Hkv, Sk, _ = x.k.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.fa_fwd_decode_noalloc(p(x.q), p(x.k), p(x.v), p(out), p(lse), B, Hq, Hkv, Sq, Sk,
                                     p(x.seqlens_k), d, scale, int(causal), stream)


def _max_err(a, b):
    same = torch.isinf(a) & torch.isinf(b) & (torch.sign(a) == torch.sign(b))
    d = torch.where(same, torch.zeros_like(a), (a - b).abs())
    assert not torch.isnan(d).any()
    return d.max().item()


def _noalloc(lib, x, scale, causal=False):
    from attention_forward_blackwell_gb300 import binding
    B, Hq, Sq, d = x.q.shape
    out = torch.full_like(x.q, float("nan"))
    lse = torch.full((B, Hq, Sq), float("nan"), device="cuda")
    assert _call_noalloc(lib, x, out, lse, scale, causal) == binding.FA_OK
    torch.cuda.synchronize()
    assert binding.get_device_error() == binding.FA_OK
    return out, lse


def test_noalloc_decode_matches_oracle_and_allocating_decode_on_consecutive_calls():
    from attention_forward_blackwell_gb300 import binding, build, inputs
    build.build()
    lib = binding.lib()
    cases = [  # calls in a row with different inputs and shapes
        dict(B=4, Hq=16, Hkv=2, Sq=1, Sk=3000, d=128, lengths=[3000, 17, 2048, 0], causal=0,
             tag=900),
        dict(B=3, Hq=8, Hkv=8, Sq=1, Sk=1500, d=64, lengths=[1, 1500, 777], causal=0, tag=901),
        dict(B=3, Hq=8, Hkv=2, Sq=4, Sk=2500, d=256, lengths=[2500, 4, 1111], causal=1, tag=903),
        dict(B=2, Hq=16, Hkv=4, Sq=4, Sk=4096, d=128, lengths=[4096, 3333], causal=1, tag=904),
    ]
    for c in cases:
        x = inputs.make_inputs(c["B"], c["Hq"], c["Hkv"], c["Sq"], c["Sk"], c["d"],
                               tag=c["tag"], device="cuda", lengths=c["lengths"])
        inputs.poison_beyond_lengths(x.k, x.seqlens_k)
        inputs.poison_beyond_lengths(x.v, x.seqlens_k)
        scale = 1.0 / math.sqrt(c["d"])
        causal = bool(c["causal"])
        ref_o, ref_l = binding.decode(x.q, x.k, x.v, scale=scale, causal=causal,
                                      seqlens_k=x.seqlens_k)
        out, lse = _noalloc(lib, x, scale, causal)
        ro, rl = oracle_for(x, scale, causal)
        compare(out, lse, ro, rl, f"noalloc vs oracle {c}")
        eo = _max_err(out.float(), ref_o.float())
        el = _max_err(lse, ref_l)
        print(f"noalloc vs decode {c}: max|dO|={eo:.3e} max|dLSE|={el:.3e}")
        assert eo <= TOL_O and el <= TOL_LSE


@pytest.mark.parametrize("Sq,causal", [(1, False), (4, True)])
def test_noalloc_decode_workload_where_the_scratch_limits_the_splits(Sq, causal):
    """The decode workload (B=64, Hq=64, Hkv=8, d=128, key lengths drawn from
    [1024, 16384]): one split's partials take 64*64*Sq*129 floats, so the
    16 MiB array holds 7 splits at Sq=1 (the allocating entry point would use
    more) and exactly one at Sq=4.  The call must use that many splits -- it
    equals fa_fwd_decode_splits with that count bit for bit -- and match the
    oracle on every row."""
    from attention_forward_blackwell_gb300 import binding, build, inputs, workloads
    build.build()
    lib = binding.lib()
    w = workloads.DECODE
    x = inputs.make_inputs(w.B, w.Hq, w.Hkv, Sq, w.Sk, w.d, tag=w.tag + Sq, device="cuda",
                           lengths=w.lengths)
    inputs.poison_beyond_lengths(x.k, x.seqlens_k)
    inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    per_split = w.B * w.Hq * Sq * (w.d + 1)
    fit = SCRATCH_FLOATS // per_split
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    pairs = w.B * w.Hkv * math.ceil(w.Hq // w.Hkv * Sq / 16)
    want = min(math.ceil(24 * n_sms / pairs), math.ceil(w.Sk / 256))
    assert fit == (7 if Sq == 1 else 1) and fit < want, (fit, want)
    out, lse = _noalloc(lib, x, w.scale, causal)
    same_o, same_l = binding.decode(x.q, x.k, x.v, scale=w.scale, causal=causal,
                                    seqlens_k=x.seqlens_k, num_splits=fit)
    torch.cuda.synchronize()
    assert torch.equal(out, same_o) and torch.equal(lse, same_l)
    auto_o, auto_l = binding.decode(x.q, x.k, x.v, scale=w.scale, causal=causal,
                                    seqlens_k=x.seqlens_k)
    torch.cuda.synchronize()
    assert _max_err(out.float(), auto_o.float()) <= TOL_O and _max_err(lse, auto_l) <= TOL_LSE
    ro, rl = oracle_for(x, w.scale, causal)
    compare(out, lse, ro, rl, f"noalloc decode workload Sq={Sq} ({fit} splits)")
    del x, out, lse, same_o, same_l, auto_o, auto_l
    torch.cuda.empty_cache()


def test_noalloc_decode_rejects_sizes_beyond_its_scratch():
    from attention_forward_blackwell_gb300 import binding, inputs
    lib = binding.lib()
    # batch * hq * (d + 1) * 4 bytes > 16 MiB: one split's partials do not fit
    x = inputs.make_inputs(300, 128, 8, 1, 64, 128, tag=902, device="cuda")
    out = torch.empty_like(x.q)
    lse = torch.empty(300, 128, 1, device="cuda")
    assert _call_noalloc(lib, x, out, lse, 0.1) == binding.FA_ERR_INVALID_ARG
    # the same oversized batch with no keys needs no partials: O = 0, LSE = -inf
    empty = inputs.make_inputs(300, 128, 8, 1, 0, 128, tag=902, device="cuda")
    out.fill_(1.0)
    lse.fill_(1.0)
    assert _call_noalloc(lib, empty, out, lse, 0.1) == binding.FA_OK
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
