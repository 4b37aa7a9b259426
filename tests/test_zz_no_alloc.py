"""fa_fwd_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (its split partials live in a fixed array inside the
library).  Its results must match fa_fwd_decode, call after call.

This file is collected last on purpose: a run that stops at the first failure
has run every other test before reaching it.
"""
import ctypes
import math

import pytest
import torch

pytestmark = pytest.mark.gpu

TOL_O = 2e-2
TOL_LSE = 1e-3


def _call_noalloc(lib, x, out, lse, scale):
    B, Hq, Sq, d = x.q.shape
    _, Hkv, Sk, _ = x.k.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.fa_fwd_decode_noalloc(p(x.q), p(x.k), p(x.v), p(out), p(lse), B, Hq, Hkv, Sq, Sk,
                                     p(x.seqlens_k), d, scale, 0, stream)


def _max_err(a, b):
    same = torch.isinf(a) & torch.isinf(b) & (torch.sign(a) == torch.sign(b))
    d = torch.where(same, torch.zeros_like(a), (a - b).abs())
    assert not torch.isnan(d).any()
    return d.max().item()


def test_noalloc_decode_matches_allocating_decode_on_consecutive_calls():
    from attention_forward_blackwell_gb300 import binding, build, inputs
    build.build()
    lib = binding.lib()
    cases = [  # two calls in a row with different inputs and shapes
        dict(B=4, Hq=16, Hkv=2, Sk=3000, d=128, lengths=[3000, 17, 2048, 0], tag=900),
        dict(B=3, Hq=8, Hkv=8, Sk=1500, d=64, lengths=[1, 1500, 777], tag=901),
    ]
    for c in cases:
        x = inputs.make_inputs(c["B"], c["Hq"], c["Hkv"], 1, c["Sk"], c["d"], tag=c["tag"],
                               device="cuda", lengths=c["lengths"])
        inputs.poison_beyond_lengths(x.k, x.seqlens_k)
        inputs.poison_beyond_lengths(x.v, x.seqlens_k)
        scale = 1.0 / math.sqrt(c["d"])
        ref_o, ref_l = binding.decode(x.q, x.k, x.v, scale=scale, seqlens_k=x.seqlens_k)
        out = torch.full_like(x.q, float("nan"))
        lse = torch.full_like(ref_l, float("nan"))
        assert _call_noalloc(lib, x, out, lse, scale) == binding.FA_OK
        torch.cuda.synchronize()
        assert binding.get_device_error() == binding.FA_OK
        eo = _max_err(out.float(), ref_o.float())
        el = _max_err(lse, ref_l)
        print(f"noalloc vs decode {c}: max|dO|={eo:.3e} max|dLSE|={el:.3e}")
        assert eo <= TOL_O and el <= TOL_LSE


def test_noalloc_decode_rejects_sizes_beyond_its_scratch():
    from attention_forward_blackwell_gb300 import binding, inputs
    lib = binding.lib()
    # batch * hq * (d + 1) * 4 bytes > 16 MiB: one split's partials do not fit
    x = inputs.make_inputs(300, 128, 8, 1, 64, 128, tag=902, device="cuda")
    out = torch.empty_like(x.q)
    lse = torch.empty(300, 128, 1, device="cuda")
    assert _call_noalloc(lib, x, out, lse, 0.1) == binding.FA_ERR_INVALID_ARG
