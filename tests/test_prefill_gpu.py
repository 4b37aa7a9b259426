"""Prefill kernel (tcgen05/TMEM, warp-specialised) against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

from gpu_parity import (check_device_error, compare, free_cuda, oracle_for, sample_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from attention_forward_blackwell_gb300 import build
    build.build()
    yield
    free_cuda()


def _run(x, scale, causal):
    from attention_forward_blackwell_gb300 import binding
    o, lse = binding.prefill(x.q, x.k, x.v, scale=scale, causal=causal,
                             seqlens_k=x.seqlens_k)
    torch.cuda.synchronize()
    check_device_error()
    return o, lse


def _full_check(x, scale, causal, what):
    o, lse = _run(x, scale, causal)
    ro, rl = oracle_for(x, scale, causal)
    return compare(o, lse, ro, rl, what)


def test_tiny_config_exact_shape():
    from attention_forward_blackwell_gb300 import inputs, workloads
    w = workloads.TINY
    x = inputs.make_inputs(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, tag=w.tag, device="cuda")
    _full_check(x, w.scale, w.causal, w.name)


SMALL = [
    # B, Hq, Hkv, Sq, Sk, d, causal
    (1, 2, 1, 300, 300, 64, False),
    (1, 2, 1, 300, 300, 64, True),
    (1, 2, 2, 300, 300, 128, False),
    (1, 2, 2, 300, 300, 128, True),
    (1, 2, 2, 300, 300, 96, False),
    (1, 2, 2, 300, 300, 96, True),
    (1, 4, 2, 300, 300, 256, False),
    (1, 4, 2, 300, 300, 256, True),
    (2, 2, 2, 200, 333, 128, True),     # Sq < Sk: bottom-right causal
    (1, 2, 2, 333, 200, 128, True),     # Sq > Sk: leading rows see no key
    (1, 1, 1, 1, 500, 128, False),      # one query
    (1, 1, 1, 257, 1, 64, False),       # one key
    (2, 4, 1, 513, 700, 128, False),    # GQA 4, ragged both ways
    (1, 8, 2, 130, 1030, 256, True),    # GQA d=256 with a long key range
    (1, 3, 3, 640, 640, 64, True),      # several CTAs per head, causal
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,d,causal", SMALL,
                         ids=[f"b{c[0]}h{c[1]}x{c[2]}q{c[3]}k{c[4]}d{c[5]}{'c' if c[6] else 'n'}"
                              for c in SMALL])
def test_small_shapes(B, Hq, Hkv, Sq, Sk, d, causal):
    from attention_forward_blackwell_gb300 import inputs
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=100 + d + Sq, device="cuda")
    _full_check(x, 1.0 / math.sqrt(d), causal, f"small {B,Hq,Hkv,Sq,Sk,d,causal}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_key_lengths_with_poisoned_padding(d, causal):
    """Rows j >= L_b hold NaN: any read of them would poison O."""
    from attention_forward_blackwell_gb300 import inputs
    x = inputs.make_inputs(3, 2, 2, 256, 400, d, tag=300 + d, device="cuda",
                           lengths=[400, 150, 0])
    inputs.poison_beyond_lengths(x.k, x.seqlens_k)
    inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    o, lse = _run(x, 1.0 / math.sqrt(d), causal)
    ro, rl = oracle_for(x, 1.0 / math.sqrt(d), causal)
    compare(o, lse, ro, rl, f"lengths d={d} causal={causal}")
    assert torch.all(o[2] == 0) and torch.all(torch.isneginf(lse[2]))


def test_extreme_logits_one_hot_key():
    """K*8 gives scores with a spread of ~8.5 (max ~25 over 300 keys); key 17
    is set to score 60.1 for every query (q_0 = 4, k_17 = (170, 0, ..., 0)),
    so its weight is ~1 and every other weight is below e^-30."""
    from attention_forward_blackwell_gb300 import inputs
    d = 128
    x = inputs.make_inputs(1, 2, 2, 300, 300, d, tag=400, device="cuda", k_scale=8.0)
    x.q[..., 0] = 4.0
    x.k[..., 17, :] = 0.0
    x.k[..., 17, 0] = 60.0 * math.sqrt(d) / 4.0
    o, lse = _run(x, 1.0 / math.sqrt(d), False)
    ro, rl = oracle_for(x, 1.0 / math.sqrt(d), False)
    compare(o, lse, ro, rl, "extreme logits")
    assert float(lse.min()) > 55.0
    assert (o.float() - x.v[:, :, 17:18].float()).abs().max().item() < 2e-2


def test_zero_query_gives_mean_of_values():
    from attention_forward_blackwell_gb300 import inputs
    x = inputs.make_inputs(1, 2, 1, 260, 260, 64, tag=401, device="cuda")
    x.q.zero_()
    o, lse = _run(x, 0.125, True)
    # closed form: row i averages v_0..v_i, LSE = ln(i + 1)
    v = x.v[0, 0].float().cpu().numpy().astype(np.float64)
    ref = np.cumsum(v, axis=0) / np.arange(1, 261)[:, None]
    err = np.abs(o[0].float().cpu().numpy() - ref[None]).max()
    lerr = np.abs(lse[0].cpu().numpy() - np.log(np.arange(1, 261))[None]).max()
    assert err <= 2e-2 and lerr <= 1e-3, (err, lerr)
    # causal row 0 sees only key 0: O_0 = V_0 exactly (weight 1, bf16 round trip)
    assert torch.equal(o[0, :, 0], x.v[0, 0, 0].expand(2, -1))


def test_empty_key_range_writes_zero_and_neg_inf():
    from attention_forward_blackwell_gb300 import binding
    q = torch.randn(1, 2, 5, 64, device="cuda").bfloat16()
    k = torch.empty(1, 2, 0, 64, device="cuda", dtype=torch.bfloat16)
    o, lse = binding.prefill(q, k, k)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


FULL = ["PREFILL_D128", "PREFILL_D128_CAUSAL", "LONG_D128", "LONG_D96", "GQA_D256"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_row(name):
    """Full configuration in the benchmark's launch configuration: every
    output row against the oracle (threaded over the host cores)."""
    from attention_forward_blackwell_gb300 import inputs, workloads
    w = getattr(workloads, name)
    x = inputs.make_inputs(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, tag=w.tag, device="cuda",
                           k_scale=w.k_scale)
    o, lse = _run(x, w.scale, w.causal)
    ro, rl = oracle_for(x, w.scale, w.causal)
    compare(o, lse, ro, rl, f"full {w.name} (all {w.B * w.Hq * w.Sq} rows)")
    del x, o, lse, ro, rl
    free_cuda()


def test_repeated_calls_are_deterministic():
    from attention_forward_blackwell_gb300 import inputs
    x = inputs.make_inputs(1, 4, 2, 700, 700, 128, tag=402, device="cuda")
    o1, l1 = _run(x, 0.09, True)
    o2, l2 = _run(x, 0.09, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_wait_timeout_selftest_reports_and_recovers():
    """A wait that nothing completes gives up, records FA_ERR_TIMEOUT, and the
    context stays usable."""
    from attention_forward_blackwell_gb300 import binding, inputs
    assert binding.selftest_wait_timeout(2_000_000) == binding.FA_OK
    st, word = binding.get_device_error_word()
    assert st == binding.FA_ERR_TIMEOUT and word == 0x10FF
    assert binding.get_device_error() == binding.FA_OK     # cleared
    x = inputs.make_inputs(1, 1, 1, 128, 128, 64, tag=1, device="cuda")
    _full_check(x, 0.125, False, "after timeout")


@pytest.mark.parametrize("B,Hq,Sq,Sk,d,causal", [
    (1, 1, 128, 128, 64, False),    # one key tile per query tile
    (1, 1, 257, 1, 64, False),      # one key, a CTA whose second tile has no rows
    (1, 2, 300, 300, 128, True),    # causal 256-key kernel: units of 1 and 2 blocks
    (1, 4, 600, 200, 256, True),    # d = 256, rows that see no key
])
def test_barrier_protocol_stress(B, Hq, Sq, Sk, d, causal):
    """Many back-to-back launches of shapes whose pipelines are short (one or
    two key tiles), where a message that runs ahead of its reader would show
    up as a wait time-out: no launch may record one, and every result stays
    equal to the first."""
    from attention_forward_blackwell_gb300 import binding, inputs
    x = inputs.make_inputs(B, Hq, Hq, Sq, Sk, d, tag=450 + Sq, device="cuda")
    o0, l0 = _run(x, 1.0 / math.sqrt(d), causal)
    for _ in range(40):
        o, l = binding.prefill(x.q, x.k, x.v, scale=1.0 / math.sqrt(d), causal=causal)
    torch.cuda.synchronize()
    check_device_error()
    assert torch.equal(o, o0) and torch.equal(l, l0)


SPLIT = [
    # B, Hq, Hkv, Sq, Sk, d, lengths: non-causal shapes whose query blocks do
    # not fill whole waves of the GPU, so the last wave's blocks are computed
    # in pieces along the key axis and merged on the device (head_dim 96 and
    # 128 split only on paged caches: test_paged_gpu.py)
    (1, 1, 1, 16384, 16384, 64, None),      # 64 blocks -> 2 pieces each
    (1, 2, 2, 3000, 9000, 256, None),       # 48 blocks -> 3 pieces each
    (3, 1, 1, 2000, 30000, 64, [30000, 0, 17]),   # 24 blocks -> 6 pieces; empty pieces
    (2, 16, 4, 4096, 4096, 64, None),       # GQA: 56 tail blocks -> 2 pieces each
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,d,lengths", SPLIT,
                         ids=[f"b{c[0]}h{c[1]}x{c[2]}q{c[3]}k{c[4]}d{c[5]}" for c in SPLIT])
def test_split_units_sampled_rows(B, Hq, Hkv, Sq, Sk, d, lengths):
    """Query blocks computed in pieces by several CTAs and merged by the last
    piece to finish: sampled rows (tile edges of a few heads plus random rows)
    against the oracle, finiteness of every output row that sees a key."""
    from attention_forward_blackwell_gb300 import binding, inputs
    assert binding.debug_prefill_plan(B, Hq, Sq, Sk, d, False, 152)[2] > 1   # split
    x = inputs.make_inputs(B, Hq, Hkv, Sq, Sk, d, tag=500 + Sq % 97, device="cuda",
                           lengths=lengths)
    if lengths is not None:
        inputs.poison_beyond_lengths(x.k, x.seqlens_k)
        inputs.poison_beyond_lengths(x.v, x.seqlens_k)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(x, scale, False)
    lens = [Sk] * B if lengths is None else lengths
    for b in range(B):
        if lens[b] > 0:
            assert torch.isfinite(o[b]).all() and torch.isfinite(lse[b]).all()
        else:
            assert torch.all(o[b] == 0) and torch.all(torch.isneginf(lse[b]))
    rows = sample_rows(B, Hq, Sq, n_random=192, seed=Sq)
    ro, rl = oracle_for(x, scale, False, rows=rows)
    idx = torch.from_numpy(rows).cuda()
    compare(o.view(-1, d)[idx], lse.view(-1)[idx], ro, rl, f"split {B, Hq, Hkv, Sq, Sk, d}")
    del x, o, lse
    free_cuda()


def test_split_units_are_deterministic():
    """The merge of split units does not depend on which piece arrives last."""
    from attention_forward_blackwell_gb300 import binding, inputs
    assert binding.debug_prefill_plan(1, 1, 16384, 16384, 64, False, 152)[2] > 1   # split
    x = inputs.make_inputs(1, 1, 1, 16384, 16384, 64, tag=503, device="cuda")
    o1, l1 = _run(x, 0.088, False)
    for _ in range(5):
        o2, l2 = _run(x, 0.088, False)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_split_units_replay_in_a_cuda_graph():
    """A launch with split units (last-arriver merge, per-launch counters)
    captured in a CUDA graph and replayed: every replay equals the eager
    result bit for bit (the last piece resets its counter)."""
    from attention_forward_blackwell_gb300 import binding, inputs
    x = inputs.make_inputs(1, 2, 2, 4096, 4096, 64, tag=990, device="cuda")
    assert binding.debug_prefill_plan(1, 2, 4096, 4096, 64, 0, 152)[2] > 1   # split
    o_ref, l_ref = binding.prefill(x.q, x.k, x.v)
    o = torch.empty_like(x.q)
    lse = torch.empty(1, 2, 4096, device="cuda")
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


@pytest.mark.parametrize("B,Hq,Hkv,S,d,causal", [
    (1, 128, 8, 300, 128, True),      # many heads: 128 x 2 units
    (64, 2, 1, 129, 64, False),       # many tiny sequences: 128 units of 129 rows
])
def test_wide_grids(B, Hq, Hkv, S, d, causal):
    """Grids of many small units (every unit boundary case at once)."""
    from attention_forward_blackwell_gb300 import binding, inputs
    x = inputs.make_inputs(B, Hq, Hkv, S, S, d, tag=660 + Hq, device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = binding.prefill(x.q, x.k, x.v, scale=scale, causal=causal)
    torch.cuda.synchronize()
    check_device_error()
    rows = sample_rows(B, Hq, S, n_random=600, seed=B + Hq)
    ro, rl = oracle_for(x, scale, causal, rows=rows)
    idx = torch.from_numpy(rows).cuda()
    compare(o.view(-1, d)[idx], lse.view(-1)[idx], ro, rl, f"wide grid {B, Hq, Hkv, S, d}")
    free_cuda()


@pytest.mark.parametrize("causal", [False, True])
def test_long_context_128k_sampled(causal):
    """One head over 131,072 keys (the non-causal launch runs the persistent
    256-key kernel over 1,024 units of 512 key blocks; the causal one runs
    units of 2 to 1,024 blocks of 128 keys heaviest first): finiteness
    everywhere, sampled rows (tile edges at the start, middle and end plus
    random rows) against the oracle."""
    from attention_forward_blackwell_gb300 import binding, inputs
    S, d = 131072, 128
    if not causal:
        assert binding.debug_prefill_plan_ex(1, 1, S, S, d, 0, 152) == (1024, 0, 1, 128, 256, True)
    x = inputs.make_inputs(1, 1, 1, S, S, d, tag=1300, device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = binding.prefill(x.q, x.k, x.v, scale=scale, causal=causal)
    torch.cuda.synchronize()
    check_device_error()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    rows = sample_rows(1, 1, S, n_random=64, seed=S + causal)
    ro, rl = oracle_for(x, scale, causal, rows=rows)
    idx = torch.from_numpy(rows).cuda()
    compare(o.view(-1, d)[idx], lse.view(-1)[idx], ro, rl, f"128K keys causal={causal}")
    del x, o, lse
    free_cuda()
