"""Host logic of the prefill work split: which kernel family runs a launch,
the sizes of its units and key blocks, and which query blocks run whole or
are split along the key axis (no GPU needed)."""
import math

import pytest

from attention_forward_blackwell_gb300 import binding

SHAPES = [
    # batch, hq, sq, sk, head_dim, causal
    (2, 16, 4096, 4096, 128, False),   # the bench workloads
    (2, 16, 4096, 4096, 128, True),
    (1, 16, 8192, 8192, 128, False),
    (2, 16, 4096, 4096, 96, False),
    (4, 32, 2048, 2048, 256, True),
    (4, 32, 2048, 2048, 64, False),
    (1, 1, 16384, 16384, 128, False),  # fewer blocks than SMs
    (1, 2, 5000, 7000, 96, False),
    (1, 2, 3000, 9000, 256, False),
    (3, 1, 2000, 30000, 64, False),
    (1, 1, 128, 128, 64, False),       # one block of one key tile
    (19, 8, 4096, 4096, 128, False),
    (19, 8, 4096, 4096, 64, False),    # 304 blocks: whole waves only
    (1, 1, 300, 1000, 128, False),
    (2, 8, 4096, 4096, 512, False),
]
KINDS = [
    # window, paged, packed
    (0, False, False),
    (0, True, False),
    (0, False, True),
    (1024, False, False),
]


def _wide(d, causal, window, paged, packed):
    """The 256-key persistent kernel: head_dim 96 / 128, dense, no window
    (causal or not)."""
    return d in (96, 128) and window <= 0 and not paged and not packed


@pytest.mark.parametrize("kind", KINDS, ids=[str(k) for k in KINDS])
@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
@pytest.mark.parametrize("sms", [152, 148, 7])
def test_plan_invariants(shape, kind, sms):
    batch, hq, sq, sk, d, causal = shape
    window, paged, packed = kind
    p = binding.debug_prefill_plan_ex(batch, hq, sq, sk, d, causal, sms, window=window,
                                      paged=paged, packed=packed)
    wide = _wide(d, causal, window, paged, packed)
    assert p.rows_per_unit == (128 if wide or d >= 256 else 256)
    assert p.keys_per_block == (256 if wide else 128)
    units = batch * hq * math.ceil(sq / p.rows_per_unit)
    nk = math.ceil(sk / p.keys_per_block)
    assert p.n_full + p.n_tail == units
    if wide:
        # persistent; whole units, except that at most half a wave of
        # non-causal units is split into k pieces of >= 4 key blocks, one
        # piece per CTA
        assert p.persistent
        k = min(sms // units, 8, nk // 4) if (not causal and units * 2 <= sms) else 1
        if k >= 2:
            assert (p.n_full, p.n_tail, p.split) == (0, units, k)
            assert units * k <= sms
        else:
            assert (p.n_full, p.n_tail, p.split) == (units, 0, 1)
        return
    assert p.persistent == (d == 256 and not packed and p.n_tail == 0 and p.n_full > 0)
    if p.split == 1:
        assert p.n_tail == 0
    else:
        # causal, windowed, packed and head_dim-512 units are never split
        assert not causal and window <= 0 and not packed and d != 512
        assert p.n_tail == units % sms and p.n_tail > 0
        assert p.n_full % sms == 0                     # whole blocks fill whole waves
        assert p.n_tail * p.split <= sms               # every piece runs in one wave
        assert nk // p.split >= 8                      # at least 8 key tiles per piece
        assert 2 <= p.split <= 8
        # the largest such split
        assert p.split == 8 or p.n_tail * (p.split + 1) > sms or nk // (p.split + 1) < 8


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_dense_plan_is_the_extended_one(shape):
    """fa_debug_prefill_plan is the dense, unwindowed case of the extended query."""
    batch, hq, sq, sk, d, causal = shape
    assert binding.debug_prefill_plan(batch, hq, sq, sk, d, causal, 152) == \
        tuple(binding.debug_prefill_plan_ex(batch, hq, sq, sk, d, causal, 152)[:3])


def test_plan_of_the_bench_workloads():
    plan = binding.debug_prefill_plan_ex
    # head_dim 128: 256-key kernel, 1024 units of 128 rows, persistent
    assert plan(2, 16, 4096, 4096, 128, False, 152) == (1024, 0, 1, 128, 256, True)
    assert plan(1, 16, 8192, 8192, 128, False, 152) == (1024, 0, 1, 128, 256, True)
    # causal: the same kernel, heaviest-first units
    assert plan(2, 16, 4096, 4096, 128, True, 152) == (1024, 0, 1, 128, 256, True)
    # with a window: two-tile kernel, one CTA per unit
    assert plan(2, 16, 4096, 4096, 128, True, 152, window=1024) == (512, 0, 1, 256, 128, False)
    # the same non-causal problem on paged caches: the last wave split in two
    assert plan(2, 16, 4096, 4096, 128, False, 152, paged=True) == (456, 56, 2, 256, 128, False)
    # causal GQA head_dim 256: persistent over 2048 units
    assert plan(4, 32, 2048, 2048, 256, True, 152) == (2048, 0, 1, 128, 128, True)
    assert binding.debug_prefill_plan(2, 16, 4096, 4096, 128, False, 152) == (1024, 0, 1)


def test_plan_rejects_bad_sizes():
    with pytest.raises(binding.FaError):
        binding.debug_prefill_plan(1, 1, 128, 128, 80, False, 152)
    with pytest.raises(binding.FaError):
        binding.debug_prefill_plan(1, 1, 128, 128, 128, False, 0)
    with pytest.raises(binding.FaError):
        binding.debug_prefill_plan_ex(1, 1, 128, 128, 128, False, 0, paged=True)


@pytest.mark.parametrize("sq", [1, 7, 16, 17, 32, 33, 64, 65, 128, 4096])
@pytest.mark.parametrize("hq,hkv", [(32, 4), (16, 8), (12, 2), (8, 8), (6, 1), (4, 1)])
@pytest.mark.parametrize("d,kind", [(128, (0, False, False)), (96, (0, False, False)),
                                    (64, (0, False, False)), (128, (64, False, False)),
                                    (128, (0, True, False))])
def test_gqa_head_packing_plan(sq, hq, hkv, d, kind):
    """Query heads per unit of the 256-key kernel: rows per head R = the next
    power of two >= sq in [16, 128], P = 128 / R reduced to a power of two
    dividing hq / hkv; units = batch x hq / P x ceil(sq / R).  Other kernels
    (head_dim 64, windows, paged caches) never pack."""
    window, paged, packed = kind
    batch, sk = 3, 1000
    p = binding.debug_prefill_plan_gqa(batch, hq, hkv, sq, sk, d, False, 152, window=window,
                                       paged=paged, packed=packed)
    g = hq // hkv
    if not _wide(d, False, window, paged, packed):
        assert p.pack == 1
        return
    rows = 16
    while rows < sq and rows < 128:
        rows *= 2
    pack = 128 // rows
    while pack > 1 and g % pack:
        pack //= 2
    assert p.pack == pack
    assert p.rows_per_unit == 128 // pack
    assert p.n_full == batch * (hq // pack) * math.ceil(sq / p.rows_per_unit)
    assert (p.n_tail, p.split, p.keys_per_block, p.persistent) == (0, 1, 256, True)
    # without the kv head count (or with hkv = hq) nothing is packed
    assert tuple(binding.debug_prefill_plan_ex(batch, hq, sq, sk, d, False, 152, window=window,
                                               paged=paged, packed=packed)) == \
        tuple(binding.debug_prefill_plan_gqa(batch, hq, hq, sq, sk, d, False, 152,
                                             window=window, paged=paged, packed=packed))[:6]


def test_gqa_plan_rejects_bad_group():
    with pytest.raises(binding.FaError):
        binding.debug_prefill_plan_gqa(1, 6, 4, 16, 128, 128, False, 152)
    with pytest.raises(binding.FaError):
        binding.debug_prefill_plan_gqa(1, 6, 0, 16, 128, 128, False, 152)


@pytest.mark.parametrize("shape,want", [
    ((1, 2, 300, 5000, 128, False), (0, 6, 5)),       # 6 units of 20 key blocks: 5 pieces each
    ((1, 1, 128, 65536, 96, False), (0, 1, 8)),       # one unit: 8 pieces
    ((1, 2, 300, 5000, 128, True), (6, 0, 1)),        # causal units are never split
    ((1, 2, 300, 1500, 128, False), (6, 0, 1)),       # 6 key blocks: pieces would be too short
    ((2, 40, 128, 8192, 128, False), (80, 0, 1)),     # more than half a wave
])
def test_few_units_of_the_256_key_kernel_are_split(shape, want):
    batch, hq, sq, sk, d, causal = shape
    assert tuple(binding.debug_prefill_plan_ex(batch, hq, sq, sk, d, causal, 152))[:3] == want


@pytest.mark.parametrize("batch,hq,hkv,sq,sk,d,causal,want", [
    # packed units (P heads x R rows), split along the keys when few
    (1, 32, 4, 16, 8192, 128, False, (0, 4, 8, 16, 256, True, 8)),
    (1, 16, 2, 8, 3000, 128, False, (0, 2, 3, 16, 256, True, 8)),
    (64, 32, 4, 16, 4096, 128, True, (256, 0, 1, 16, 256, True, 8)),
    (64, 32, 4, 16, 4096, 128, False, (256, 0, 1, 16, 256, True, 8)),
    (2, 8, 2, 40, 9000, 96, False, (0, 8, 8, 64, 256, True, 2)),    # 40 queries: 64 rows per head
    (1, 8, 8, 16, 9000, 128, False, (0, 8, 8, 128, 256, True, 1)),   # MHA: no packing
])
def test_packing_with_splits(batch, hq, hkv, sq, sk, d, causal, want):
    p = binding.debug_prefill_plan_gqa(batch, hq, hkv, sq, sk, d, causal, 152)
    assert tuple(p) == want
    n_full, n_tail, split = want[:3]
    assert n_full + n_tail == batch * (hq // want[6]) * math.ceil(sq / want[3])
    assert n_tail * split <= 152
