"""Host logic of the prefill work split: which query blocks run whole and
which are split along the key axis (no GPU needed)."""
import math

import pytest

from attention_forward_blackwell_gb300 import binding

SHAPES = [
    # batch, hq, sq, sk, head_dim, causal
    (2, 16, 4096, 4096, 128, False),   # the bench: 512 blocks, 56 in the last wave
    (2, 16, 4096, 4096, 128, True),
    (1, 16, 8192, 8192, 128, False),
    (2, 16, 4096, 4096, 96, False),
    (4, 32, 2048, 2048, 256, True),
    (1, 1, 16384, 16384, 128, False),  # fewer blocks than SMs
    (1, 2, 5000, 7000, 96, False),
    (1, 2, 3000, 9000, 256, False),
    (3, 1, 2000, 30000, 64, False),
    (1, 1, 128, 128, 64, False),       # one block of one key tile
    (19, 8, 4096, 4096, 128, False),   # 304 blocks: whole waves only
    (1, 1, 300, 1000, 128, False),     # key tiles too few to split
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
@pytest.mark.parametrize("sms", [152, 148, 7])
def test_plan_invariants(shape, sms):
    batch, hq, sq, sk, d, causal = shape
    n_full, n_tail, split = binding.debug_prefill_plan(batch, hq, sq, sk, d, causal, sms)
    rows = 256 if d <= 128 else 128
    units = batch * hq * math.ceil(sq / rows)
    nk = math.ceil(sk / 128)
    assert n_full + n_tail == units
    if split == 1:
        assert n_tail == 0
    else:
        assert not causal                          # causal blocks are never split
        assert n_tail == units % sms and n_tail > 0
        assert n_full % sms == 0                   # whole blocks fill whole waves
        assert n_tail * split <= sms               # every piece runs in one wave
        assert nk // split >= 8                    # at least 8 key tiles per piece
        assert 2 <= split <= 8
        # the largest such split
        assert split == 8 or n_tail * (split + 1) > sms or nk // (split + 1) < 8


def test_plan_of_the_bench_workload():
    assert binding.debug_prefill_plan(2, 16, 4096, 4096, 128, False, 152) == (456, 56, 2)
    assert binding.debug_prefill_plan(2, 16, 4096, 4096, 128, True, 152) == (512, 0, 1)


def test_plan_rejects_bad_sizes():
    with pytest.raises(binding.FaError):
        binding.debug_prefill_plan(1, 1, 128, 128, 80, False, 152)
    with pytest.raises(binding.FaError):
        binding.debug_prefill_plan(1, 1, 128, 128, 128, False, 0)
