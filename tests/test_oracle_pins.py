"""The fp64 oracle against closed forms, golden values, invariants, brute
force and an independent library routine (CPU only)."""
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle.attention_fwd)


def test_oracle_threads_match_single_thread():
    import numpy as np
    rng = np.random.default_rng(3)
    q = rng.standard_normal((2, 4, 37, 16))
    k = rng.standard_normal((2, 2, 41, 16))
    v = rng.standard_normal((2, 2, 41, 16))
    o1, l1 = oracle.attention_fwd(q, k, v, scale=0.25, causal=True,
                                  seqlens_k=[41, 20])
    o2, l2 = oracle.attention_fwd(q, k, v, scale=0.25, causal=True,
                                  seqlens_k=[41, 20], threads=5)
    assert (o1 == o2).all() and (l1 == l2).all()


def test_oracle_rejects_bad_arguments():
    import numpy as np
    q = np.zeros((1, 3, 2, 4))
    k = np.zeros((1, 2, 2, 4))
    with pytest.raises(RuntimeError):
        oracle.attention_fwd(q, k, k, scale=1.0)   # Hq % Hkv != 0
    with pytest.raises(RuntimeError):
        oracle.attention_fwd(np.zeros((1, 2, 2, 4)), k, k, scale=1.0, rows=[99])
