"""The float64 oracle against what the pages and the mathematics fix.

Runs on CPU only.  Each pin is documented in ``tests/oracle_pins.py``.
"""

import pytest

import oracle
import oracle.backward
import oracle.fp8
from oracle_pins import ALL_PINS, BWD_PINS, FP8_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(pin):
    pin(oracle)


@pytest.mark.parametrize("pin", FP8_PINS, ids=[p.__name__ for p in FP8_PINS])
def test_fp8_pin(pin):
    pin(oracle.fp8)


@pytest.mark.parametrize("pin", BWD_PINS, ids=[p.__name__ for p in BWD_PINS])
def test_bwd_pin(pin):
    pin(oracle.backward, oracle)


def test_head_pool_is_the_per_head_oracle():
    """oracle.parallel.HeadPool runs attention_f64 per head in spawn-started
    worker processes: every head's result is bit-identical to the in-process
    call on that head, for each mask, and each index comes back once."""
    import numpy as np

    from oracle.parallel import HeadPool

    rng = np.random.default_rng(3)
    heads, nq, nk, d = 5, 37, 53, 16
    q = rng.standard_normal((heads, nq, d)).astype(np.float32)
    k = rng.standard_normal((heads, nk, d)).astype(np.float32)
    v = rng.standard_normal((heads, nk, d)).astype(np.float32)
    with HeadPool(workers=2) as pool:
        for causal in (False, True, "bottom_right"):
            tasks = ((h, q[h], k[h], v[h], 0.25, causal) for h in range(heads))
            seen = set()
            for h, o, lse in pool.heads(tasks):
                o_ref, lse_ref = oracle.attention_f64(q[h].astype(np.float64), k[h].astype(np.float64),
                                                      v[h].astype(np.float64), 0.25, causal)
                assert np.array_equal(o, o_ref) and np.array_equal(lse, lse_ref)
                seen.add(h)
            assert seen == set(range(heads))
