"""The seeded input generators beyond the five workloads (no GPU): the PageGram report's slot
sweep tables (section 4: S in {1, 4, 8, 15, 60} at ~200M parameters, within 0.1 %) and the
distinct n-grams the collision statistic runs over."""
import numpy as np
import pytest

from hashed_head_gram_gb300 import workloads as W


def _is_prime(x):
    if x < 2:
        return False
    f = 2
    while f * f <= x:
        if x % f == 0:
            return False
        f += 1
    return True


def test_slot_sweep_is_the_reports():
    assert W.SLOT_SWEEP == (1, 4, 8, 15, 60)
    assert W.pagegram_slots(4).pages == [48823, 48821]          # the report's primes at S = 4


@pytest.mark.parametrize("S", W.SLOT_SWEEP)
def test_slot_sweep_tables_keep_the_budget(S):
    spec = W.pagegram_slots(S)
    base = W.make_workload(2).tables[0]
    assert spec.S == S and spec.K == base.K and spec.r == base.r and spec.orders == base.orders
    assert all(_is_prime(p) for p in spec.pages) and spec.pages[0] > spec.pages[1]
    params = spec.table_rows * spec.r
    assert abs(params / 200e6 - 1) < 1e-3                       # ~200M parameters, within 0.1 %
    # the largest primes under the budget: nothing between them and 48,823 * 4 / S
    top = (48823 * 4) // S
    assert not any(_is_prime(x) for x in range(spec.pages[0] + 1, top + 1))


@pytest.mark.parametrize("n,order", [(1, 2), (1000, 2), (4097, 2), (30000, 3), (5000, 1)])
def test_distinct_ngrams_are_distinct_and_reproducible(n, order):
    a = W.distinct_ngrams(n, order, 50304, seed=3)
    b = W.distinct_ngrams(n, order, 50304, seed=3)
    c = W.distinct_ngrams(n, order, 50304, seed=4)
    assert a.shape == (n, order) and a.dtype == np.int32
    assert np.array_equal(a, b) and (n < 50 or not np.array_equal(a, c))
    assert a.min() >= 0 and a.max() < 50304
    keys = np.zeros(n, np.int64)
    for j in range(order):
        keys = keys * 50304 + a[:, j]
    assert len(np.unique(keys)) == n


def test_distinct_ngrams_reject_a_too_small_vocabulary():
    with pytest.raises(ValueError):
        W.distinct_ngrams(10001, 2, 100, seed=0)


def test_uniform_control_tokens():
    w = W.make_workload(2)
    z = W.make_tokens(w)
    u = W.make_tokens(w, uniform=True)
    assert u.shape == z.shape and u.dtype == np.int32 and u.max() < w.vocab and u.min() >= 0
    assert np.array_equal(u, W.make_tokens(w, uniform=True))
    # Zipf repeats IDs far more often than uniform draws do
    assert len(np.unique(z)) < 0.5 * len(np.unique(u))
