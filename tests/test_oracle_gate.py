"""CPU pins of the oracle's gate support (WitCert §6.3.5 block-level paging).

* The per-page contributions sum to A - 1 exactly (the block decomposition of A).
* The contribution of a page equals the drop of A - 1 when its radii are set to 0 (its tokens exact)
  with the compressed distribution held fixed — the page's statement.
* Greedy by contribution is the shortest page-in list that brings the meter to tau (brute force over
  all subsets on small cases), with ties to the lower page index.
"""
import itertools
import math

import numpy as np
import pytest

from oracle import attention as A
from oracle.meter import greedy_page_in, page_log_contrib


def _case(rng, S):
    x = rng.standard_normal(S) * 2.0
    c = np.abs(rng.standard_normal(S)) * rng.choice([0.01, 0.3, 1.5])
    c[rng.random(S) < 0.1] = 0.0
    return x, c


@pytest.mark.parametrize("S", [1, 15, 16, 17, 100, 333])
def test_contributions_sum_to_a_minus_1(S):
    rng = np.random.default_rng(S)
    for _ in range(20):
        x, c = _case(rng, S)
        lc = page_log_contrib(x, c)
        lse = A.logsumexp(x)
        total = np.sum(np.exp(lc - lse))
        am1 = math.exp(A.log_a_minus_1(x - lse, c)) if np.any(c > 0) else 0.0
        assert total == pytest.approx(am1, rel=1e-12, abs=1e-300)


def test_contribution_is_the_drop_when_a_page_is_exact():
    rng = np.random.default_rng(5)
    x, c = _case(rng, 80)
    lse = A.logsumexp(x)
    pt = np.exp(x - lse)
    am1 = float(pt @ np.expm1(c))
    contrib = np.exp(page_log_contrib(x, c) - lse)
    for j in range(5):
        c2 = c.copy()
        c2[16 * j:16 * (j + 1)] = 0.0
        assert am1 - float(pt @ np.expm1(c2)) == pytest.approx(contrib[j], rel=1e-12)


def test_greedy_is_the_shortest_list_brute_force():
    rng = np.random.default_rng(7)
    for _ in range(200):
        n = int(rng.integers(1, 8))
        contrib = rng.exponential(size=n) * rng.choice([0.01, 0.2, 1.0])
        am1 = float(np.sum(contrib))
        tau = float(rng.choice([0.05, 0.2, 0.5]))
        k, chosen = greedy_page_in(contrib, am1, tau)
        target = math.sqrt(1 + 2 * tau) - 1
        # the greedy list reaches the target ...
        assert am1 - contrib[chosen].sum() <= target + 1e-12
        # ... and no shorter subset does
        best = next(r for r in range(n + 1) for sub in itertools.combinations(range(n), r)
                    if am1 - contrib[list(sub)].sum() <= target + 1e-12)
        assert k == best


def test_greedy_order_and_no_work_below_tau():
    contrib = np.array([0.1, 0.3, 0.3, 0.05])
    k, chosen = greedy_page_in(contrib, 0.75, 0.2)
    # target A - 1 = sqrt(1.4) - 1 = 0.1832: 0.75 - 0.3 - 0.3 = 0.15 (the two 0.3 pages, lower index first)
    assert k == 2 and list(chosen) == [1, 2]
    k0, ch0 = greedy_page_in(contrib, 0.05, 0.2)      # meter already <= tau
    assert k0 == 0 and ch0.size == 0
