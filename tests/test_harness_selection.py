"""The kept-set comparison of the parity tests, checked on the CPU.

check_selection decides whether a GPU kept set may differ from the oracle's:
only where the pages that differ are tied (1e-5 relative) or within the fp32
summation bounds of those two pages.  These cases plant each kind of
difference in hand-made score arrays and check the verdict and the tally.
"""
import numpy as np
import pytest

from tests import harness as H


@pytest.fixture(autouse=True)
def _keep_session_tally():
    # these planted cases must not count in the session's parity tally
    saved = dict(H.SEL_STATS)
    yield
    H.SEL_STATS.update(saved)


def _oracle_set(scores, k):
    N = len(scores)
    cand = np.arange(1, N - 1)
    order = cand[np.lexsort((cand, -scores[cand]))]
    return np.sort(np.concatenate([[0, N - 1], order[:k - 2]]))


def _row(ids, width):
    out = np.full(width, -1, dtype=np.int64)
    out[:len(ids)] = np.sort(ids)
    return out


# pages 1..8 are candidates; page 0 and 9 are forced; k = 5 keeps 3 candidates
S = np.array([0.0, 9.0, 3.0, 10.0, 8.0, 1.0, 2.0, 7.5, 0.5, -1.0])
K = 5
TOL = np.full(len(S), 1e-9)


def _delta(before):
    return {k: H.SEL_STATS[k] - before[k] for k in H.SEL_STATS}


def test_identical_sets_pass():
    o = _oracle_set(S, K)
    assert list(o) == [0, 1, 3, 4, 9]
    before = dict(H.SEL_STATS)
    assert H.check_selection(_row(o, 8), S, S, o, K, TOL) is True
    d = _delta(before)
    assert d["units"] == 1 and d["identical"] == 1


def test_exact_tie_may_go_either_way():
    s = S.copy()
    s[7] = 8.0                         # page 7 ties page 4 at the boundary
    o = _oracle_set(s, K)
    assert list(o) == [0, 1, 3, 4, 9]  # lower index wins in the oracle
    gpu = np.array([0, 1, 3, 7, 9])
    before = dict(H.SEL_STATS)
    assert H.check_selection(_row(gpu, 8), None, s, o, K, TOL) is False
    assert _delta(before)["tie_band"] == 1


def test_difference_within_the_pages_fp32_bound_passes_and_is_counted():
    s = S.copy()
    s[7] = 8.0 - 5e-4                  # 6e-5 relative: outside the tie rule
    tol = TOL.copy()
    tol[4] = tol[7] = 3e-4             # but inside the two pages' fp32 bounds
    o = _oracle_set(s, K)
    gpu = np.array([0, 1, 3, 7, 9])
    before = dict(H.SEL_STATS)
    assert H.check_selection(_row(gpu, 8), None, s, o, K, tol) is False
    assert _delta(before)["fp32_band"] == 1


def test_bound_of_other_pages_does_not_widen_the_band():
    s = S.copy()
    s[7] = 8.0 - 5e-4
    tol = TOL.copy()
    tol[2] = 1.0                       # a large bound on a page that is not involved
    o = _oracle_set(s, K)
    with pytest.raises(AssertionError, match="outside the tie band"):
        H.check_selection(_row(np.array([0, 1, 3, 7, 9]), 8), None, s, o, K, tol)


@pytest.mark.parametrize("gpu", [
    [0, 1, 3, 7, 9],                   # 7.5 kept instead of 8.0: not tied
    [0, 1, 3, 2, 9],                   # a low page kept
    [0, 3, 4, 7, 9],                   # the best candidate dropped
])
def test_untied_differences_fail(gpu):
    o = _oracle_set(S, K)
    with pytest.raises(AssertionError):
        H.check_selection(_row(np.array(gpu), 8), None, S, o, K, TOL)


def test_structural_errors_fail():
    o = _oracle_set(S, K)
    bad_order = np.array([0, 3, 1, 4, 9, -1, -1, -1])
    with pytest.raises(AssertionError):
        H.check_selection(bad_order, None, S, o, K, TOL)
    no_sink = _row(np.array([1, 3, 4, 7, 9]), 8)
    with pytest.raises(AssertionError):
        H.check_selection(no_sink, None, S, o, K, TOL)
    short = _row(np.array([0, 1, 3, 9]), 8)
    with pytest.raises(AssertionError):
        H.check_selection(short, None, S, o, K, TOL)
    garbage_tail = _row(o, 8)
    garbage_tail[-1] = 5
    with pytest.raises(AssertionError):
        H.check_selection(garbage_tail, None, S, o, K, TOL)


def test_gpu_set_must_follow_its_own_scores():
    s = S.copy()
    s[7] = 8.0
    o = _oracle_set(s, K)
    gpu = np.array([0, 1, 3, 7, 9])
    g_scores = s.copy()                # the GPU's own ranking keeps page 4, not 7
    with pytest.raises(AssertionError):
        H.check_selection(_row(gpu, 8), g_scores, s, o, K, TOL)
    g_scores[7] = 8.0 + 1e-6           # now its ranking keeps 7
    assert H.check_selection(_row(gpu, 8), g_scores, s, o, K, TOL) is False
