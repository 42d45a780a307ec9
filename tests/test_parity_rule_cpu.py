"""The parity harness itself (tests/_parity.py), on hand-made outcomes: which GPU/oracle
differences it forgives and which fail a test.  Exact decisions must match; a decision
whose oracle margin is below 1e-6 may differ (and is counted); an exact tie among cache
scores is decided by the lowest id on both sides, so a swap there is a hard failure."""
import numpy as np
import pytest

_parity = pytest.importorskip("_parity")


def _verify_outcome(a, bonus, acc_margin, bonus_margin, K):
    B = len(a)
    p = np.full((B, K), 0.25)
    q = np.full((B, K), 0.5)
    for b in range(B):
        p[b, a[b] + 1:] = np.nan
        q[b, a[b] + 1:] = np.nan
    return {"accept_len": np.array(a), "bonus": np.array(bonus), "acc_margin": np.array(acc_margin),
            "bonus_margin": np.array(bonus_margin), "p_tok": p, "q_tok": q}


def test_identical_outcomes_pass():
    K = 3
    o = _verify_outcome([0, 3], [5, 9], np.full((2, K), 0.1), [0.1, 0.1], K)
    t = _parity.Tally()
    _parity.compare_verify(dict(o), o, K, t)
    assert not t.hard and t.exempt == 0 and t.decisions > 0


def test_accept_length_differs_only_at_a_near_tie():
    K = 3
    am = np.full((2, K), 0.1)
    am[0, 1] = 1e-7  # the oracle's |u - p/q| at position 1 of sequence 0
    o = _verify_outcome([1, 2], [5, 9], am, [0.1, 0.1], K)
    g = _verify_outcome([2, 2], [7, 9], am, [0.1, 0.1], K)
    t = _parity.Tally()
    _parity.compare_verify(g, o, K, t)
    assert not t.hard and t.exempt == 1
    o["acc_margin"][0, 1] = 1e-3  # the same difference with a clear margin fails
    t = _parity.Tally()
    _parity.compare_verify(g, o, K, t)
    assert len(t.hard) == 1 and "accept_len" in t.hard[0]


def test_bonus_differs_only_at_a_near_tie():
    K = 2
    o = _verify_outcome([1], [4], np.full((1, K), 0.1), [5e-7], K)
    g = _verify_outcome([1], [5], np.full((1, K), 0.1), [5e-7], K)
    t = _parity.Tally()
    _parity.compare_verify(g, o, K, t)
    assert not t.hard and t.exempt == 1
    o["bonus_margin"] = np.array([2e-6])
    t = _parity.Tally()
    _parity.compare_verify(g, o, K, t)
    assert len(t.hard) == 1 and "bonus" in t.hard[0]


def test_probabilities_within_1e5():
    K = 2
    o = _verify_outcome([1], [4], np.full((1, K), 0.1), [0.1], K)
    g = {k: np.array(v, copy=True) for k, v in o.items()}
    g["p_tok"][0, 0] += 9e-6
    t = _parity.Tally()
    _parity.compare_verify(g, o, K, t)
    assert not t.hard
    g["p_tok"][0, 0] += 2e-6  # now 1.1e-5 away
    t = _parity.Tally()
    _parity.compare_verify(g, o, K, t)
    assert len(t.hard) == 1
    o = _verify_outcome([0], [4], np.full((1, K), 0.1), [0.1], K)
    g = {k: np.array(v, copy=True) for k, v in o.items()}
    g["q_tok"][0, 1] = 0.5  # past the accepted length (a = 0) the outputs must be NaN
    t = _parity.Tally()
    _parity.compare_verify(g, o, K, t)
    assert len(t.hard) == 1 and "NaN" in t.hard[0]


def _cache_outcome(tokens, scores, margin, tau=1.0):
    return {"cache_tok": np.array([tokens], np.int32), "cache_score": np.array([scores], np.float64),
            "cache_margin": np.array([[margin]]), "temperature": np.array([tau], np.float32)}


def test_cache_exact_tie_is_a_hard_failure():
    off = [0, 3]
    o = _cache_outcome([2, 7, 9], [0.3, 0.1, 0.1], 0.05)  # ids 7 and 9 tie: lowest id first
    t = _parity.Tally()
    _parity.compare_cache(np.array([[2, 9, 7]]), o, off, 0, t)
    assert len(t.hard) == 1 and t.exempt == 0


def test_cache_near_gap_is_forgiven():
    off = [0, 3]
    o = _cache_outcome([2, 7, 9], [0.3, 0.1 + 5e-7, 0.1], 0.05)
    t = _parity.Tally()
    _parity.compare_cache(np.array([[2, 9, 7]]), o, off, 0, t)
    assert not t.hard and t.exempt == 1


def test_cache_boundary_near_tie_is_forgiven_and_a_clear_one_is_not():
    off = [0, 2]
    o = _cache_outcome([2, 7], [0.3, 0.1], 2e-7)  # the next score outside is 2e-7 below
    t = _parity.Tally()
    _parity.compare_cache(np.array([[2, 8]]), o, off, 0, t)
    assert not t.hard and t.exempt == 1
    o = _cache_outcome([2, 7], [0.3, 0.1], 1e-3)
    t = _parity.Tally()
    _parity.compare_cache(np.array([[2, 8]]), o, off, 0, t)
    assert len(t.hard) == 1


def test_clamped_zero_residuals_are_exempt_only_when_sampled():
    off = [0, 3]
    o = _cache_outcome([2, 7, 9], [0.3, 0.0, 0.0], 0.05, tau=1.0)  # (p - q)^+ clamped to 0
    t = _parity.Tally()
    _parity.compare_cache(np.array([[2, 9, 7]]), o, off, 0, t)
    assert not t.hard and t.exempt == 1
    o = _cache_outcome([2, 7, 9], [0.3, 0.0, 0.0], 0.05, tau=0.0)  # greedy: raw logits tie
    t = _parity.Tally()
    _parity.compare_cache(np.array([[2, 9, 7]]), o, off, 0, t)
    assert len(t.hard) == 1


def test_lookup_reference():
    cache = np.array([[4, 5, 6, 7], [1, 2, 3, 3]], np.int32)
    off = [0, 2, 4]
    hit, slot = _parity.lookup_from(cache, off, np.array([1, 0]), np.array([7, 3]))
    assert hit.tolist() == [1, 0] and slot.tolist() == [3, -1]
