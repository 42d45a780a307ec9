"""The group bounds behind the streaming kernel's bounded second pass, checked in
float64 against the oracle's probabilities (no GPU).

At a position whose drafted token is accepted, the residual max(0, p - q) only
ranks the cache top-F ([SSD] "整体框架" with item 1; [SD] "The Algorithm
(Step-by-Step)" step 3 samples the residual only at a rejection).  Per 64-token
group g, with t* the token holding the group's largest target logit:
  r(t*) >= p(t*) - max_{t in g} q(t)   (a lower bound reached by t*),
  r(t)  <= max_{t in g} p(t)           for every t in g (an upper bound),
and both sides are monotone in the raw maxima, so the kernel needs only each
group's largest target and draft logits.  It takes the F-th largest of the largest
lower bound of 256 strided subsets of the groups (one per thread); this file checks
that at least F tokens reach that value and that every token of the exact top-F
(residual descending, id ascending) lies in a group whose upper bound reaches it --
for plain drafts, sigma_{F,C}-reshaped drafts (which only lower q inside the top-F
set) and identical rows (no positive bound: every group is kept)."""
import numpy as np
import pytest

import oracle

G_TOK = 64
THREADS = 256


def _bounds(zt, qbound):
    """Per-group (lower, upper) bounds from the raw maxima, as the kernel forms them:
    qbound[g] bounds every draft probability of group g from above."""
    p = oracle.softmax(zt, 1.0)
    V = zt.size
    G = (V + G_TOK - 1) // G_TOK
    lo = np.empty(G)
    up = np.empty(G)
    for g in range(G):
        sl = slice(g * G_TOK, min(V, (g + 1) * G_TOK))
        tstar = g * G_TOK + int(np.argmax(zt[sl]))
        lo[g] = p[tstar] - qbound[g]
        up[g] = p[tstar]
    return p, lo, up


def _group_max(x):
    V = x.size
    return np.array([x[g * G_TOK:min(V, (g + 1) * G_TOK)].max() for g in range((V + G_TOK - 1) // G_TOK)])


def _threshold(lo, F):
    """F-th largest of the threads' largest lower bounds (thread t: groups t, t+256, ...)."""
    per = [lo[t::THREADS].max() for t in range(min(THREADS, lo.size))]
    per.sort(reverse=True)
    return per[F - 1] if F <= len(per) else -np.inf


def _check(zt, q, qbound, F):
    p, lo, up = _bounds(zt, qbound)
    r = np.maximum(p - q, 0.0)
    T = _threshold(lo, F)
    order = np.lexsort((np.arange(r.size), -r))  # residual descending, id ascending
    top = order[:F]
    if T > 0:
        assert (r >= T).sum() >= F
        kept = up >= T
        assert kept[top // G_TOK].all()
        return int(kept.sum())
    return lo.size  # no positive bound: every group is computed


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("F", [1, 4, 9, 32])
def test_bounds_keep_the_exact_top_f(seed, F):
    rng = np.random.default_rng(700 + seed)
    V = 12000
    zd = rng.standard_normal(V) * 2.5 - 1.1 * np.log1p(np.arange(V))
    zt = zd + rng.standard_normal(V) * 0.8
    q = oracle.softmax(zd, 1.0)
    kept = _check(zt, q, _group_max(q), F)  # q is monotone in z_q: its group maximum
    assert kept < (V + G_TOK - 1) // G_TOK  # the bound prunes something on these rows


@pytest.mark.parametrize("C", [0.0, 0.3, 1.0])
def test_bounds_hold_for_reshaped_drafts(C):
    rng = np.random.default_rng(711)
    V = 9000
    zd = rng.standard_normal(V) * 2.5
    zt = zd + rng.standard_normal(V) * 0.8
    qs, _ = oracle.sigma(zd, 1.0, 16, C)
    # the kernel bounds q by the draft's raw group maximum against the reshaped
    # normaliser Z' = sum_t c_t e_t (e_t = exp(z_t - max z)): q'_t = c_t e_t / Z' <= e_t / Z'
    e = np.exp(zd - zd.max())
    with np.errstate(divide="ignore"):
        Zr = np.min((e / qs)[qs > 0])  # = Z' / max c_t = Z'
    qbound = _group_max(e) / Zr
    for g in range(qbound.size):
        assert qs[g * G_TOK:(g + 1) * G_TOK].max() <= qbound[g] * (1 + 1e-12)
    _check(zt, qs, qbound, 8)


def test_identical_rows_keep_every_group():
    rng = np.random.default_rng(712)
    z = rng.standard_normal(5000) * 2.0
    q = oracle.softmax(z, 1.0)
    assert _check(z, q, _group_max(q), 6) == (5000 + G_TOK - 1) // G_TOK
