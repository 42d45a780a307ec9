"""Pins of the float64 CPU oracle against what the pages and mathematics fix.

Nothing here retypes the oracle's own formulas: each test checks the oracle
(through its C entry points) against a value the pages print, a closed form, a
library routine on a special case, exact enumeration, brute force or a Monte
Carlo test with a stated error bound.
"""
import json
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
import synth


def _logits(prob_rows):
    """fp32 logits whose tau=1 softmax is the given probability rows."""
    return np.log(np.asarray(prob_rows, dtype=np.float64)).astype(np.float32)


def _batch(rows, B):
    return np.ascontiguousarray(np.broadcast_to(rows, (B,) + rows.shape))


def _sample(rng, probs, n):
    """n draws from a probability vector (inverse CDF on numpy's cumulative sum)."""
    c = np.cumsum(probs)
    return np.minimum(np.searchsorted(c, rng.random(n) * c[-1], side="right"),
                      len(probs) - 1).astype(np.int32)


# ---------------------------------------------------------------------------
# Worked example table.
# ---------------------------------------------------------------------------

def test_worked_table(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "worked_table.json")))
    pos = g["positions"]
    K = len(pos)
    p_rows = [r["p"] for r in pos] + [[1 / 3, 1 / 3, 1 / 3]]
    q_rows = [r["q"] for r in pos]
    tgt = _logits(p_rows)[None]
    drf = _logits(q_rows)[None]
    x = np.array([[r["drafted"] for r in pos]], np.int32)
    tau = np.ones(1, np.float32)
    # u = 0.3 on the third draw: min(1, 0.2/0.4) = 0.5 > 0.3 -> accepted.
    for u_last in (0.0, 0.3, 0.4999):
        u = np.array([[0.999, 0.999, u_last, 0.5]], np.float32)
        o = oracle.verify(tgt, drf, x, u, tau, "f32")
        assert o["accept_len"][0] == K
    # u = 0.7: the coin flip fails -> a = 2, residual [0, .4, 0] -> bonus "." for every u_K.
    for u_k in (0.0, 0.25, 0.5, 0.999):
        u = np.array([[0.999, 0.999, 0.7, u_k]], np.float32)
        o = oracle.verify(tgt, drf, x, u, tau, "f32")
        assert o["accept_len"][0] == g["outcome_when_third_rejected"]["accepted"]
        assert o["bonus"][0] == g["residual_favourite"]
        assert o["Z"][0] == pytest.approx(sum(g["residual_at_t+2"]), abs=1e-6)
        np.testing.assert_allclose(o["p_tok"][0], [r["p_tok"] for r in pos], atol=1e-6)
        np.testing.assert_allclose(o["q_tok"][0], [r["q_tok"] for r in pos], atol=1e-6)
        ratio = o["p_tok"][0] / o["q_tok"][0]
        np.testing.assert_allclose(np.minimum(1, ratio), [r["ratio"] for r in pos], atol=1e-6)
        assert o["acc_margin"][0][2] == pytest.approx(0.2, abs=1e-6)
        assert np.isinf(o["acc_margin"][0][:2]).all()


# ---------------------------------------------------------------------------
# Losslessness: the first emitted token is distributed as p.
# ---------------------------------------------------------------------------

def _mc_first_token(rng, p_rows, q_rows, n):
    K = len(q_rows)
    V = len(p_rows[0])
    tgt = _batch(_logits(p_rows), n)
    drf = _batch(_logits(q_rows), n)
    q_norm = [np.asarray(q) / np.sum(q) for q in q_rows]
    x = np.stack([_sample(rng, q_norm[i], n) for i in range(K)], axis=1)
    u = rng.random((n, K + 1), dtype=np.float32)
    tau = np.ones(n, np.float32)
    o = oracle.verify(tgt, drf, x, u, tau, "f32")
    assert o["invalid"] == 0
    first = np.where(o["accept_len"] >= 1, x[:, 0], o["bonus"])
    return o, first, x, V


@pytest.mark.parametrize("K", [1, 3])
def test_lossless_chi_square(K):
    rng = np.random.default_rng(11 + K)
    V = 8
    p_rows = rng.dirichlet(np.ones(V), size=K + 1)
    q_rows = rng.dirichlet(np.ones(V), size=K)
    n = 1_000_000
    o, first, x, _ = _mc_first_token(rng, p_rows, q_rows, n)
    p0 = p_rows[0] / p_rows[0].sum()
    hist = np.bincount(first, minlength=V)
    pval = scipy.stats.chisquare(hist, p0 * n).pvalue
    assert pval > 1e-3, (hist, p0 * n, pval)
    # All K accepted: the bonus follows the extra target row p_K.
    allacc = o["accept_len"] == K
    pK = p_rows[K] / p_rows[K].sum()
    hK = np.bincount(o["bonus"][allacc], minlength=V)
    assert scipy.stats.chisquare(hK, pK * allacc.sum()).pvalue > 1e-3


def test_lossless_exact_enumeration():
    """P_final(x) = sum over drafts of q(d)[min(1,p/q) 1{x=d} + (1-min(1,p/q)) r(x)] = p(x),
    with the acceptance probability and the bonus law read off the oracle's own decisions
    (the accept threshold in u and the bonus intervals in u_K, found by bisection)."""
    rng = np.random.default_rng(5)
    V = 8
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V))
    tgt = _logits([p, p])[None]
    drf = _logits([q])[None]
    tau = np.ones(1, np.float32)

    def run(d, u0, uk):
        u = np.array([[u0, uk]], np.float32)
        return oracle.verify(tgt, drf, np.array([[d]], np.int32), u, tau, "f32")

    def threshold(pred):  # smallest fp32 u in [0,1) with pred(u) False (bisection)
        lo, hi = 0.0, 1.0
        if not pred(np.float32(0.0)):
            return 0.0
        for _ in range(40):
            mid = 0.5 * (lo + hi)
            if pred(np.float32(mid)):
                lo = mid
            else:
                hi = mid
        return hi

    # Bonus law on rejection at row 0 (independent of which draft was rejected).
    d_rej = int(np.argmax(q - p))
    edges = [0.0]
    for t in range(V):
        edges.append(threshold(lambda uk: run(d_rej, 0.99999, uk)["bonus"][0] <= t))
    r = np.diff(np.minimum(edges, 1.0))
    final = np.zeros(V)
    for d in range(V):
        acc = threshold(lambda u0: run(d, u0, 0.5)["accept_len"][0] == 1)
        final[d] += q[d] * acc
        final += q[d] * (1.0 - acc) * r
    np.testing.assert_allclose(final, p, atol=1e-6)


# ---------------------------------------------------------------------------
# Expected tokens per round under a constant per-position acceptance alpha.
# ---------------------------------------------------------------------------

def _const_alpha_rows(rng, alpha, V=8):
    """q on tokens 0..3, p = alpha q + (1-alpha) r with r on tokens 4..7:
    sum_t min(p_t, q_t) = alpha, so every position accepts with probability alpha."""
    q = np.zeros(V)
    q[:4] = rng.dirichlet(np.ones(4))
    r = np.zeros(V)
    r[4:] = rng.dirichlet(np.ones(4))
    p = alpha * q + (1 - alpha) * r
    q = np.where(q > 0, q, 1e-30)  # log-domain storage needs q > 0 (1e-30 is far below fp32 rounding of 1)
    p = np.where(p > 0, p, 1e-30)
    return p, q


@pytest.mark.parametrize("K", [4, 8])
def test_expected_tokens_closed_form(golden_dir, K):
    g = json.load(open(os.path.join(golden_dir, "expected_tokens.json")))
    alpha = g["alpha"]
    rng = np.random.default_rng(100 + K)
    p, q = _const_alpha_rows(rng, alpha)
    n = 400_000
    p_rows = [p] * (K + 1)
    q_rows = [q] * K
    o, _, _, _ = _mc_first_token(rng, p_rows, q_rows, n)
    a = o["accept_len"]
    closed = (1 - alpha ** (K + 1)) / (1 - alpha)
    series = sum((i + 1) * alpha ** i * (1 - alpha) for i in range(K)) + (K + 1) * alpha ** K
    assert closed == pytest.approx(series, rel=1e-12)
    tokens = a + 1
    se = tokens.std() / np.sqrt(n)
    assert abs(tokens.mean() - closed) < 4 * se
    case = [c for c in g["cases"] if c["K"] == K][0]
    assert abs(closed - case["approx"]) < case["printed_precision"]
    # P(a = i) = alpha^i (1 - alpha) for i < K, P(a = K) = alpha^K.
    pmf = np.array([alpha ** i * (1 - alpha) for i in range(K)] + [alpha ** K])
    hist = np.bincount(a, minlength=K + 1)
    assert scipy.stats.chisquare(hist, pmf * n).pvalue > 1e-3


# ---------------------------------------------------------------------------
# Temperature softmax and greedy decisions.
# ---------------------------------------------------------------------------

def test_softmax_matches_library():
    rng = np.random.default_rng(3)
    for V, tau in [(2, 1.0), (33, 0.7), (1000, 1.3), (128256, 1.0)]:
        z = rng.standard_normal(V) * 3
        p = oracle.softmax(z, tau)
        np.testing.assert_allclose(p, scipy.special.softmax(z / tau), rtol=1e-12, atol=1e-300)
        assert p.sum() == pytest.approx(1.0, abs=1e-12)


def test_greedy_matches_argmax():
    rng = np.random.default_rng(4)
    B, K, V = 64, 4, 37
    # integer-valued logits so that ties are frequent; numpy argmax returns the lowest id.
    tgt = rng.integers(-3, 4, size=(B, K + 1, V)).astype(np.float32)
    drf = np.zeros((B, K, V), np.float32)
    am = np.argmax(tgt, axis=-1)
    x = np.where(rng.random((B, K)) < 0.7, am[:, :K], rng.integers(0, V, (B, K))).astype(np.int32)
    u = rng.random((B, K + 1), dtype=np.float32)
    tau = np.zeros(B, np.float32)
    o = oracle.verify(tgt, drf, x, u, tau, "f32")
    for b in range(B):
        mism = np.nonzero(x[b] != am[b, :K])[0]
        a = int(mism[0]) if len(mism) else K
        assert o["accept_len"][b] == a
        assert o["bonus"][b] == am[b, a]


def test_bf16_storage_reads_exact_values():
    rng = np.random.default_rng(6)
    B, K, V = 4, 2, 300
    z = rng.standard_normal((B, K + 1, V)).astype(np.float32) * 3
    zb = synth.bf16_bits_from_f32(z)
    z_round = synth.f32_from_bf16_bits(zb)
    d = rng.standard_normal((B, K, V)).astype(np.float32) * 3
    db = synth.bf16_bits_from_f32(d)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K + 1), dtype=np.float32)
    tau = np.full(B, 0.8, np.float32)
    o1 = oracle.verify(zb, db, x, u, tau, "bf16")
    o2 = oracle.verify(z_round, synth.f32_from_bf16_bits(db), x, u, tau, "f32")
    for key in ("accept_len", "bonus"):
        np.testing.assert_array_equal(o1[key], o2[key])
    np.testing.assert_array_equal(o1["p_tok"], o2["p_tok"])


def test_bf16_conversion_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 50,
                        np.array([0.0, -0.0, 1e-40, -1e-40, 3.4e38, np.inf, -np.inf], np.float32)])
    ours = synth.bf16_bits_from_f32(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


# ---------------------------------------------------------------------------
# Bonus draws: inverse CDF over ascending token id.
# ---------------------------------------------------------------------------

def test_bonus_all_accepted_is_inverse_cdf_of_pK():
    rng = np.random.default_rng(8)
    V, K, n = 50, 2, 200
    z = rng.standard_normal((K + 1, V)).astype(np.float32) * 2
    tgt = _batch(z, n)
    drf = _batch(z[:K], n)          # q == p: every draft is accepted
    x = rng.integers(0, V, (n, K)).astype(np.int32)
    u = rng.random((n, K + 1), dtype=np.float32)
    o = oracle.verify(tgt, drf, x, u, np.ones(n, np.float32), "f32")
    assert (o["accept_len"] == K).all()
    pK = scipy.special.softmax(z[K].astype(np.float64))
    want = np.searchsorted(np.cumsum(pK), u[:, K].astype(np.float64) * pK.sum(), side="right")
    np.testing.assert_array_equal(o["bonus"], want)


def test_bonus_on_rejection_is_inverse_cdf_of_residual():
    rng = np.random.default_rng(9)
    V, K, n = 64, 1, 300
    zp = (rng.standard_normal((K + 1, V)) * 2).astype(np.float32)
    zq = (rng.standard_normal((K, V)) * 2).astype(np.float32)
    p = scipy.special.softmax(zp[0].astype(np.float64))
    q = scipy.special.softmax(zq[0].astype(np.float64))
    d = int(np.argmax(q / p))                     # q(d) >> p(d): rejected unless u < p/q
    x = np.full((n, K), d, np.int32)
    u = rng.random((n, K + 1), dtype=np.float32)
    u[:, 0] = np.maximum(u[:, 0], np.float32(p[d] / q[d] + 1e-3))
    o = oracle.verify(_batch(zp, n), _batch(zq, n), x, u, np.ones(n, np.float32), "f32")
    assert (o["accept_len"] == 0).all()
    w = np.maximum(p - q, 0.0)
    want = np.searchsorted(np.cumsum(w), u[:, K].astype(np.float64) * w.sum(), side="right")
    np.testing.assert_array_equal(o["bonus"], want)
    np.testing.assert_allclose(o["Z"], w.sum(), rtol=1e-12)


def _z0_rows(rng, K, V, reject_at):
    """Target = draft at every position (p_i == q_i, so the residual is zero
    everywhere), with the drafted token at -inf in both rows at `reject_at`: that
    token has p = q = 0, u * 0 < 0 fails for every u, so the draft is rejected there
    with Z = 0.  Earlier positions draft a finite token with p == q > 0, accepted for
    every u < 1.  Each position has its own row, so a draw from the wrong row shows."""
    z = (rng.standard_normal((K + 1, V)) * 2).astype(np.float32)
    x = np.array([int(np.argmax(z[i])) for i in range(K)], np.int32)
    x[reject_at] = (x[reject_at] + 3) % V
    z[reject_at, x[reject_at]] = -np.inf
    return z, x


@pytest.mark.parametrize("reject_at", [0, 1, 2])
def test_bonus_when_residual_is_zero_is_drawn_from_p(reject_at):
    """Z = 0 at the rejected row (p_a == q_a): the reading draws the bonus from p_a,
    the residual's limit.  Pinned against numpy's inverse CDF of the library softmax
    of row a, so drawing from the all-zero residual, from another row or with another
    uniform fails."""
    rng = np.random.default_rng(17 + reject_at)
    V, K, n = 40, 3, 400
    z, x = _z0_rows(rng, K, V, reject_at)
    p = scipy.special.softmax(z[reject_at].astype(np.float64))
    assert p[x[reject_at]] == 0.0
    c = np.cumsum(p)
    u = rng.random((n, K + 1), dtype=np.float32)
    T = u[:, K].astype(np.float64) * c[-1]
    keep = np.min(np.abs(T[:, None] - c[None, :]), axis=1) > 1e-9   # away from CDF steps
    o = oracle.verify(_batch(z, n), _batch(z[:K], n), _batch(x, n), u, np.ones(n, np.float32),
                      "f32")
    assert (o["accept_len"] == reject_at).all()
    want = np.searchsorted(c, T, side="right")
    np.testing.assert_array_equal(o["bonus"][keep], want[keep])
    assert keep.mean() > 0.95
    # the draw covers the support of p_a, never the rejected token
    assert x[reject_at] not in set(o["bonus"].tolist())
    assert len(set(o["bonus"].tolist())) > 5


@pytest.mark.parametrize("reject_at", [0, 2])
def test_p_hit_when_residual_is_zero_is_the_cached_mass_of_p(reject_at):
    """With every draft before `reject_at` accepted for sure and the one at
    `reject_at` rejected for sure with Z = 0, the outcome length is fixed and
    P_hit = sum_{t in S_a} p_a(t) (closed form from the library softmax); the hit
    frequency of the oracle's own rounds agrees within Monte Carlo error."""
    rng = np.random.default_rng(31 + reject_at)
    V, K, n = 40, 3, 100_000
    z, x = _z0_rows(rng, K, V, reject_at)
    F = [5, 4, 6, 3]
    off = np.concatenate([[0], np.cumsum(F)]).astype(np.int32)
    budget = int(off[-1])
    # segment a holds some likely and some unlikely tokens of p_a; other segments hold
    # the tokens p_a favours most, so a wrong segment changes the answer
    order = np.argsort(-z[reject_at], kind="stable")
    cache = np.zeros((1, budget), np.int32)
    for k in range(K + 1):
        cache[0, off[k]:off[k + 1]] = order[:F[k]] if k != reject_at else order[[1, 3, 7, 12, 20, 25]][:F[k]]
    p = scipy.special.softmax(z[reject_at].astype(np.float64))
    want = p[cache[0, off[reject_at]:off[reject_at + 1]]].sum()
    got = oracle.p_hit(z[None], z[None, :K], x[None], np.ones(1, np.float32), "f32", off,
                       budget, cache)[0]
    assert got == pytest.approx(want, abs=1e-12)
    u = rng.random((n, K + 1), dtype=np.float32)
    v = oracle.verify(_batch(z, n), _batch(z[:K], n), _batch(x, n), u, np.ones(n, np.float32),
                      "f32")
    h = oracle.lookup(_batch(cache[0], n), off, v["accept_len"], v["bonus"])["hit"]
    se = np.sqrt(want * (1 - want) / n)
    assert abs(h.mean() - want) < 4 * se, (h.mean(), want)


def test_invalid_inputs_are_flagged():
    rng = np.random.default_rng(10)
    B, K, V = 4, 2, 16
    tgt = rng.standard_normal((B, K + 1, V)).astype(np.float32)
    drf = rng.standard_normal((B, K, V)).astype(np.float32)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    x[1, 1] = V          # out of range token
    x[2, 0] = -1
    tau = np.array([1.0, 1.0, 1.0, -0.5], np.float32)
    u = rng.random((B, K + 1), dtype=np.float32)
    o = oracle.verify(tgt, drf, x, u, tau, "f32")
    assert o["invalid"] == 3
    assert list(o["accept_len"][1:]) == [-1, -1, -1]
    assert o["accept_len"][0] >= 0
    tau2 = np.array([np.nan, 1, 1, 1], np.float32)
    x2 = rng.integers(0, V, (B, K)).astype(np.int32)
    o2 = oracle.verify(tgt, drf, x2, u, tau2, "f32")
    assert o2["accept_len"][0] == -1 and o2["invalid"] == 1


# ---------------------------------------------------------------------------
# Geometric fan-out.
# ---------------------------------------------------------------------------

def test_fanout_page_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "fanout_example.json")))
    F, off, x = oracle.fanout(g["K"], g["budget"], g["a_p"], g["r"])
    assert list(F) == g["F"]
    assert off[-1] == g["budget"]


@pytest.mark.parametrize("K,budget,a_p,r", [(6, 64, 0.8, 1.0), (4, 32, 0.75, 0.5),
                                            (3, 12, 0.5625, 1.0), (8, 100, 0.6, 0.0),
                                            (1, 5, 0.3, 2.0), (10, 7, 0.9, 0.25)])
def test_fanout_closed_form(K, budget, a_p, r):
    F, off, x = oracle.fanout(K, budget, a_p, r)
    g = a_p ** (1.0 / (1.0 + r))
    # shape: x_{k+1}/x_k = a_p^{1/(1+r)} for k+1 < K; x_K/x_{K-1} adds (1-a_p)^{-1/(1+r)}
    for k in range(K - 1):
        assert x[k + 1] / x[k] == pytest.approx(g, rel=1e-12)
    assert x[K] / x[K - 1] == pytest.approx(g * (1 - a_p) ** (-1.0 / (1.0 + r)), rel=1e-12)
    assert x.sum() == pytest.approx(budget, rel=1e-12)
    # integers: sum == budget, each within (floor, floor+1], the +1s on the largest remainders
    assert F.sum() == budget and off[-1] == budget
    np.testing.assert_array_equal(np.diff(off), F)
    fl = np.floor(x)
    assert ((F == fl) | (F == fl + 1)).all()
    frac = x - fl
    bumped = F == fl + 1
    if bumped.any() and (~bumped).any():
        assert frac[bumped].min() >= frac[~bumped].max()


def test_fanout_workload_shapes():
    # the cache shapes of the two cache workloads (K=6, budget 64, a_p=0.8, r=1) and
    # (K=4, budget 32, a_p=0.75, r=0.5): geometric decay with a larger all-accepted tail
    F, _, _ = oracle.fanout(6, 64, 0.8, 1.0)
    assert list(F) == [11, 10, 9, 8, 7, 6, 13]
    F, _, _ = oracle.fanout(4, 32, 0.75, 0.5)
    assert list(F) == [8, 6, 5, 4, 9]


def test_fanout_clamps_to_vocab():
    F, off, _ = oracle.fanout(2, 100, 0.5, 1.0, V=20)
    assert F.max() <= 20 and off[-1] == F.sum() and F.sum() < 100


def test_fanout_rejects_bad_parameters():
    for args in [(0, 10, 0.5, 1.0), (3, 10, 1.0, 1.0), (3, 10, 0.0, 1.0), (3, 10, 0.5, -1.0),
                 (3, -1, 0.5, 1.0)]:
        with pytest.raises(ValueError):
            oracle.fanout(*args)


@pytest.mark.parametrize("K,budget", [(1, 0), (1, 5), (2, 7), (3, 4), (3, 9), (4, 6)])
def test_fanout_uniform_is_the_even_split(K, budget):
    """Brute force over every allocation of the budget to the K+1 lengths: the even
    split is the only one whose shares differ by at most one and that gives the
    spare slots to the shortest accepted lengths (non-increasing in k)."""
    import itertools
    best = [F for F in itertools.product(range(budget + 1), repeat=K + 1)
            if sum(F) == budget and max(F) - min(F) <= 1
            and all(F[k] >= F[k + 1] for k in range(K))]
    assert len(best) == 1
    F, off = oracle.fanout_uniform(K, budget)
    assert tuple(F) == best[0]
    assert list(off) == [0] + list(np.cumsum(best[0]))


@pytest.mark.parametrize("K,budget", [(4, 32), (6, 64), (3, 10), (8, 100), (2, 1)])
def test_fanout_uniform_is_the_flat_limit_of_the_geometric_shape(K, budget):
    """As r grows the geometric shape F_0 a_p^{k/(1+r)} flattens to one value for every
    k (the all-accepted factor (1-a_p)^{-1/(1+r)} goes to 1 as well): the geometric
    allocation at r = 1e6 must equal the uniform one."""
    Fu, offu = oracle.fanout_uniform(K, budget)
    Fg, offg, _ = oracle.fanout(K, budget, 0.5, 1e6)
    np.testing.assert_array_equal(Fu, Fg)
    np.testing.assert_array_equal(offu, offg)


def test_fanout_uniform_clamps_and_rejects():
    F, off = oracle.fanout_uniform(2, 100, V=20)
    assert list(F) == [20, 20, 20] and off[-1] == 60
    for args in [(0, 10), (3, -1)]:
        with pytest.raises(ValueError):
            oracle.fanout_uniform(*args)


# ---------------------------------------------------------------------------
# Draft-only cache keys and the analytic hit probability.
# ---------------------------------------------------------------------------

def test_draft_cache_brute_force():
    """Library sort (numpy lexsort on (-value, id)) of every draft row, the drafted
    token dropped from its own segment; bf16-quantised rows make ties common."""
    rng = np.random.default_rng(50)
    B, K, V = 6, 3, 40
    z = np.round(rng.standard_normal((B, K + 1, V)) * 2).astype(np.float32) / 2
    drf = synth.store(z, "bf16")
    zs = synth.stored_to_f32(drf, "bf16").astype(np.float64)
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    tok[0] = np.argmax(zs[0, :K], axis=-1)           # drafted token at the top of its row
    for F in ([5, 3, 2, 7], [0, 1, 40, 4], [40, 40, 40, 40]):
        off = np.concatenate([[0], np.cumsum(F)]).astype(np.int32)
        budget = int(off[-1]) + 3
        got = oracle.draft_cache(drf, tok, "bf16", off, budget)
        for b in range(B):
            for k in range(K + 1):
                order = np.lexsort((np.arange(V), -zs[b, k]))
                if k < K:
                    order = order[order != tok[b, k]]
                want = np.full(F[k], -1)
                n = min(F[k], len(order))
                want[:n] = order[:n]
                np.testing.assert_array_equal(got[b, off[k]:off[k + 1]], want)
            assert (got[b, off[-1]:] == -2).all()  # columns past the segments untouched
    no_excl = oracle.draft_cache(drf, None, "bf16", off, budget)
    assert (no_excl[:, :off[-1]] >= 0).all()


def _sigma_np(z, F, C):
    """sigma_{F,C} of one row at tau = 1 with numpy: weight C on the F largest
    logits (lowest id on ties), 1 elsewhere."""
    order = np.lexsort((np.arange(len(z)), -z))
    c = np.ones(len(z))
    c[order[:F]] = C
    w = c * np.exp(z - z.max())
    return w / w.sum()


def test_p_hit_matches_monte_carlo():
    """The analytic per-sequence hit probability against the frequency of hits over
    200k rounds of the oracle's own sampling (same drafted tokens, fresh uniforms),
    with per-position sigma_{F_k, C} and draft-only cache keys."""
    rng = np.random.default_rng(51)
    K, V, n = 3, 48, 200_000
    F = [4, 3, 2, 5]
    off = np.concatenate([[0], np.cumsum(F)]).astype(np.int32)
    budget = int(off[-1])
    zp = (rng.standard_normal((K + 1, V)) * 1.5).astype(np.float32)
    zq = (zp + rng.standard_normal((K + 1, V)) * 0.8).astype(np.float32)
    x = np.array([int(np.argsort(-zq[i])[1]) for i in range(K)], np.int32)  # a top-F token
    C = 0.4
    cache = oracle.draft_cache(zq[None], x[None], "f32", off, budget)
    ph = oracle.p_hit(zp[None], zq[None], x[None], np.ones(1, np.float32), "f32", off, budget,
                      cache, reshape_F=F[:K], reshape_C=C)[0]
    u = rng.random((n, K + 1), dtype=np.float32)
    v = oracle.verify(_batch(zp, n), _batch(zq, n), _batch(x, n), u, np.ones(n, np.float32),
                      "f32", reshape_F=F[:K], reshape_C=C)
    h = oracle.lookup(_batch(cache[0], n), off, v["accept_len"], v["bonus"])["hit"]
    se = np.sqrt(ph * (1 - ph) / n)
    assert 0.05 < ph < 0.95
    assert abs(h.mean() - ph) < 4 * se, (h.mean(), ph)
    # greedy: the outcome is fixed, so the probability is exactly the hit
    g = oracle.p_hit(zp[None], zq[None], x[None], np.zeros(1, np.float32), "f32", off, budget,
                     cache)[0]
    vg = oracle.verify(zp[None], zq[None], x[None], u[:1], np.zeros(1, np.float32), "f32")
    hg = oracle.lookup(cache, off, vg["accept_len"], vg["bonus"])["hit"][0]
    assert g == float(hg)


@pytest.mark.parametrize("C", [1.0, 0.6, 0.2, 0.0])
def test_p_hit_averaged_over_the_draft_is_the_residual_mass(C):
    """K = 1, cache keys without the drafted token left out: averaged over
    x~ ~ q' = sigma_{F,C}(z_d), the probability of (reject, t* = t) is
    max(0, p(t) - q'(t)) for every t, and all-accepted has probability
    sum_t min(p, q'), so E[P_hit] = sum_{t in S_0} max(0, p - q') +
    sum_t min(p, q') * p_1(S_1) -- exact enumeration over the V drafted tokens.
    As C falls, q' shrinks on S_0 = top-F_0(z_d), so the first term grows."""
    rng = np.random.default_rng(52)
    V, F = 10, [3, 2]
    off = np.array([0, 3, 5], np.int32)
    zp = rng.standard_normal((2, V)).astype(np.float32)
    zq = (zp + rng.standard_normal((2, V)) * 0.9).astype(np.float32)
    cache = oracle.draft_cache(zq[None], None, "f32", off, 5)
    S0, S1 = cache[0, 0:3], cache[0, 3:5]
    tok = np.arange(V, dtype=np.int32).reshape(V, 1)
    ph = oracle.p_hit(_batch(zp, V), _batch(zq[:1], V), tok, np.ones(V, np.float32), "f32", off,
                      5, _batch(cache[0], V), reshape_F=[F[0]], reshape_C=C)
    p0 = scipy.special.softmax(zp[0].astype(np.float64))
    p1 = scipy.special.softmax(zp[1].astype(np.float64))
    q0 = _sigma_np(zq[0].astype(np.float64), F[0], C)
    expect = np.maximum(p0 - q0, 0)[S0].sum() + np.minimum(p0, q0).sum() * p1[S1].sum()
    assert abs(float(q0 @ ph) - expect) < 1e-12
    if C < 1.0:
        q1 = _sigma_np(zq[0].astype(np.float64), F[0], 1.0)
        assert np.maximum(p0 - q0, 0)[S0].sum() >= np.maximum(p0 - q1, 0)[S0].sum()


# ---------------------------------------------------------------------------
# Random-token backup.
# ---------------------------------------------------------------------------

def test_backup_fill_brute_force():
    """Exact rational arithmetic: token = floor(u * V) of the float u as a fraction,
    only on the rows that missed; rows that hit keep their previous contents."""
    from fractions import Fraction
    rng = np.random.default_rng(7)
    B, K = 12, 5
    below1 = np.nextafter(np.float32(1), np.float32(0))
    for V in [1, 2, 3, 1000, 128256, 152064, (1 << 24) + 3]:
        u = rng.random((B, K)).astype(np.float32)
        u[0, 0], u[0, 1] = 0.0, below1
        u[0, 2] = np.float32(0.5)
        hit = (rng.random(B) < 0.4).astype(np.uint8)
        hit[0] = 0
        nxt = np.full((B, K), -7, np.int32)
        oracle.backup_fill(hit, u, V, nxt)
        for b in range(B):
            for i in range(K):
                want = -7 if hit[b] else int(Fraction(float(u[b, i])) * V // 1)
                assert nxt[b, i] == want, (V, b, i)
        assert nxt[0, 0] == 0 and nxt[0, 2] == V // 2
        if V <= 1 << 24:  # an fp32 uniform resolves 2^-24: larger vocabularies lose the top ids
            assert nxt[0, 1] == V - 1


def test_backup_fill_is_uniform_over_the_vocabulary():
    """Uniforms on an even grid of n = 64 V points land exactly 64 times on each
    token; random uniforms pass a chi-square test."""
    V = 1000
    n = 64 * V
    u = ((np.arange(n, dtype=np.float64) + 0.5) / n).astype(np.float32).reshape(1, n)
    nxt = np.zeros((1, n), np.int32)
    oracle.backup_fill(np.zeros(1, np.uint8), u, V, nxt)
    np.testing.assert_array_equal(np.bincount(nxt[0], minlength=V), np.full(V, 64))
    rng = np.random.default_rng(8)
    u = rng.random((200, 500)).astype(np.float32)
    nxt = np.zeros((200, 500), np.int32)
    oracle.backup_fill(np.zeros(200, np.uint8), u, V, nxt)
    counts = np.bincount(nxt.ravel(), minlength=V)
    assert scipy.stats.chisquare(counts).pvalue > 1e-4


# ---------------------------------------------------------------------------
# sigma_{F,C} reshape.
# ---------------------------------------------------------------------------

def _brute_topf(z, F):
    order = np.lexsort((np.arange(len(z)), -np.asarray(z, np.float64)))
    return order[:F]


def test_topf_matches_library_sort():
    rng = np.random.default_rng(12)
    for V, F in [(10, 3), (300, 8), (1000, 64), (5000, 1)]:
        z = rng.integers(-5, 5, V).astype(np.float64)  # many ties -> lowest id first
        np.testing.assert_array_equal(oracle.topf(z, F), _brute_topf(z, F))


def test_sigma_special_cases():
    rng = np.random.default_rng(13)
    V, F, tau = 200, 8, 0.7
    z = rng.standard_normal(V) * 3
    S = np.zeros(V, bool)
    S[_brute_topf(z, F)] = True
    # C = 1: plain temperature softmax
    q1, m1 = oracle.sigma(z, tau, F, 1.0)
    np.testing.assert_allclose(q1, scipy.special.softmax(z / tau), rtol=1e-12)
    np.testing.assert_array_equal(m1, S)
    # C = 0: the top-F get zero, the rest renormalised
    q0, _ = oracle.sigma(z, tau, F, 0.0)
    assert (q0[S] == 0).all()
    np.testing.assert_allclose(q0[~S], scipy.special.softmax(z[~S] / tau), rtol=1e-12)
    # general C: ratios C e^{(z_i - z_j)/tau} across the set boundary, plain inside
    C = 0.37
    qc, _ = oracle.sigma(z, tau, F, C)
    assert qc.sum() == pytest.approx(1.0, abs=1e-12)
    i, j = np.nonzero(S)[0][0], np.nonzero(~S)[0][0]
    assert qc[i] / qc[j] == pytest.approx(C * np.exp((z[i] - z[j]) / tau), rel=1e-12)
    i2 = np.nonzero(S)[0][1]
    assert qc[i] / qc[i2] == pytest.approx(np.exp((z[i] - z[i2]) / tau), rel=1e-12)
    # the top-F set does not depend on tau
    _, m2 = oracle.sigma(z, 2.5, F, C)
    np.testing.assert_array_equal(m2, S)
    # lowering C moves mass off the top-F set (monotone)
    mass = [oracle.sigma(z, tau, F, c)[0][S].sum() for c in (1.0, 0.5, 0.1, 0.0)]
    assert all(a > b for a, b in zip(mass, mass[1:]))
    with pytest.raises(ValueError):
        oracle.sigma(z[:5], tau, 5, 0.0)


def test_verify_uses_reshaped_draft():
    rng = np.random.default_rng(14)
    B, K, V, F, C = 32, 3, 40, 4, 0.5
    tau = float(np.float32(0.7))   # the oracle reads the fp32 temperature
    tgt = (rng.standard_normal((B, K + 1, V)) * 2).astype(np.float32)
    drf = (rng.standard_normal((B, K, V)) * 2).astype(np.float32)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K + 1), dtype=np.float32)
    taus = np.full(B, tau, np.float32)
    o = oracle.verify(tgt, drf, x, u, taus, "f32", reshape_F=F, reshape_C=C)
    for b in range(B):
        for i in range(o["accept_len"][b] + (1 if o["accept_len"][b] < K else 0)):
            if i >= K:
                break
            qz = drf[b, i].astype(np.float64)
            S = np.zeros(V, bool)
            S[_brute_topf(qz, F)] = True
            w = np.where(S, C, 1.0) * np.exp(qz / tau - (qz / tau).max())
            assert o["q_tok"][b, i] == pytest.approx(w[x[b, i]] / w.sum(), rel=1e-12)


# ---------------------------------------------------------------------------
# Cache build, lookup and the hit probability.
# ---------------------------------------------------------------------------

def test_cache_build_brute_force():
    rng = np.random.default_rng(15)
    B, K, V, budget = 12, 3, 24, 14
    F, off, _ = oracle.fanout(K, budget, 0.7, 1.0, V)
    tgt = rng.integers(-4, 4, (B, K + 1, V)).astype(np.float32)   # ties on purpose
    drf = rng.integers(-4, 4, (B, K, V)).astype(np.float32)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    tau = np.where(np.arange(B) % 2 == 0, 0.0, 0.9).astype(np.float32)
    c = oracle.build_cache(tgt, drf, x, tau, "f32", off, budget)
    for b in range(B):
        for k in range(K + 1):
            seg = c["cache_tok"][b, off[k]:off[k + 1]]
            if tau[b] == 0:
                score = tgt[b, k].astype(np.float64)
                if k < K:
                    score = score.copy()
                    score[x[b, k]] = -np.inf
                    # the excluded token ranks below every other token
                    order = np.lexsort((np.arange(V), np.where(np.arange(V) == x[b, k], 1, 0),
                                        -np.where(np.isinf(score), 0, score)))
                    order = [t for t in order if t != x[b, k]] + [x[b, k]]
                else:
                    order = _brute_topf(score, V)
            else:
                p = scipy.special.softmax(tgt[b, k].astype(np.float64) / tau[b])
                if k < K:
                    q = scipy.special.softmax(drf[b, k].astype(np.float64) / tau[b])
                    score = np.maximum(p - q, 0.0)
                else:
                    score = p
                order = _brute_topf(score, V)
            np.testing.assert_array_equal(seg, np.asarray(order)[:F[k]])


def test_lookup_semantics():
    off = np.array([0, 2, 2, 5], np.int32)          # K = 2, F = [2, 0, 3]
    cache = np.array([[7, 3, 9, 1, 4], [7, 3, 9, 1, 4], [7, 3, 9, 1, 4], [7, 3, 9, 1, 4],
                      [7, 3, 9, 1, 4]], np.int32)
    a = np.array([0, 0, 1, 2, -1], np.int32)
    t = np.array([3, 9, 7, 4, 7], np.int32)
    h = oracle.lookup(cache, off, a, t)
    np.testing.assert_array_equal(h["hit"], [1, 0, 0, 1, 0])
    np.testing.assert_array_equal(h["slot"], [1, -1, -1, 4, -1])


def test_hit_rate_matches_analytic_p_hit():
    """P_hit = sum_k P(a = k) * sum_{t in S_k} P(t* = t | a = k)  (the accept-length
    distribution weighted by the cached bonus mass), checked by Monte Carlo."""
    rng = np.random.default_rng(16)
    K, V, budget, n = 3, 48, 10, 200_000
    F, off, _ = oracle.fanout(K, budget, 0.7, 0.5, V)
    zp = (rng.standard_normal((K + 1, V)) * 1.5).astype(np.float32)
    zq = (zp[:K] + rng.standard_normal((K, V)) * 0.8).astype(np.float32)
    p = [scipy.special.softmax(zp[i].astype(np.float64)) for i in range(K + 1)]
    q = [scipy.special.softmax(zq[i].astype(np.float64)) for i in range(K)]
    x = np.stack([_sample(rng, q[i], n) for i in range(K)], axis=1)
    u = rng.random((n, K + 1), dtype=np.float32)
    o = oracle.round_(_batch(zp, n), _batch(zq, n), x, u, np.ones(n, np.float32), "f32", off,
                      budget)
    alpha = [np.minimum(p[i], q[i]).sum() for i in range(K)]
    p_a = [np.prod(alpha[:k]) * (1 - alpha[k]) for k in range(K)] + [np.prod(alpha)]
    cache = o["cache_tok"][0]
    analytic = 0.0
    for k in range(K + 1):
        w = np.maximum(p[k] - q[k], 0) if k < K else p[K]
        w = w / w.sum()
        analytic += p_a[k] * w[cache[off[k]:off[k + 1]]].sum()
    emp = o["hit"].mean()
    se = np.sqrt(analytic * (1 - analytic) / n)
    assert abs(emp - analytic) < 4 * se, (emp, analytic)
    # the hit slot indexes the true bonus inside the accepted-length segment
    h = o["hit"].astype(bool)
    assert (o["cache_tok"][h, o["slot"][h]] == o["bonus"][h]).all()
    assert ((o["slot"][h] >= off[o["accept_len"][h]]) & (o["slot"][h] < off[o["accept_len"][h] + 1])).all()
