"""The cache-miss side of a Saguaro round on the GPU, against the float64 oracle:

* the fast random-token backup (ssd_backup_fill) bit for bit, on its own and on
  the hit mask a round produced;
* a round whose cache uses the uniform fan-out instead of the geometric one;
* the hit rate of many rounds, for both fan-out shapes, against the analytic
  probability that the true outcome (a, t*) is cached, and the rate at which a
  whole group of b sequences hits against the product of their probabilities.
"""
import numpy as np
import pytest

import oracle
import synth
from tests._parity import Tally, compare_cache, compare_verify, lookup_from, np_out, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ssd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_ssd_gb300 as m
    from speculative_decoding_verification_ssd_gb300 import _build
    _build.build()
    return m


@pytest.mark.parametrize("V", [1, 2, 7, 128256, 152064, (1 << 24) + 3])
def test_backup_fill_matches_oracle(ssd, V):
    rng = np.random.default_rng(40 + V % 97)
    B, K = 1037, 8                       # several blocks and a ragged tail
    u = rng.random((B, K)).astype(np.float32)
    below1 = np.nextafter(np.float32(1), np.float32(0))
    u[0] = [0.0, below1, 0.5, 0.25, np.float32(1.0 / 3.0), 1e-30, 0.75, below1]
    # uniforms sitting on and just below the token boundaries t / V
    t = rng.integers(0, V, K)
    edge = (t / V).astype(np.float32)
    u[1] = edge
    u[2] = np.nextafter(edge, np.float32(0))
    hit = (rng.random(B) < 0.3).astype(np.uint8)
    hit[:3] = 0
    prev = rng.integers(-5, V, (B, K)).astype(np.int32)
    want = prev.copy()
    oracle.backup_fill(hit, u, V, want)
    got = ssd.ssd_backup_fill(torch.from_numpy(hit).cuda(), torch.from_numpy(u).cuda(), V,
                              torch.from_numpy(prev).cuda())
    np.testing.assert_array_equal(got.cpu().numpy(), want)


def test_backup_fill_on_a_round_hit_mask(ssd):
    """The round's own hit output drives the backup on the same stream: missed sequences
    get floor(u V), sequences that hit keep what the caller wrote there."""
    wl = synth.WORKLOADS["c4"].replace(B=24, V=20000)
    inp = synth.make_inputs(wl, 4101)
    F, off = ssd.ssd_fanout(wl.K, wl.budget, wl.a_p, wl.r, wl.V)
    d = to_device(inp)
    g = ssd.ssd_round(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"], F,
                      wl.budget)
    rng = np.random.default_rng(4102)
    u_next = rng.random((wl.B, wl.K)).astype(np.float32)
    prev = np.full((wl.B, wl.K), -1, np.int32)
    nxt = ssd.ssd_backup_fill(g["hit"], torch.from_numpy(u_next).cuda(), wl.V,
                              torch.from_numpy(prev).cuda()).cpu().numpy()
    o = oracle.round_(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"], inp["temperature"],
                      wl.dtype, off, wl.budget)
    hit = g["hit"].cpu().numpy()
    np.testing.assert_array_equal(hit, o["hit"])
    want = prev.copy()
    oracle.backup_fill(hit, u_next, wl.V, want)
    np.testing.assert_array_equal(nxt, want)
    assert 0 < hit.sum() < wl.B  # both branches taken


@pytest.mark.parametrize("dtype,V", [("f32", 24000), ("bf16", 24000), ("f32", 20011)])
def test_uniform_fanout_round_matches_oracle(ssd, dtype, V):
    wl = synth.WORKLOADS["c5"].replace(B=20, V=V, dtype=dtype, greedy_first=6)
    inp = synth.make_inputs(wl, 4200 + V % 13)
    F, off = ssd.ssd_fanout_uniform(wl.K, wl.budget, V)
    d = to_device(inp)
    g = np_out(ssd.ssd_round(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"], F,
                             wl.budget))
    o = oracle.round_(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"], inp["temperature"],
                      dtype, off, wl.budget)
    t = Tally()
    compare_verify(g, o, wl.K, t)
    compare_cache(g["cache_tok"], o, off, wl.K, t)
    h, s = lookup_from(g["cache_tok"], off, g["accept_len"], g["bonus"])
    np.testing.assert_array_equal(g["hit"], h)
    np.testing.assert_array_equal(g["slot"], s)
    t.check()


def _analytic_p_hit(inp, o, off, K):
    """P(true outcome cached | drafted tokens) per sequence: accept position i with
    probability min(1, p_i(x_i) / q_i(x_i)); a rejection at k draws the bonus from
    (p_k - q_k)^+, acceptance of all K from p_K; the outcome hits when that bonus is
    among the cached keys of its accepted length."""
    zt = synth.stored_to_f32(inp["tgt"], "f32").astype(np.float64)
    zd = synth.stored_to_f32(inp["drf"], "f32").astype(np.float64)
    B = zt.shape[0]
    out = np.empty(B)
    for b in range(B):
        tau = float(inp["temperature"][b])
        p = [oracle.softmax(zt[b, i], tau) for i in range(K + 1)]
        q = [oracle.softmax(zd[b, i], tau) for i in range(K)]
        x = inp["tokens"][b]
        acc = [min(1.0, p[i][x[i]] / q[i][x[i]]) for i in range(K)]
        total, reach = 0.0, 1.0
        for k in range(K + 1):
            if k < K:
                pa = reach * (1.0 - acc[k])
                w = np.maximum(p[k] - q[k], 0.0)
            else:
                pa = reach
                w = p[K]
            if pa > 0 and w.sum() > 0:
                keys = o["cache_tok"][b, off[k]:off[k + 1]]
                total += pa * w[keys].sum() / w.sum()
            if k < K:
                reach *= acc[k]
        out[b] = total
    return out


@pytest.mark.parametrize("shape", ["geometric", "uniform"])
def test_hit_rate_tracks_analytic_probability(ssd, shape):
    B, K, V, budget, R = 32, 3, 4096, 12, 400
    wl = synth.Workload("hits", B=B, K=K, V=V, dtype="f32", sigma_d=2.0, zipf_s=1.1,
                        sigma_n=0.6, tau=1.0, budget=budget, a_p=0.7, r=0.5, mode="round")
    inp = synth.make_inputs(wl, 4300)
    F, off = (ssd.ssd_fanout(K, budget, wl.a_p, wl.r, V) if shape == "geometric"
              else ssd.ssd_fanout_uniform(K, budget, V))
    o = oracle.round_(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"], inp["temperature"],
                      "f32", off, budget)
    P = _analytic_p_hit(inp, o, off, K)
    d = to_device(inp)
    rng = np.random.default_rng(4301)
    U = torch.from_numpy(rng.random((R, B, K + 1), dtype=np.float32)).cuda()
    hits = []
    for r in range(R):
        g = ssd.ssd_round(d["tgt"], d["drf"], d["tokens"], U[r].contiguous(), d["temperature"], F,
                          budget, probs=False)
        hits.append(g["hit"])
    H = torch.stack(hits).cpu().numpy().astype(bool)            # [R, B]
    n = H.sum()
    mean, sd = R * P.sum(), np.sqrt(R * (P * (1 - P)).sum())
    assert abs(n - mean) < 4 * sd + 1, (shape, n, mean, sd)
    # all four sequences of a group hit: probability = product of their P
    Pg = P.reshape(B // 4, 4).prod(axis=1)
    ng = H.reshape(R, B // 4, 4).all(axis=2).sum()
    mean_g, sd_g = R * Pg.sum(), np.sqrt(R * (Pg * (1 - Pg)).sum())
    assert abs(ng - mean_g) < 4 * sd_g + 1, (shape, ng, mean_g, sd_g)
