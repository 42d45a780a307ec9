"""Draft-only cache keys and per-position sigma_{F_k,C} on the GPU (ssd_draft_cache),
against the float64 oracle:

* the cache keys bit for bit (ties, the drafted token at the top of its row,
  F_k = 0, F_k above 64, F_k = V), on aligned and unaligned rows;
* the per-position descriptors, and verification on the q they describe;
* the C sweep: the hit rate of many rounds against the analytic probability
  that the outcome (a, t*) is cached, for C from 1 down to 0.
"""
import numpy as np
import pytest

import oracle
import synth
from tests._parity import Tally, compare_verify, np_out

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


def _rows(rng, B, K, V, dtype, quantise=False):
    z = (rng.standard_normal((B, K + 1, V)) * 2.5).astype(np.float32) \
        + synth.zipf_log_bias(V, 1.1)
    if quantise:
        z = np.round(z * 2).astype(np.float32) / 2
    return synth.store(z, dtype)


def _dev_logits(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if dtype == "bf16" else a)
    t = t.cuda()
    return t.view(torch.bfloat16) if dtype == "bf16" else t


def _check_desc(ssd, desc, drf, F, K, dtype):
    thr_val, thr_id, Fd, _ = ssd.desc_fields(desc)
    thr_val, thr_id, Fd = thr_val.cpu().numpy(), thr_id.cpu().numpy(), Fd.cpu().numpy()
    zs = synth.stored_to_f32(drf, dtype).astype(np.float64)
    B = drf.shape[0]
    for b in range(B):
        for k in range(K):
            r = b * K + k
            assert Fd[r] == F[k]
            if F[k] == 0:
                assert thr_id[r] == -1 and np.isinf(thr_val[r])
                continue
            top = oracle.topf(zs[b, k], F[k])
            assert thr_id[r] == top[-1] and thr_val[r] == zs[b, k, top[-1]], (b, k)


@pytest.mark.parametrize("dtype,V,F", [
    ("bf16", 20000, [8, 6, 5, 4, 9]),
    ("f32", 24011, [11, 0, 7, 3, 13]),          # unaligned rows, an empty segment
    ("bf16", 128256, [90, 70, 40, 30, 120]),     # F_k above 64
    ("f32", 40, [40, 5, 40, 1, 40]),             # F_k = V: a slot left at -1
])
def test_draft_cache_matches_oracle(ssd, dtype, V, F):
    rng = np.random.default_rng(60 + V % 101)
    B, K = 9, 4
    drf = _rows(rng, B, K, V, dtype, quantise=(V == 20000))
    zs = synth.stored_to_f32(drf, dtype)
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    tok[0] = np.argmax(zs[0, :K], axis=-1)                       # drafted token ranked first
    tok[1] = np.argsort(-zs[1, :K], axis=-1, kind="stable")[:, 2]  # ranked third
    off = np.concatenate([[0], np.cumsum(F)]).astype(np.int32)
    budget = int(off[-1]) + 5
    cache = torch.full((B, budget), -7, dtype=torch.int32, device="cuda")
    c, desc = ssd.ssd_draft_cache(_dev_logits(drf, dtype), torch.from_numpy(tok).cuda(), F,
                                  budget, 0.5, cache_tok=cache, reshape=True)
    got = c.cpu().numpy()
    want = oracle.draft_cache(drf, tok, dtype, off, budget)
    np.testing.assert_array_equal(got[:, : off[-1]], want[:, : off[-1]])
    assert (got[:, off[-1]:] == -7).all()
    _check_desc(ssd, desc, drf, F, K, dtype)
    # without drafted tokens nothing is left out
    c2, _ = ssd.ssd_draft_cache(_dev_logits(drf, dtype), None, F, budget)
    np.testing.assert_array_equal(c2.cpu().numpy()[:, : off[-1]],
                                  oracle.draft_cache(drf, None, dtype, off, budget)[:, : off[-1]])


def _sigma_log_bias(drf_f32, F, C):
    """log c_t of sigma_{F_k,C} on each draft row k < K (for drafting from q')."""
    B, K1, V = drf_f32.shape
    K = K1 - 1
    bias = np.zeros((B, K, V), np.float64)
    lc = np.log(C) if C > 0 else -np.inf
    for b in range(B):
        for k in range(K):
            bias[b, k, oracle.topf(drf_f32[b, k].astype(np.float64), F[k])] = lc
    return bias


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_verify_on_per_position_reshape(ssd, dtype):
    rng = np.random.default_rng(61)
    B, K, V = 12, 4, 24000
    F = [8, 6, 5, 4, 9]
    C = 0.3
    drf = _rows(rng, B, K, V, dtype)
    zd = synth.stored_to_f32(drf, dtype)
    zt = zd + rng.standard_normal(zd.shape).astype(np.float32) * 0.8
    tgt = synth.store(zt, dtype)
    tau = np.where(np.arange(B) % 3 == 0, 0.0, 0.8).astype(np.float32)
    tok = synth.sample_draft_tokens(rng, synth.stored_to_f32(drf, dtype)[:, :K], tau,
                                    _sigma_log_bias(zd, F, C))
    u = rng.random((B, K + 1), dtype=np.float32)
    dd = _dev_logits(drf, dtype)
    _, desc = ssd.ssd_draft_cache(dd, torch.from_numpy(tok).cuda(), F, sum(F), C, cache=False,
                                  reshape=True)
    g = np_out(ssd.ssd_verify(_dev_logits(tgt, dtype), dd, torch.from_numpy(tok).cuda(),
                              torch.from_numpy(u).cuda(), torch.from_numpy(tau).cuda(),
                              reshape=desc))
    o = oracle.verify(tgt, drf, tok, u, tau, dtype, reshape_F=F[:K], reshape_C=C)
    t = Tally()
    compare_verify(g, o, K, t)
    t.check()


@pytest.mark.parametrize("C", [1.0, 0.4, 0.0])
def test_c_sweep_hit_rate_tracks_analytic_probability(ssd, C):
    B, K, V, R = 32, 3, 4096, 300
    F = [5, 4, 3, 6]
    off = np.concatenate([[0], np.cumsum(F)]).astype(np.int32)
    budget = int(off[-1])
    rng = np.random.default_rng(62)
    drf = _rows(rng, B, K, V, "f32")
    zd = drf
    tgt = (zd + rng.standard_normal(zd.shape).astype(np.float32) * 0.7).astype(np.float32)
    tau = np.ones(B, np.float32)
    tok = synth.sample_draft_tokens(rng, zd[:, :K], tau, _sigma_log_bias(zd, F, C))
    dt, dd = torch.from_numpy(tgt).cuda(), torch.from_numpy(drf).cuda()
    tk = torch.from_numpy(tok).cuda()
    cache, desc = ssd.ssd_draft_cache(dd, tk, F, budget, C, reshape=True)
    want = oracle.draft_cache(drf, tok, "f32", off, budget)
    np.testing.assert_array_equal(cache.cpu().numpy(), want)
    P = oracle.p_hit(tgt, drf, tok, tau, "f32", off, budget, want, reshape_F=F[:K], reshape_C=C)
    U = torch.from_numpy(rng.random((R, B, K + 1), dtype=np.float32)).cuda()
    td = torch.from_numpy(tau).cuda()
    hits = []
    for r in range(R):
        v = ssd.ssd_verify(dt, dd, tk, U[r].contiguous(), td, reshape=desc, probs=False)
        h, _ = ssd.ssd_cache_lookup(cache, F, v["accept_len"], v["bonus"])
        hits.append(h)
    H = torch.stack(hits).cpu().numpy().astype(bool)
    n = H.sum()
    mean, sd = R * P.sum(), np.sqrt(R * (P * (1 - P)).sum())
    assert abs(n - mean) < 4 * sd + 1, (C, n, mean, sd)
