"""sigma_{F_k,C} found in the verification pass (ssd_verify_sigma / ssd_round_sigma)
against the float64 oracle on the reshaped draft:

* verification with C = 1, 0.5, 0.05 and 0 (the last two on rows whose top-F_k
  tokens hold nearly all of the mass, where the normaliser is summed afresh);
* the descriptors it returns against ssd_draft_cache's;
* a full round (cache keys ranked on the reshaped residual);
* unaligned rows, which find the descriptors in a separate pass first;
* F_k = 256, where the selection starts from every group.
"""
import numpy as np
import pytest

import oracle
import synth
from tests._parity import Tally, compare_cache, compare_verify, lookup_from, np_out, use_dispatch

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", params=["default", "wide"])
def ssd(request):
    """The library under its default kernel choice, and with the streaming kernel's
    wide form forced (both consumer groups of a CTA on each unit)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_ssd_gb300 as m
    from speculative_decoding_verification_ssd_gb300 import _build
    _build.build()
    policy = m.SSD_DISPATCH_AUTO if request.param == "default" else m.SSD_DISPATCH_WIDE
    with use_dispatch(m, policy):
        yield m


def _dev_logits(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if dtype == "bf16" else a)
    t = t.cuda()
    return t.view(torch.bfloat16) if dtype == "bf16" else t


def _sigma_log_bias(zd, F, C):
    B, K, V = zd.shape
    bias = np.zeros((B, K, V), np.float64)
    lc = np.log(C) if C > 0 else -np.inf
    for b in range(B):
        for k in range(K):
            if F[k] > 0:
                bias[b, k, oracle.topf(zd[b, k].astype(np.float64), F[k])] = lc
    return bias


def _problem(seed, B, K, V, dtype, F, C, peaked=False, taus=None):
    rng = np.random.default_rng(seed)
    zd = (rng.standard_normal((B, K + 1, V)) * 2.0).astype(np.float32) + synth.zipf_log_bias(V, 1.1)
    if peaked:
        for b in range(B):
            for k in range(K):
                zd[b, k, rng.choice(V, max(F[k], 1), replace=False)] += 14.0
    zt = zd + (rng.standard_normal(zd.shape) * 0.8).astype(np.float32)
    drf = synth.store(zd[:, :K], dtype)
    tgt = synth.store(zt, dtype)
    tau = np.asarray(taus if taus is not None else [0.7] * B, np.float32)
    zds = synth.stored_to_f32(drf, dtype)
    tok = synth.sample_draft_tokens(rng, zds, tau, _sigma_log_bias(zds, F, C))
    u = rng.random((B, K + 1), dtype=np.float32)
    return tgt, drf, tok, u, tau


@pytest.mark.parametrize("dtype,V,C,peaked", [
    ("bf16", 24000, 0.5, False),
    ("f32", 24000, 1.0, False),
    ("bf16", 24000, 0.05, True),
    ("f32", 24000, 0.0, True),
    ("bf16", 128256, 0.5, False),
])
def test_verify_sigma_matches_oracle(ssd, dtype, V, C, peaked):
    B, K = 12, 4
    F = [8, 6, 0, 5]
    taus = [0.7, 1.0, 0.0, 0.7] * 3
    tgt, drf, tok, u, tau = _problem(70 + int(C * 100), B, K, V, dtype, F, C, peaked, taus)
    dd = _dev_logits(drf, dtype)
    g = ssd.ssd_verify_sigma(_dev_logits(tgt, dtype), dd, torch.from_numpy(tok).cuda(),
                             torch.from_numpy(u).cuda(), torch.from_numpy(tau).cuda(), F, C)
    desc = g.pop("desc")
    gn = np_out(g)
    o = oracle.verify(tgt, drf, tok, u, tau, dtype, reshape_F=F, reshape_C=C)
    t = Tally()
    compare_verify(gn, o, K, t)
    t.check()
    # the descriptors of the sampled sequences' verified positions (up to the accepted
    # length; later ones may be skipped) equal the draft side's
    pad = np.concatenate([drf, drf[:, :1]], axis=1)  # a row K for ssd_draft_cache's layout
    _, ref = ssd.ssd_draft_cache(_dev_logits(pad, dtype), None, F + [0], sum(F), C, cache=False,
                                 reshape=True)
    got, want = desc.cpu().numpy().reshape(B, K, 4), ref.cpu().numpy().reshape(B, K, 4)
    verified = (tau > 0)[:, None] & (np.arange(K)[None, :] <= gn["accept_len"][:, None])
    np.testing.assert_array_equal(got[verified], want[verified])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_round_sigma_matches_oracle(ssd, dtype):
    B, K, V = 10, 4, 24000
    Fc = [8, 6, 5, 4, 9]
    C = 0.5
    tgt, drf, tok, u, tau = _problem(80, B, K, V, dtype, Fc[:K], C,
                                     taus=[0.7, 1.0, 0.0, 0.7, 1.0] * 2)
    budget = sum(Fc)
    off = np.concatenate([[0], np.cumsum(Fc)]).astype(np.int32)
    g = np_out(ssd.ssd_round_sigma(_dev_logits(tgt, dtype), _dev_logits(drf, dtype),
                                   torch.from_numpy(tok).cuda(), torch.from_numpy(u).cuda(),
                                   torch.from_numpy(tau).cuda(), Fc[:K], C, Fc, budget))
    o = oracle.round_(tgt, drf, tok, u, tau, dtype, off, budget, reshape_F=Fc[:K], reshape_C=C)
    t = Tally()
    compare_verify(g, o, K, t)
    compare_cache(g["cache_tok"], o, off, K, t)
    h, s = lookup_from(g["cache_tok"], off, g["accept_len"], g["bonus"])
    np.testing.assert_array_equal(g["hit"], h)
    np.testing.assert_array_equal(g["slot"], s)
    t.check()


def test_unaligned_rows_find_descriptors_first(ssd):
    B, K, V = 8, 3, 20011                   # f32 rows off the 16-byte grid
    F, C = [7, 3, 5], 0.3
    tgt, drf, tok, u, tau = _problem(90, B, K, V, "f32", F, C, taus=[0.8, 0.0] * 4)
    g = ssd.ssd_verify_sigma(torch.from_numpy(tgt).cuda(), torch.from_numpy(drf).cuda(),
                             torch.from_numpy(tok).cuda(), torch.from_numpy(u).cuda(),
                             torch.from_numpy(tau).cuda(), F, C)
    g.pop("desc")
    o = oracle.verify(tgt, drf, tok, u, tau, "f32", reshape_F=F, reshape_C=C)
    t = Tally()
    compare_verify(np_out(g), o, K, t)
    t.check()


def test_f_256_starts_from_every_group(ssd):
    B, K, V = 4, 2, 24000
    F, C = [256, 200], 0.4
    tgt, drf, tok, u, tau = _problem(91, B, K, V, "bf16", F, C, taus=[0.7] * B)
    g = ssd.ssd_verify_sigma(_dev_logits(tgt, "bf16"), _dev_logits(drf, "bf16"),
                             torch.from_numpy(tok).cuda(), torch.from_numpy(u).cuda(),
                             torch.from_numpy(tau).cuda(), F, C)
    g.pop("desc")
    o = oracle.verify(tgt, drf, tok, u, tau, "bf16", reshape_F=F, reshape_C=C)
    t = Tally()
    compare_verify(np_out(g), o, K, t)
    t.check()


def test_sigma_argument_checks(ssd):
    B, K, V = 2, 2, 64
    z = torch.zeros((B, K + 1, V), dtype=torch.float32, device="cuda")
    d = torch.zeros((B, K, V), dtype=torch.float32, device="cuda")
    tok = torch.zeros((B, K), dtype=torch.int32, device="cuda")
    u = torch.zeros((B, K + 1), dtype=torch.float32, device="cuda")
    tau = torch.ones(B, dtype=torch.float32, device="cuda")
    for F, C in [([3, 65], 0.5), ([3, -1], 0.5), ([3, 3], 1.5), ([64, 3], 0.0)]:
        with pytest.raises(ssd.SSDError) as e:
            ssd.ssd_verify_sigma(z, d, tok, u, tau, F, C)
        assert e.value.status == ssd.SSD_ERR_INVALID_ARG
