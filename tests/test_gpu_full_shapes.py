"""GPU parity at the full shapes of the two workloads the other parity tests only
run with a reduced batch:

* B = 64, K = 8, V = 128256 bf16 logits, tau = 0.7, drafts drawn from
  sigma_{F,C} (F = 8, C = 0.5): verification on the reshaped q, both with the
  descriptors found in the verification pass (ssd_verify_sigma, under either
  kernel choice) and with a separate reshape pass (ssd_reshape_draft, then
  ssd_verify on its descriptors);
* B = 32, K = 6, V = 152064 fp32 logits, cache budget 64 with the geometric
  fan-out a_p = 0.8, r = 1: the fused round under either kernel choice (224
  units: the streaming kernel's own unit count, order and workspace size).

Every sequence is compared with the float64 oracle; the standalone hit-lookup
kernel is compared with the oracle's lookup on the same cache and outcomes.
"""
import numpy as np
import pytest

import oracle
import synth
from tests._parity import Tally, compare_cache, compare_verify, lookup_from, np_out, to_device, \
    use_dispatch

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


@pytest.fixture(scope="module")
def sigma_case():
    """The sigma-reshaped verification workload at its own shape, drafts drawn from
    sigma_{F,C} of each stored draft row, and the oracle's verification of it."""
    wl = synth.WORKLOADS["c3"]
    F, C = wl.reshape_F, wl.reshape_C

    def bias(drf_f32):
        out = np.zeros(drf_f32.shape, np.float64)
        for b in range(drf_f32.shape[0]):
            for i in range(drf_f32.shape[1]):
                out[b, i, oracle.topf(drf_f32[b, i].astype(np.float64), F)] = np.log(C)
        return out

    inp = synth.make_inputs(wl, synth.PARITY_SEED["c3"] + 50, draft_log_bias=bias)
    o = oracle.verify(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"],
                      inp["temperature"], wl.dtype, F, C)
    assert o["invalid"] == 0
    return wl, inp, o


@pytest.mark.parametrize("policy", [1, 2, 4])  # streaming kernel, cluster kernel, wide streaming
def test_sigma_verify_full_shape(ssd, sigma_case, policy):
    wl, inp, o = sigma_case
    d = to_device(inp)
    with use_dispatch(ssd, policy):
        g = ssd.ssd_verify_sigma(d["tgt"], d["drf"], d["tokens"], d["uniforms"],
                                 d["temperature"], [wl.reshape_F] * wl.K, wl.reshape_C)
        torch.cuda.synchronize()
    desc = g.pop("desc")
    gn = np_out(g)
    t = Tally()
    compare_verify(gn, o, wl.K, t)
    t.check()
    # descriptors: the F-th largest raw logit (value, id) of every verified draft row
    # (positions after the accepted length may be skipped, their entries untouched)
    thr_val, thr_id, Fd, _ = [x.cpu().numpy().reshape(-1) for x in ssd.desc_fields(desc)]
    drf32 = synth.stored_to_f32(inp["drf"], wl.dtype).reshape(-1, wl.V)
    a = gn["accept_len"]
    verified = np.array([r for r in range(drf32.shape[0]) if r % wl.K <= a[r // wl.K]])
    rows = np.random.default_rng(3).choice(verified, min(48, len(verified)), replace=False)
    for r in rows:
        ids = oracle.topf(drf32[r].astype(np.float64), wl.reshape_F)
        assert thr_id[r] == ids[-1] and thr_val[r] == drf32[r, ids[-1]]
        assert Fd[r] == wl.reshape_F


@pytest.mark.parametrize("policy", [0, 4])  # default choice, wide streaming
def test_sigma_two_pass_full_shape(ssd, sigma_case, policy):
    wl, inp, o = sigma_case
    d = to_device(inp)
    tau_rows = d["temperature"].repeat_interleave(wl.K)
    desc, _ = ssd.ssd_reshape_draft(d["drf"], wl.reshape_F, wl.reshape_C, tau_rows)
    with use_dispatch(ssd, policy):
        g = ssd.ssd_verify(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"],
                           reshape=desc)
        torch.cuda.synchronize()
    t = Tally()
    compare_verify(np_out(g), o, wl.K, t)
    t.check()


@pytest.fixture(scope="module")
def round_case():
    wl = synth.WORKLOADS["c4"]
    inp = synth.make_inputs(wl, synth.PARITY_SEED["c4"] + 50)
    Fo, off, _ = oracle.fanout(wl.K, wl.budget, wl.a_p, wl.r, wl.V)
    o = oracle.round_(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"],
                      inp["temperature"], wl.dtype, off, wl.budget)
    assert o["invalid"] == 0
    return wl, inp, Fo, off, o


@pytest.mark.parametrize("policy", [1, 2, 3, 4])  # streaming, cluster, slice kernel, wide streaming
def test_round_full_shape_fp32(ssd, round_case, policy):
    wl, inp, Fo, off, o = round_case
    F, off_g = ssd.ssd_fanout(wl.K, wl.budget, wl.a_p, wl.r, wl.V)
    np.testing.assert_array_equal(F, Fo)
    np.testing.assert_array_equal(off_g, off)
    d = to_device(inp)
    with use_dispatch(ssd, policy):
        out = ssd.ssd_round(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"],
                            F, wl.budget)
        assert ssd.ssd_last_kernel() == {1: "stream", 2: "cluster", 3: "slice", 4: "stream-wide"}[policy]
        torch.cuda.synchronize()
    g = np_out(out)
    t = Tally()
    compare_verify(g, o, wl.K, t)
    compare_cache(g["cache_tok"], o, off, wl.K, t)
    h, s = lookup_from(g["cache_tok"], off, g["accept_len"], g["bonus"])
    np.testing.assert_array_equal(g["hit"], h)
    np.testing.assert_array_equal(g["slot"], s)
    same = (g["accept_len"] == o["accept_len"]) & (g["bonus"] == o["bonus"])
    np.testing.assert_array_equal(g["hit"][same], o["hit"][same])
    t.check()


def test_standalone_lookup_matches_oracle(ssd):
    """ssd_cache_lookup against the oracle's lookup on caches with repeated tokens,
    empty segments, outcomes of every length, invalid sequences (a = -1) and bonus
    tokens inside and outside the cache."""
    rng = np.random.default_rng(77)
    K, B, V = 5, 3000, 10
    F = np.array([4, 0, 3, 7, 1, 6], np.int32)
    off = np.concatenate([[0], np.cumsum(F)]).astype(np.int32)
    budget = int(off[-1]) + 3                       # slots past the last segment: never read
    cache = rng.integers(0, V, (B, budget)).astype(np.int32)
    a = rng.integers(-1, K + 1, B).astype(np.int32)
    t = rng.integers(0, V, B).astype(np.int32)
    hit, slot = ssd.ssd_cache_lookup(torch.from_numpy(cache).cuda(), F,
                                     torch.from_numpy(a).cuda(), torch.from_numpy(t).cuda())
    torch.cuda.synchronize()
    want = oracle.lookup(cache, off, a, t)
    np.testing.assert_array_equal(hit.cpu().numpy(), want["hit"])
    np.testing.assert_array_equal(slot.cpu().numpy(), want["slot"])
    assert 0.1 < want["hit"].mean() < 0.9
