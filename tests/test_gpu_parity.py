"""GPU parity: libssd (through its C ABI) against the float64 oracle on seeded inputs.

Sizes: the workloads' own shapes (full vocabularies, so every row spans many
CTA slices; V = 128256 and 152064 are not multiples of the slice so the last
slice is ragged), with the batch reduced where the oracle needs it, plus the
full batch of the benchmark's round workload in the launch configuration the
benchmark times.
"""
import numpy as np
import pytest

import oracle
import synth
from tests._parity import (Tally, compare_cache, compare_verify, lookup_from, np_out, to_device,
                           use_dispatch)

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


def _reduced(name, B, **kw):
    wl = synth.WORKLOADS[name]
    g = wl.greedy_first * B // wl.B if wl.greedy_first else 0
    return wl.replace(B=B, greedy_first=g, **kw)


def _oracle_verify(inp, wl):
    return oracle.verify(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"],
                         inp["temperature"], wl.dtype, wl.reshape_F, wl.reshape_C)


def _run_verify(ssd, inp, reshape=None):
    d = to_device(inp)
    out = ssd.ssd_verify(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"],
                         reshape=reshape)
    torch.cuda.synchronize()
    return np_out(out)


@pytest.mark.parametrize("policy", [1, 2, 3, 4])  # streaming, cluster, slice kernel, wide streaming
@pytest.mark.parametrize("name,B,seed_off", [("c1", 1, 0), ("c1", 64, 1), ("c2", 8, 0),
                                             ("c2", 24, 1)])
def test_verify_parity(ssd, name, B, seed_off, policy):
    wl = _reduced(name, B)
    inp = synth.make_inputs(wl, synth.PARITY_SEED[name] + 100 * seed_off)
    with use_dispatch(ssd, policy):
        g = _run_verify(ssd, inp)
        assert ssd.ssd_last_kernel() == {1: "stream", 2: "cluster", 3: "slice", 4: "stream-wide"}[policy]
    o = _oracle_verify(inp, wl)
    t = Tally()
    compare_verify(g, o, wl.K, t)
    t.check()


def test_verify_reshaped_parity(ssd):
    """sigma_{F,C}-reshaped drafting (F=8, C=0.5, tau=0.7): descriptors from the GPU
    reshape kernel feed the verify kernel; the oracle reshapes on its own."""
    wl = _reduced("c3", 12)
    F, C = wl.reshape_F, wl.reshape_C

    def bias(drf_f32):
        out = np.zeros(drf_f32.shape, np.float64)
        for b in range(drf_f32.shape[0]):
            for i in range(drf_f32.shape[1]):
                out[b, i, oracle.topf(drf_f32[b, i].astype(np.float64), F)] = np.log(C)
        return out

    inp = synth.make_inputs(wl, synth.PARITY_SEED["c3"], draft_log_bias=bias)
    d = to_device(inp)
    tau_rows = d["temperature"].repeat_interleave(wl.K)
    desc, q = ssd.ssd_reshape_draft(d["drf"], F, C, tau_rows, want_q=True)
    out = ssd.ssd_verify(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"],
                         reshape=desc)
    torch.cuda.synchronize()
    g = np_out(out)
    o = _oracle_verify(inp, wl)
    t = Tally()
    compare_verify(g, o, wl.K, t)
    t.check()
    # descriptors: the F-th largest raw logit (value and id) of each draft row
    thr_val, thr_id, Fd, Cd = [x.cpu().numpy() for x in ssd.desc_fields(desc)]
    drf32 = synth.stored_to_f32(inp["drf"], wl.dtype).reshape(-1, wl.V)
    taus = np.repeat(inp["temperature"], wl.K)
    ro = oracle.reshape_rows(inp["drf"].reshape(-1, wl.V), taus, wl.dtype, F, C)
    for r in range(drf32.shape[0]):
        ids = oracle.topf(drf32[r].astype(np.float64), F)
        assert thr_id[r] == ids[-1] and thr_val[r] == drf32[r, ids[-1]]
        assert Fd[r] == F and Cd[r] == np.float32(C)
        np.testing.assert_array_equal(ro["member"][r], np.isin(np.arange(wl.V), ids))
    qg = q.cpu().numpy()
    err = np.abs(qg - ro["q"]).max()
    assert err <= 1e-5, err


@pytest.mark.parametrize("policy", [1, 2, 3, 4])  # streaming, cluster, slice kernel, wide streaming
@pytest.mark.parametrize("name,B", [("c4", 6), ("c5", 32)])
def test_round_parity(ssd, name, B, policy):
    wl = _reduced(name, B)
    inp = synth.make_inputs(wl, synth.PARITY_SEED[name])
    F, off = ssd.ssd_fanout(wl.K, wl.budget, wl.a_p, wl.r, wl.V)
    Fo, offo, _ = oracle.fanout(wl.K, wl.budget, wl.a_p, wl.r, wl.V)
    np.testing.assert_array_equal(F, Fo)
    d = to_device(inp)
    with use_dispatch(ssd, policy):
        out = ssd.ssd_round(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"], F,
                            wl.budget)
        assert ssd.ssd_last_kernel() == {1: "stream", 2: "cluster", 3: "slice", 4: "stream-wide"}[policy]
    torch.cuda.synchronize()
    g = np_out(out)
    o = oracle.round_(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"],
                      inp["temperature"], wl.dtype, off, wl.budget)
    t = Tally()
    compare_verify(g, o, wl.K, t)
    compare_cache(g["cache_tok"], o, off, wl.K, t)
    h, s = lookup_from(g["cache_tok"], off, g["accept_len"], g["bonus"])
    np.testing.assert_array_equal(g["hit"], h)
    np.testing.assert_array_equal(g["slot"], s)
    same = (g["accept_len"] == o["accept_len"]) & (g["bonus"] == o["bonus"])
    np.testing.assert_array_equal(g["hit"][same], o["hit"][same])
    t.check()


def test_round_full_batch_bench_config(ssd):
    """The benchmark's workload at full size (B=256, K=4, V=128256 bf16, half greedy)
    in the same launch configuration: every sequence compared with the oracle."""
    wl = synth.WORKLOADS["c5"]
    inp = synth.make_inputs(wl, synth.PARITY_SEED["c5"])
    F, off = ssd.ssd_fanout(wl.K, wl.budget, wl.a_p, wl.r, wl.V)
    d = to_device(inp)
    ws = ssd.workspace(wl.B, wl.K)
    g = None
    for _ in range(2):  # second call reuses the workspace (counters reset by the epilogue)
        out = ssd.ssd_round(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"], F,
                            wl.budget, workspace=ws)
        torch.cuda.synchronize()
        g2 = np_out(out)
        if g is not None:
            for key in ("accept_len", "bonus", "cache_tok", "hit", "slot"):
                np.testing.assert_array_equal(g[key], g2[key])
        g = g2
    o = oracle.round_(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"],
                      inp["temperature"], wl.dtype, off, wl.budget)
    t = Tally()
    compare_verify(g, o, wl.K, t)
    compare_cache(g["cache_tok"], o, off, wl.K, t)
    h, s = lookup_from(g["cache_tok"], off, g["accept_len"], g["bonus"])
    np.testing.assert_array_equal(g["hit"], h)
    np.testing.assert_array_equal(g["slot"], s)
    t.check()


def test_build_cache_and_lookup_match_round(ssd):
    wl = _reduced("c5", 16)
    inp = synth.make_inputs(wl, synth.PARITY_SEED["c5"] + 7)
    F, off = ssd.ssd_fanout(wl.K, wl.budget, wl.a_p, wl.r, wl.V)
    d = to_device(inp)
    r = ssd.ssd_round(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"], F, wl.budget)
    c = ssd.ssd_build_cache(d["tgt"], d["drf"], d["tokens"], d["temperature"], F, wl.budget)
    v = ssd.ssd_verify(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"])
    hit, slot = ssd.ssd_cache_lookup(c, F, v["accept_len"], v["bonus"])
    torch.cuda.synchronize()
    np.testing.assert_array_equal(r["cache_tok"].cpu().numpy(), c.cpu().numpy())
    np.testing.assert_array_equal(r["accept_len"].cpu().numpy(), v["accept_len"].cpu().numpy())
    np.testing.assert_array_equal(r["bonus"].cpu().numpy(), v["bonus"].cpu().numpy())
    np.testing.assert_array_equal(r["hit"].cpu().numpy(), hit.cpu().numpy())
    np.testing.assert_array_equal(r["slot"].cpu().numpy(), slot.cpu().numpy())
