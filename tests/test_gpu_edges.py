"""GPU edge cases: tiny and ragged vocabularies, ties, empty cache segments,
misaligned base pointers, draft tensors with K+1 rows, invalid inputs, the
lossless property measured on the GPU, and run-to-run determinism."""
import numpy as np
import pytest
import scipy.stats

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


def _inputs(rng, B, K, V, dtype, taus, integer=False, drf_rows=None):
    drf_rows = drf_rows or K
    if integer:  # many exact ties
        zt = rng.integers(-4, 5, (B, K + 1, V)).astype(np.float32)
        zd = rng.integers(-4, 5, (B, drf_rows, V)).astype(np.float32)
    else:
        zt = (rng.standard_normal((B, K + 1, V)) * 2.5).astype(np.float32)
        zd = (zt[:, :drf_rows] + rng.standard_normal((B, drf_rows, V)) * 0.8).astype(np.float32) \
            if drf_rows <= K + 1 else None
    wl = synth.Workload("edge", B=B, K=K, V=V, dtype=dtype, sigma_d=0, zipf_s=0, sigma_n=0, tau=1.0)
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    # make about half the drafted tokens the draft argmax so acceptances happen
    am = np.argmax(zd[:, :K], axis=-1)
    tok = np.where(rng.random((B, K)) < 0.5, am, tok).astype(np.int32)
    return {"tgt": synth.store(zt, dtype), "drf": synth.store(zd, dtype), "tokens": tok,
            "uniforms": rng.random((B, K + 1), dtype=np.float32),
            "temperature": np.asarray(taus, np.float32), "workload": wl}


@pytest.mark.parametrize("V", [2, 3, 8, 33, 257, 1000, 4099, 40961])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K", [1, 3])
def test_small_and_ragged_vocab(ssd, V, dtype, K):
    rng = np.random.default_rng(V * 10 + K + (dtype == "bf16"))
    B = 16
    taus = [0.0, 0.5, 1.0, 2.0] * (B // 4)
    inp = _inputs(rng, B, K, V, dtype, taus, integer=(V % 2 == 1))
    budget = 7
    F, off = ssd.ssd_fanout(K, budget, 0.7, 0.5, V)
    Fo, offo, _ = oracle.fanout(K, budget, 0.7, 0.5, V)
    np.testing.assert_array_equal(F, Fo)
    d = to_device(inp)
    g = np_out(ssd.ssd_round(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"], F,
                             budget))
    gv = np_out(ssd.ssd_verify(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"]))
    o = oracle.round_(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"], inp["temperature"],
                      dtype, off, budget)
    t = Tally()
    compare_verify(g, o, K, t)
    compare_verify(gv, o, K, t)
    compare_cache(g["cache_tok"], o, off, K, t)
    h, s = lookup_from(g["cache_tok"], off, g["accept_len"], g["bonus"])
    np.testing.assert_array_equal(g["hit"], h)
    np.testing.assert_array_equal(g["slot"], s)
    t.check()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_misaligned_pointers_and_draft_stride(ssd, dtype):
    """Row bases off the 16-byte grid (tensor views starting one element into an
    allocation) and a draft tensor with K+1 rows per sequence."""
    rng = np.random.default_rng(77)
    B, K, V = 6, 3, 5003
    inp = _inputs(rng, B, K, V, dtype, [1.0, 0.0, 0.7] * 2, drf_rows=K + 1)
    d = to_device(inp)

    def shifted(t):
        flat = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
        flat[1:] = t.reshape(-1)
        return flat[1:].view(t.shape)

    tgt, drf = shifted(d["tgt"]), shifted(d["drf"])
    assert tgt.data_ptr() % 16 != 0
    budget = 9
    F, off = ssd.ssd_fanout(K, budget, 0.6, 1.0, V)
    g = np_out(ssd.ssd_round(tgt, drf, d["tokens"], d["uniforms"], d["temperature"], F, budget))
    o = oracle.round_(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"], inp["temperature"],
                      dtype, off, budget)
    t = Tally()
    compare_verify(g, o, K, t)
    compare_cache(g["cache_tok"], o, off, K, t)
    t.check()


def test_invalid_sequences_are_flagged(ssd):
    rng = np.random.default_rng(5)
    B, K, V = 8, 3, 3000
    inp = _inputs(rng, B, K, V, "f32", [1.0] * B)
    inp["tokens"][1, 2] = V          # out of range
    inp["tokens"][2, 0] = -3
    inp["temperature"][3] = -1.0
    inp["temperature"][4] = np.nan
    d = to_device(inp)
    d["tgt"][5, 0, 17] = float("nan")  # non-finite logits in a sampled row read by the round
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    F, off = ssd.ssd_fanout(K, 8, 0.7, 1.0, V)
    g = np_out(ssd.ssd_round(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"], F, 8,
                             dev_status=status))
    st = int(status.item())
    assert st & ssd.SSD_DEV_BAD_TOKEN and st & ssd.SSD_DEV_BAD_TEMPERATURE and st & ssd.SSD_DEV_NONFINITE
    for b in (1, 2, 3, 4, 5):
        assert g["accept_len"][b] == -1 and g["bonus"][b] == -1 and g["hit"][b] == 0
    o = oracle.round_(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"], inp["temperature"],
                      "f32", off, 8)
    for b in (0, 6, 7):
        assert g["accept_len"][b] == o["accept_len"][b] and g["bonus"][b] == o["bonus"][b]


@pytest.mark.parametrize("K", [1, 3])
def test_lossless_on_gpu(ssd, K):
    """First emitted token ~ p (chi-square, 10^6 draws, V = 8) through the CUDA path,
    and every one of the ~10^6 (K=1) to ~3x10^6 (K=3) decisions compared with the oracle."""
    rng = np.random.default_rng(900 + K)
    V, n = 8, 1_000_000
    p = rng.dirichlet(np.ones(V), size=K + 1)
    q = rng.dirichlet(np.ones(V), size=K)
    zt = np.log(p).astype(np.float32)
    zd = np.log(q).astype(np.float32)
    qn = [qq / qq.sum() for qq in q]
    x = np.stack([np.minimum(np.searchsorted(np.cumsum(qn[i]), rng.random(n), side="right"), V - 1)
                  for i in range(K)], axis=1).astype(np.int32)
    u = rng.random((n, K + 1), dtype=np.float32)
    tau = np.ones(n, np.float32)
    tgt_np = np.ascontiguousarray(np.broadcast_to(zt, (n, K + 1, V)))
    drf_np = np.ascontiguousarray(np.broadcast_to(zd, (n, K, V)))
    dev = "cuda"
    out = ssd.ssd_verify(torch.from_numpy(tgt_np).to(dev), torch.from_numpy(drf_np).to(dev),
                         torch.from_numpy(x).to(dev), torch.from_numpy(u).to(dev),
                         torch.from_numpy(tau).to(dev))
    g = np_out(out)
    a, bonus = g["accept_len"], g["bonus"]
    assert (a >= 0).all()
    first = np.where(a >= 1, x[:, 0], bonus)
    hist = np.bincount(first, minlength=V)
    p0 = p[0] / p[0].sum()
    assert scipy.stats.chisquare(hist, p0 * n).pvalue > 1e-3
    allacc = a == K
    pK = p[K] / p[K].sum()
    assert scipy.stats.chisquare(np.bincount(bonus[allacc], minlength=V), pK * allacc.sum()).pvalue > 1e-3
    o = oracle.verify(tgt_np, drf_np, x, u, tau, "f32")
    t = Tally()
    compare_verify(g, o, K, t)
    t.check()


def test_deterministic_repeats(ssd):
    wl = synth.WORKLOADS["c5"].replace(B=24, greedy_first=12)
    inp = synth.make_inputs(wl, 4242)
    d = to_device(inp)
    F, off = ssd.ssd_fanout(wl.K, wl.budget, wl.a_p, wl.r, wl.V)
    ref = None
    for _ in range(3):
        g = np_out(ssd.ssd_round(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"],
                                 F, wl.budget))
        if ref is None:
            ref = g
        else:
            for k in ref:
                np.testing.assert_array_equal(ref[k], g[k])


def test_zero_budget_and_empty_segments(ssd):
    rng = np.random.default_rng(8)
    B, K, V = 5, 4, 700
    inp = _inputs(rng, B, K, V, "bf16", [1.0, 0.0, 1.0, 0.0, 1.0])
    d = to_device(inp)
    F = np.array([3, 0, 0, 2, 0], np.int32)
    off = np.concatenate([[0], np.cumsum(F)]).astype(np.int32)
    budget = 6  # one spare column beyond off[K+1] stays untouched
    g = np_out(ssd.ssd_round(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"], F,
                             budget))
    assert (g["cache_tok"][:, 5] == -1).all()
    o = oracle.round_(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"], inp["temperature"],
                      "bf16", off, budget)
    t = Tally()
    compare_verify(g, o, K, t)
    compare_cache(g["cache_tok"], o, off, K, t)
    t.check()
    Fz = np.zeros(K + 1, np.int32)
    g0 = np_out(ssd.ssd_round(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"], Fz,
                              0))
    assert (g0["hit"] == 0).all() and (g0["slot"] == -1).all()


def test_bounded_wait_gives_up_and_context_stays_usable(ssd):
    """A wait that nothing completes ends after its limit with SSD_DEV_TIMEOUT set,
    and the next round on the same context is still correct."""
    import time
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ssd.ssd_check_wait_timeout(st, 50)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st.item()) == ssd.SSD_DEV_TIMEOUT
    assert 0.04 < dt < 5.0
    wl = synth.WORKLOADS["c4"].replace(B=4, V=4096)
    inp = synth.make_inputs(wl, 7070)
    F, off = ssd.ssd_fanout(wl.K, wl.budget, wl.a_p, wl.r, wl.V)
    d = to_device(inp)
    g = np_out(ssd.ssd_round(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"], F,
                             wl.budget))
    o = oracle.round_(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"], inp["temperature"],
                      wl.dtype, off, wl.budget)
    t = Tally()
    compare_verify(g, o, wl.K, t)
    compare_cache(g["cache_tok"], o, off, wl.K, t)
    t.check()
