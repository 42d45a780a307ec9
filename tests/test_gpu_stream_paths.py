"""Rarely taken paths of the streaming kernel (rows on the 16-byte grid), each
compared with the float64 oracle:

* a draft row equal to its target row, rejected at a token both give
  probability 0: no residual mass, so the bonus is drawn from p;
* accepted positions, whose second pass computes residuals only for the groups
  that can hold the cache top-F (bounded from the first pass's group maxima),
  with those groups clustered at the lowest ids (a few tail lanes) or with no
  residual at all (draft equal to target: every group is computed);
* a fan-out with F_k above 64, where the top-F threshold is found by bisection
  over the group maxima instead of from the lanes' two largest maxima;
* pair rows of one chunk, of exactly the chunks a second pass streams unasked,
  and of one chunk more;
* rows whose logits are all equal, where every group reaches the threshold
  (the candidate-group list overflows and all groups are re-read) and every
  element ties (the candidate-key buffer overflows and the threshold is raised
  by sorting) -- ties rank by ascending token id.
"""
import numpy as np
import pytest

import oracle
import synth
from tests._parity import (Tally, compare_cache, compare_verify, lookup_from, np_out, to_device,
                           use_dispatch)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", params=["stream", "slice", "wide"])
def ssd(request):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_ssd_gb300 as m
    from speculative_decoding_verification_ssd_gb300 import _build
    _build.build()
    # these batches are small: force the persistent kernel whose paths they exercise
    # (the streaming kernel in either form, or the slice kernel, which has the same
    # paths per slice)
    policy = {"stream": m.SSD_DISPATCH_STREAM, "slice": m.SSD_DISPATCH_SLICE,
              "wide": m.SSD_DISPATCH_WIDE}[request.param]
    with use_dispatch(m, policy):
        yield m


def _pack(zt, zd, tok, u, taus, dtype):
    B, K1, V = zt.shape
    wl = synth.Workload("paths", B=B, K=K1 - 1, V=V, dtype=dtype, sigma_d=0, zipf_s=0, sigma_n=0,
                        tau=1.0)
    return {"tgt": synth.store(zt, dtype), "drf": synth.store(zd, dtype),
            "tokens": tok.astype(np.int32), "uniforms": u.astype(np.float32),
            "temperature": np.asarray(taus, np.float32), "workload": wl}


def _round_and_compare(ssd, inp, budget, a_p, r):
    wl = inp["workload"]
    K, V = wl.K, wl.V
    F, off = ssd.ssd_fanout(K, budget, a_p, r, V)
    d = to_device(inp)
    assert d["tgt"].data_ptr() % 16 == 0 and (V * wl.elem_bytes) % 16 == 0  # streaming path
    g = np_out(ssd.ssd_round(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"], F,
                             budget))
    o = oracle.round_(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"], inp["temperature"],
                      wl.dtype, off, budget)
    t = Tally()
    compare_verify(g, o, K, t)
    compare_cache(g["cache_tok"], o, off, K, t)
    h, s = lookup_from(g["cache_tok"], off, g["accept_len"], g["bonus"])
    np.testing.assert_array_equal(g["hit"], h)
    np.testing.assert_array_equal(g["slot"], s)
    t.check()
    return g, o, F


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_draft_equal_to_target_draws_bonus_from_p(ssd, dtype):
    """q = p, and the drafted token at position a = b mod K has logit -inf in both
    rows: positions before a accept (u < 1), a rejects (u * 0 < 0 fails), and the
    residual at a has no mass, so the bonus is drawn from p_a."""
    rng = np.random.default_rng(31)
    B, K, V = 8, 3, 20000
    zt = (rng.standard_normal((B, K + 1, V)) * 2.5).astype(np.float32)
    tok = rng.integers(0, V, (B, K))
    want_a = np.arange(B) % K
    for b in range(B):
        zt[b, want_a[b], tok[b, want_a[b]]] = -np.inf
    zd = zt[:, :K].copy()
    u = rng.random((B, K + 1))
    inp = _pack(zt, zd, tok, u, [1.0] * B, dtype)
    g, o, F = _round_and_compare(ssd, inp, 24, 0.7, 0.5)
    np.testing.assert_array_equal(g["accept_len"], want_a)
    zs = synth.stored_to_f32(inp["tgt"], dtype)
    checked = 0
    for b in range(B):
        p = oracle.softmax(zs[b, want_a[b]].astype(np.float64), 1.0)
        cum = np.cumsum(p)
        T = float(inp["uniforms"][b, K]) * cum[-1]
        want = int(np.searchsorted(cum, T, side="right"))
        if abs(cum[min(want, V - 1)] - T) < 1e-6 or (want > 0 and abs(cum[want - 1] - T) < 1e-6):
            continue  # too close to a boundary to be a clean decision
        assert g["bonus"][b] == want, (b, g["bonus"][b], want)
        checked += 1
    assert checked >= B - 1


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fanout_above_64_uses_bisection(ssd, dtype):
    rng = np.random.default_rng(32)
    B, K, V = 6, 2, 24000
    zt = (rng.standard_normal((B, K + 1, V)) * 2.5).astype(np.float32)
    zd = (zt[:, :K] + rng.standard_normal((B, K, V)) * 0.8).astype(np.float32)
    tok = np.argmax(zd, axis=-1)
    u = rng.random((B, K + 1))
    _, _, F = _round_and_compare(ssd, _pack(zt, zd, tok, u, [1.0, 0.0, 0.7] * 2, dtype), 450, 0.8, 0.5)
    assert max(F) > 64


# pair rows of one 8 KB chunk (the wide form ends each pass on its second ring with a
# header-only stage), of exactly the eight chunks both rings take unasked in a second
# pass, and of one chunk more (a chunk list of one entry); single rows of one 16 KB chunk
@pytest.mark.parametrize("dtype,V", [("bf16", 1000), ("bf16", 4096), ("f32", 2000),
                                     ("bf16", 32768), ("bf16", 36864), ("f32", 16384),
                                     ("f32", 18432)])
def test_row_lengths_around_the_rings(ssd, dtype, V):
    rng = np.random.default_rng(V + (7 if dtype == "f32" else 0))
    B, K = 6, 3
    zt = (rng.standard_normal((B, K + 1, V)) * 2.5).astype(np.float32)
    zd = (zt[:, :K] + rng.standard_normal((B, K, V)) * 0.9).astype(np.float32)
    tok = np.argmax(zd + rng.gumbel(size=zd.shape), axis=-1)
    u = rng.random((B, K + 1))
    inp = _pack(zt, zd, tok, u, [1.0, 0.0, 0.7, 1.0, 1.0, 0.0], dtype)
    _round_and_compare(ssd, inp, 24, 0.75, 0.5)
    # verification alone (the early-exit form)
    d = to_device(inp)
    g = np_out(ssd.ssd_verify(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"]))
    o = oracle.verify(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"], inp["temperature"],
                      inp["workload"].dtype)
    t = Tally()
    compare_verify(g, o, K, t)
    t.check()


def test_all_equal_rows_overflow_both_candidate_buffers(ssd):
    rng = np.random.default_rng(33)
    B, K, V = 4, 2, 128256
    zt = (rng.standard_normal((B, K + 1, V)) * 2.0).astype(np.float32)
    zd = (zt[:, :K] + rng.standard_normal((B, K, V)) * 0.8).astype(np.float32)
    zt[0] = 0.0          # sampled sequence, all rows flat; draft flat too
    zd[0] = 0.0
    zt[1, :, :] = 1.5    # greedy sequence with flat target rows
    zt[2, 1] = -3.0      # one flat target row among random ones
    tok = rng.integers(0, V, (B, K))
    u = rng.random((B, K + 1))
    _round_and_compare(ssd, _pack(zt, zd, tok, u, [1.0, 0.0, 1.0, 0.0], "bf16"), 32, 0.75, 0.5)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_signed_zeros_tie(ssd, dtype):
    """-0.0 and +0.0 are one value: a row whose largest logit is zero, stored as -0.0
    at a low id and +0.0 at a higher id, has its argmax at the low id, and zero-valued
    cache candidates rank by id."""
    rng = np.random.default_rng(34)
    B, K, V = 4, 2, 24000
    zt = -np.abs(rng.standard_normal((B, K + 1, V)).astype(np.float32)) - 0.5
    zd = -np.abs(rng.standard_normal((B, K, V)).astype(np.float32)) - 0.5
    for b in range(B):
        for k in range(K + 1):
            zt[b, k, 100 + k] = -0.0
            zt[b, k, 5000 + k] = 0.0
            zt[b, k, 7000 + k] = -0.0
    zd[:, :, 300] = 0.0
    zd[:, :, 200] = -0.0
    tok = np.zeros((B, K), np.int64)
    tok[:, 0] = 100
    tok[:, 1] = 5001               # not the argmax (101): rejected, greedy bonus 101
    u = rng.random((B, K + 1))
    _round_and_compare(ssd, _pack(zt, zd, tok, u, [0.0, 1.0, 0.0, 0.5], dtype), 12, 0.7, 0.5)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("same", [False, True])
def test_accepted_pairs_bound_the_groups_they_compute(ssd, dtype, same):
    """u = 0 accepts every drafted token with p > 0, so each pair's residual only ranks
    its cache top-F: the second pass computes the groups whose bound p(max z_p) reaches
    the F-th largest lower bound p(max z_p) - q(max z_q).  The large logits sit in
    groups 0-7 (the first two tail lanes), or the draft equals the target (no positive
    bound: every group is computed)."""
    rng = np.random.default_rng(35)
    B, K, V = 6, 3, 24000
    zd = (rng.standard_normal((B, K + 1, V)) * 2.5).astype(np.float32)
    zd[:, :, :512] += 6.0
    zt = zd if same else (zd + rng.standard_normal((B, K + 1, V)) * 0.8).astype(np.float32)
    tok = rng.integers(0, 512, (B, K))
    u = rng.random((B, K + 1))
    u[:, :K] = 0.0
    inp = _pack(zt, zd[:, :K].copy(), tok, u, [1.0] * B, dtype)
    g, o, F = _round_and_compare(ssd, inp, 28, 0.75, 0.5)
    assert (g["accept_len"] == K).all()


def test_round_reads_inputs_written_just_before_it(ssd):
    """The streaming kernel is launched so that it may start while the kernel before
    it on the stream drains; it must still see what that kernel wrote.  Temperatures
    and uniforms are rewritten by torch kernels right before each round (the greedy
    and sampled halves swapped, fresh uniforms), and every round is compared with the
    oracle on the values written last."""
    wl = synth.WORKLOADS["c5"].replace(B=64, greedy_first=32)
    inp = synth.make_inputs(wl, synth.PARITY_SEED["c5"] + 31)
    F, off = ssd.ssd_fanout(wl.K, wl.budget, wl.a_p, wl.r, wl.V)
    d = to_device(inp)
    tau_a = inp["temperature"]
    tau_b = np.where(tau_a > 0, 0.0, 1.0).astype(np.float32)
    rng = np.random.default_rng(5)
    tau_dev = torch.empty_like(d["temperature"])
    u_dev = torch.empty_like(d["uniforms"])
    ws = ssd.workspace(wl.B, wl.K, V=wl.V, dtype=ssd.SSD_BF16, budget=wl.budget)
    outs, cases = [], []
    for tau_np in (tau_a, tau_b, tau_a):
        u_np = rng.random((wl.B, wl.K + 1), dtype=np.float32)
        tau_src = torch.from_numpy(tau_np).cuda()
        u_src = torch.from_numpy(u_np).cuda()
        torch.cuda.synchronize()
        tau_dev.copy_(tau_src)          # written by a torch kernel right before the round
        u_dev.copy_(u_src)
        out = ssd.ssd_round(d["tgt"], d["drf"], d["tokens"], u_dev, tau_dev, F, wl.budget,
                            workspace=ws)
        outs.append({k: v.clone() for k, v in out.items()})
        cases.append((tau_np, u_np))
    torch.cuda.synchronize()
    for out, (tau_np, u_np) in zip(outs, cases):
        g = np_out(out)
        o = oracle.round_(inp["tgt"], inp["drf"], inp["tokens"], u_np, tau_np, wl.dtype, off,
                          wl.budget)
        t = Tally()
        compare_verify(g, o, wl.K, t)
        compare_cache(g["cache_tok"], o, off, wl.K, t)
        t.check()
