"""The seeded input generators that both the CUDA path and the oracle consume:
determinism by seed, shapes and storage, bf16 rounding (checked against torch's own
float32 -> bfloat16 conversion), the Zipf log-bias, the greedy split, and the
drafting step's Gumbel-max law (chi-square against softmax(z / tau))."""
import numpy as np
import pytest
from scipy import stats

import synth


def test_inputs_are_determined_by_the_seed():
    wl = synth.WORKLOADS["c5"].replace(B=3, V=4096)
    a, b, c = synth.make_inputs(wl, 11), synth.make_inputs(wl, 11), synth.make_inputs(wl, 12)
    for k in ("tgt", "drf", "tokens", "uniforms", "temperature"):
        np.testing.assert_array_equal(a[k], b[k])
    assert not np.array_equal(a["tgt"], c["tgt"]) and not np.array_equal(a["uniforms"], c["uniforms"])


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5"])
def test_shapes_and_storage(name):
    wl = synth.WORKLOADS[name].replace(B=2, V=1024)
    inp = synth.make_inputs(wl, 3)
    B, K, V = wl.B, wl.K, wl.V
    assert inp["tgt"].shape == (B, K + 1, V) and inp["drf"].shape == (B, K, V)
    assert inp["tgt"].dtype == (np.float32 if wl.dtype == "f32" else np.uint16)
    assert inp["tokens"].shape == (B, K) and inp["tokens"].dtype == np.int32
    assert ((inp["tokens"] >= 0) & (inp["tokens"] < V)).all()
    u = inp["uniforms"]
    assert u.shape == (B, K + 1) and u.dtype == np.float32 and ((u >= 0) & (u < 1)).all()
    assert np.isfinite(synth.stored_to_f32(inp["tgt"], wl.dtype)).all()


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 30,
                        np.float32([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0, -0.0,
                                    np.inf, -np.inf, 3.0e38, 1e-40])])
    ours = synth.bf16_bits_from_f32(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    back = synth.f32_from_bf16_bits(ours)
    np.testing.assert_array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_zipf_bias_is_a_power_law():
    V, s = 5000, 1.1
    bias = synth.zipf_log_bias(V, s)
    assert bias[0] == 0 and (np.diff(bias) < 0).all()
    t = np.arange(V, dtype=np.float64)
    np.testing.assert_allclose(np.exp(bias.astype(np.float64)), np.power(t + 1, -s), rtol=1e-5)


def test_greedy_split():
    wl = synth.WORKLOADS["c5"]
    tau = synth.temperatures(wl)
    assert (tau[: wl.greedy_first] == 0).all() and (tau[wl.greedy_first:] == wl.tau).all()


def test_drafting_follows_softmax_of_the_scaled_logits():
    rng = np.random.default_rng(9)
    z = np.float32([1.5, 0.0, -0.7, 2.2, 0.3])
    n, tau = 40000, 0.7
    tokens = synth.sample_draft_tokens(rng, np.broadcast_to(z, (n, 1, z.size)).copy(),
                                       np.full(n, tau, np.float32))
    counts = np.bincount(tokens.ravel(), minlength=z.size)
    p = np.exp(z.astype(np.float64) / tau)
    p /= p.sum()
    assert stats.chisquare(counts, p * n).pvalue > 1e-4
    greedy = synth.sample_draft_tokens(rng, np.broadcast_to(z, (3, 1, z.size)).copy(),
                                       np.zeros(3, np.float32))
    assert (greedy == 3).all()


def test_algorithmic_bytes_closed_forms():
    """The roofline numerator: distinct logit bytes a round must read.  A round reads
    2K+1 rows of a sampled sequence and K+1 of a greedy one; verification alone stops
    after the first rejection (2(a+1) rows, or a+1 greedy); a reshape reads each sampled
    draft row once more.  Counted here row by row from the shapes."""
    c5 = synth.WORKLOADS["c5"]
    tau = synth.temperatures(c5)
    V, K = c5.V, c5.K
    n_s = int(np.count_nonzero(tau > 0))
    assert n_s == 128
    assert synth.algorithmic_bytes(c5, tau) == 128 * 9 * V * 2 + 128 * 5 * V * 2 == 459_669_504

    c2 = synth.WORKLOADS["c2"]
    tau2 = synth.temperatures(c2)
    a = np.array([0, 1, 5, 2, 0, 5, 3, 4])      # accepted lengths, K = 5 (5 = every draft)
    rows = sum(2 * (x + 1) if x < c2.K else 2 * c2.K + 1 for x in a)
    assert synth.algorithmic_bytes(c2, tau2, a) == rows * c2.V * 2

    c3 = synth.WORKLOADS["c3"]
    tau3 = synth.temperatures(c3)
    a3 = np.full(c3.B, 2)
    extra = int(np.count_nonzero(tau3 > 0)) * c3.K * c3.V * 2   # the reshape's draft rows
    assert synth.algorithmic_bytes(c3, tau3, a3) == c3.B * 6 * c3.V * 2 + extra

    g = c5.replace(B=4, greedy_first=4)                 # every sequence greedy
    tg = synth.temperatures(g)
    assert synth.algorithmic_bytes(g, tg) == 4 * (K + 1) * V * 2
    gv = g.replace(mode="verify")
    assert synth.algorithmic_bytes(gv, tg, np.array([0, 1, 4, 2])) == (1 + 2 + 5 + 3) * V * 2
