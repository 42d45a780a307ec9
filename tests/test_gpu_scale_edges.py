"""Limits of the fused round against the float64 oracle: the largest lookahead
(K = SSD_MAX_K = 32), a batch above the streaming kernel's ordered-unit list
(B > 2048: units are handed out in a strided order instead), and vocabularies at
and beyond the streaming kernel's group-array capacity (V = 160000 streams;
V = 200000 takes the cluster kernel)."""
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


def _round(ssd, wl, seed, F=None):
    inp = synth.make_inputs(wl, seed)
    if F is None:
        F, off = ssd.ssd_fanout(wl.K, wl.budget, wl.a_p, wl.r, wl.V)
    else:
        off = np.concatenate([[0], np.cumsum(F)]).astype(np.int32)
    d = to_device(inp)
    g = np_out(ssd.ssd_round(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"], F,
                             wl.budget))
    o = oracle.round_(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"], inp["temperature"],
                      wl.dtype, off, wl.budget)
    t = Tally()
    compare_verify(g, o, wl.K, t)
    compare_cache(g["cache_tok"], o, off, wl.K, t)
    h, s = lookup_from(g["cache_tok"], off, g["accept_len"], g["bonus"])
    np.testing.assert_array_equal(g["hit"], h)
    np.testing.assert_array_equal(g["slot"], s)
    t.check()
    return g


@pytest.mark.parametrize("policy", [1, 2])  # streaming kernel, cluster kernel
def test_largest_lookahead(ssd, policy):
    wl = synth.WORKLOADS["c5"].replace(B=6, K=32, V=8192, greedy_first=2, budget=100,
                                       sigma_n=0.3)
    with use_dispatch(ssd, policy):
        g = _round(ssd, wl, 5101)
    assert (g["accept_len"] >= 0).all()


def test_batch_above_the_ordered_unit_list(ssd):
    wl = synth.WORKLOADS["c4"].replace(B=2100, K=1, V=1024, budget=8, greedy_first=700)
    _round(ssd, wl, 5102)


@pytest.mark.parametrize("V", [160000, 200000])
def test_vocabularies_at_the_group_array_limit(ssd, V):
    wl = synth.WORKLOADS["c5"].replace(B=4, K=2, V=V, greedy_first=2)
    with use_dispatch(ssd, ssd.SSD_DISPATCH_STREAM):  # 160000 streams, 200000 cannot
        _round(ssd, wl, 5103 + V % 7)
