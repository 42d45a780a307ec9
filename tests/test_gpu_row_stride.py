"""Logit rows spaced ld > V elements apart ([..., :V] views of padded rows), with
vocabularies whose rows are not whole 16-byte vectors, against the float64 oracle
on the same V columns.  The padding holds NaN: any use of it would show.  Rows on
the 16-byte grid stream (the partial last vector masked); other strides take the
cluster kernel."""
import numpy as np
import pytest

import oracle
import synth
from tests._parity import Tally, compare_cache, compare_verify, lookup_from, np_out, use_dispatch

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


def _padded(stored, dtype, ld):
    B, R, V = stored.shape
    if dtype == "bf16":
        pad = np.full((B, R, ld), 0x7FC0, np.uint16)   # bf16 NaN
        pad[:, :, :V] = stored
        t = torch.from_numpy(pad.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        pad = np.full((B, R, ld), np.nan, np.float32)
        pad[:, :, :V] = stored
        t = torch.from_numpy(pad).cuda()
    return t[:, :, :V]


@pytest.mark.parametrize("policy", [1, 2])  # streaming kernel, cluster kernel
@pytest.mark.parametrize("dtype,V,ld,B", [("bf16", 50257, 50304, 12), ("f32", 32001, 32004, 10),
                                          ("f32", 32001, 32002, 6), ("bf16", 4099, 4104, 40),
                                          ("bf16", 50257, 50304, 200)])
def test_round_on_strided_rows(ssd, dtype, V, ld, B, policy):
    wl = synth.WORKLOADS["c5"].replace(B=B, V=V, dtype=dtype, greedy_first=B // 3)
    inp = synth.make_inputs(wl, 6100 + V % 97 + B)
    F, off = ssd.ssd_fanout(wl.K, wl.budget, wl.a_p, wl.r, V)
    tgt, drf = _padded(inp["tgt"], dtype, ld), _padded(inp["drf"], dtype, ld)
    assert tgt.stride(1) == ld and not tgt.is_contiguous()
    with use_dispatch(ssd, policy):
        g = np_out(ssd.ssd_round(tgt, drf, torch.from_numpy(inp["tokens"]).cuda(),
                                 torch.from_numpy(inp["uniforms"]).cuda(),
                                 torch.from_numpy(inp["temperature"]).cuda(), F, wl.budget))
    o = oracle.round_(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"], inp["temperature"],
                      dtype, off, wl.budget)
    t = Tally()
    compare_verify(g, o, wl.K, t)
    compare_cache(g["cache_tok"], o, off, wl.K, t)
    h, s = lookup_from(g["cache_tok"], off, g["accept_len"], g["bonus"])
    np.testing.assert_array_equal(g["hit"], h)
    np.testing.assert_array_equal(g["slot"], s)
    t.check()


def test_verify_on_strided_rows(ssd):
    wl = synth.WORKLOADS["c2"].replace(B=8, V=50257)
    inp = synth.make_inputs(wl, 6201)
    tgt, drf = _padded(inp["tgt"], "bf16", 50304), _padded(inp["drf"], "bf16", 50304)
    with use_dispatch(ssd, ssd.SSD_DISPATCH_STREAM):
        g = np_out(ssd.ssd_verify(tgt, drf, torch.from_numpy(inp["tokens"]).cuda(),
                                  torch.from_numpy(inp["uniforms"]).cuda(),
                                  torch.from_numpy(inp["temperature"]).cuda()))
    o = oracle.verify(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"], inp["temperature"],
                      "bf16")
    t = Tally()
    compare_verify(g, o, wl.K, t)
    t.check()
