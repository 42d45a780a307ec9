"""The workspace-free round (ssd_round_noalloc) against the ordinary round.

For callers that cannot allocate device memory (a plugin whose host framework
owns all device buffers, a runtime with a fixed footprint), the library offers
one entry point that keeps its scratch in a static device array instead of a
caller-provided workspace.  This test calls it through the C ABI twice in a
row -- the second call sees the array as the first call left it -- and checks
both results against ssd_round with its own workspace: every integer output
must be identical and the probabilities equal within 1e-5.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes when run on its own.
"""
import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ssd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_ssd_gb300 import _build
    _build.build()
    import speculative_decoding_verification_ssd_gb300 as m
    return m


def _device_inputs(inp, dev="cuda"):
    wl = inp["workload"]
    t = torch.from_numpy(inp["tgt"].view(np.int16)).to(dev).view(torch.bfloat16)
    d = torch.from_numpy(inp["drf"].view(np.int16)).to(dev).view(torch.bfloat16)
    assert wl.dtype == synth.BF16
    return (t, d, torch.from_numpy(inp["tokens"]).to(dev), torch.from_numpy(inp["uniforms"]).to(dev),
            torch.from_numpy(inp["temperature"]).to(dev))


def _noalloc_round(ssd, tgt, drf, tok, u, tau, F, budget):
    B, K1, V = tgt.shape
    K = K1 - 1
    dev = tgt.device
    out = {"accept_len": torch.full((B,), -7, dtype=torch.int32, device=dev),
           "bonus": torch.full((B,), -7, dtype=torch.int32, device=dev),
           "p_tok": torch.full((B, K), -7.0, dtype=torch.float32, device=dev),
           "q_tok": torch.full((B, K), -7.0, dtype=torch.float32, device=dev),
           "cache_tok": torch.full((B, budget), -1, dtype=torch.int32, device=dev),
           "hit": torch.full((B,), 7, dtype=torch.uint8, device=dev),
           "slot": torch.full((B,), -7, dtype=torch.int32, device=dev)}
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    Fh = np.ascontiguousarray(F, dtype=np.int32)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = ssd.lib().ssd_round_noalloc(
        p(tgt), p(drf), ssd.SSD_BF16, B, K, V, int(drf.shape[1]), p(tok), p(u), p(tau), None,
        Fh.ctypes.data_as(ctypes.c_void_p), budget, p(out["accept_len"]), p(out["bonus"]),
        p(out["p_tok"]), p(out["q_tok"]), p(out["cache_tok"]), p(out["hit"]), p(out["slot"]),
        p(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == ssd.SSD_OK, ssd.strerror(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return {k: v.cpu().numpy() for k, v in out.items()}


@pytest.mark.parametrize("B,policy", [(48, "auto"), (48, "stream"), (48, "cluster"), (8, "auto")])
def test_noalloc_round_matches_round_on_two_calls(ssd, B, policy):
    """B = 48 (240 units, between one and two per SM) runs the persistent streaming
    kernel in its wide form by default, in its one-group-per-unit form or the cluster
    kernel when forced; B = 8 (40 units, fewer than the SMs) takes the cluster kernel
    by itself.  Every kernel uses the same counters and records in the array."""
    wl = synth.WORKLOADS["c5"].replace(B=B, greedy_first=B // 2)
    inp = synth.make_inputs(wl, 777 + B)
    tgt, drf, tok, u, tau = _device_inputs(inp)
    F, off = ssd.ssd_fanout(wl.K, wl.budget, wl.a_p, wl.r, wl.V)
    pol = {"auto": ssd.SSD_DISPATCH_AUTO, "stream": ssd.SSD_DISPATCH_STREAM,
           "cluster": ssd.SSD_DISPATCH_CLUSTER}[policy]
    prev = ssd.ssd_set_dispatch(pol)
    try:
        ref = ssd.ssd_round(tgt, drf, tok, u, tau, F, wl.budget)
        torch.cuda.synchronize()
        ref = {k: v.cpu().numpy() for k, v in ref.items()}
        gots = [_noalloc_round(ssd, tgt, drf, tok, u, tau, F, wl.budget) for _ in range(2)]
    finally:
        ssd.ssd_set_dispatch(prev)
    for got in gots:
        for key in ("accept_len", "bonus", "cache_tok", "hit", "slot"):
            np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
        for key in ("p_tok", "q_tok"):
            np.testing.assert_array_equal(np.isnan(got[key]), np.isnan(ref[key]))
            ok = ~np.isnan(ref[key])
            np.testing.assert_allclose(got[key][ok], ref[key][ok], atol=1e-5, rtol=0)


def test_noalloc_rejects_batches_beyond_the_array(ssd):
    L = ssd.lib()
    cap = L.ssd_noalloc_max_scratch()
    B = 8192
    assert ssd.ssd_workspace_size(B, 32) > cap
    p = ctypes.c_void_p(0x10000)
    F = np.zeros(33, np.int32)
    rc = L.ssd_round_noalloc(p, p, ssd.SSD_BF16, B, 32, 1024, 32, p, p, p, None,
                             F.ctypes.data_as(ctypes.c_void_p), 0, p, p, None, None, p, p, p, None,
                             None)
    assert rc == ssd.SSD_ERR_UNSUPPORTED
