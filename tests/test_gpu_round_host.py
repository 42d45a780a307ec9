"""ssd_round_host: the round on host buffers gives exactly the device round's
outputs, copies only the sampled sequences' draft rows (a greedy sequence's draft
logits are NaN here and must not matter), and agrees with the float64 oracle --
also when the batch is copied and run in chunks that overlap."""
import numpy as np
import pytest

import oracle
import synth
from tests._parity import Tally, compare_cache, compare_verify, np_out, to_device

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


def _host_logits(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if dtype == "bf16" else np.ascontiguousarray(a))
    return (t.view(torch.bfloat16) if dtype == "bf16" else t).pin_memory()


@pytest.mark.parametrize("dtype,B,K,V,greedy", [("bf16", 24, 3, 20480, [0, 1, 2, 9, 10, 23]),
                                                 ("f32", 12, 2, 4096, [5]),
                                                 ("bf16", 8, 4, 8192, list(range(8))),
                                                 # copied and run in chunks (64 sequences or
                                                 # more each); greedy runs cross the boundaries
                                                 ("bf16", 160, 2, 4096,
                                                  list(range(10)) + list(range(75, 91)) + [150, 159]),
                                                 ("f32", 300, 2, 2048, list(range(60, 170)))])
def test_round_host_matches_device_round_and_oracle(ssd, dtype, B, K, V, greedy):
    wl = synth.WORKLOADS["c5"].replace(B=B, K=K, V=V, dtype=dtype, greedy_first=0, budget=24)
    inp = synth.make_inputs(wl, 6100 + B)
    tau = inp["temperature"].copy()
    tau[greedy] = 0.0
    inp["temperature"] = tau
    F, off = ssd.ssd_fanout(wl.K, wl.budget, wl.a_p, wl.r, wl.V)
    d = to_device(inp)
    g_dev = np_out(ssd.ssd_round(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"], F,
                                 wl.budget, probs=False))
    drf_poison = inp["drf"].copy()
    nan = np.float32(np.nan)
    drf_poison[greedy] = synth.store(np.full((len(greedy), K, V), nan, np.float32), dtype)
    host = {"tgt": _host_logits(inp["tgt"], dtype), "drf": _host_logits(drf_poison, dtype),
            "tokens": torch.from_numpy(inp["tokens"]).pin_memory(),
            "uniforms": torch.from_numpy(inp["uniforms"]).pin_memory(),
            "temperature": torch.from_numpy(tau).pin_memory()}
    o, h2d = ssd.ssd_round_host(host["tgt"], host["drf"], host["tokens"], host["uniforms"],
                                host["temperature"], F, wl.budget)
    torch.cuda.synchronize()
    g = {k: v.numpy() for k, v in o.items()}
    for k in ("accept_len", "bonus", "cache_tok", "hit", "slot"):
        np.testing.assert_array_equal(g[k], g_dev[k], err_msg=k)
    s = 2 if dtype == "bf16" else 4
    n_sampled = B - len(set(greedy))
    assert h2d == B * (K + 1) * V * s + n_sampled * K * V * s + B * K * 4 + B * (K + 1) * 4 + B * 4
    o_ref = oracle.round_(inp["tgt"], inp["drf"], inp["tokens"], inp["uniforms"], tau, dtype, off,
                          wl.budget)
    t = Tally()
    compare_verify(g, o_ref, K, t)
    compare_cache(g["cache_tok"], o_ref, off, K, t)
    t.check()


def test_round_host_rejects_device_tensors(ssd):
    x = torch.zeros((2, 3, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(TypeError):
        ssd.ssd_round_host(x, x[:, :2], torch.zeros((2, 2), dtype=torch.int32),
                           torch.zeros((2, 3)), torch.ones(2), [1, 1, 1], 3)
