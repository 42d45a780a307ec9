"""CPU checks of the C ABI: the library builds and loads without a GPU, exports
every function include/ssd.h declares, and its host-only logic (argument
validation, workspace sizing, the fan-out) behaves as documented.  No call
here reaches a kernel: every device call is rejected by host validation."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ssd():
    from speculative_decoding_verification_ssd_gb300 import _build
    _build.build()
    import speculative_decoding_verification_ssd_gb300 as m
    return m


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "ssd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssd_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(ssd):
    declared = _declared_functions()
    assert set(declared) == set(ssd.ABI_SYMBOLS)
    L = ctypes.CDLL(ssd.LIB_PATH)
    for name in declared:
        assert hasattr(L, name), name


def test_strerror_and_version(ssd):
    for code in range(6):
        assert ssd.strerror(code)
    assert "unknown" in ssd.strerror(99)
    assert "sm_103a" in ssd.version()


def test_dispatch_policy(ssd):
    assert ssd.ssd_set_dispatch(ssd.SSD_DISPATCH_STREAM) == ssd.SSD_DISPATCH_AUTO
    assert ssd.ssd_set_dispatch(ssd.SSD_DISPATCH_CLUSTER) == ssd.SSD_DISPATCH_STREAM
    assert ssd.ssd_set_dispatch(ssd.SSD_DISPATCH_SLICE) == ssd.SSD_DISPATCH_CLUSTER
    assert ssd.ssd_set_dispatch(ssd.SSD_DISPATCH_WIDE) == ssd.SSD_DISPATCH_SLICE
    assert ssd.ssd_set_dispatch(ssd.SSD_DISPATCH_AUTO) == ssd.SSD_DISPATCH_WIDE
    with pytest.raises(ValueError):
        ssd.ssd_set_dispatch(7)
    with pytest.raises(ValueError):
        ssd.ssd_set_dispatch(5)
    assert ssd.lib().ssd_set_dispatch(-3) == -1
    assert ssd.ssd_set_dispatch(ssd.SSD_DISPATCH_AUTO) == ssd.SSD_DISPATCH_AUTO


def test_workspace_size(ssd):
    assert ssd.ssd_workspace_size(0, 4) == 0
    assert ssd.ssd_workspace_size(4, 0) == 0
    assert ssd.ssd_workspace_size(4, 33) == 0
    n = ssd.ssd_workspace_size(256, 4)
    assert n % 256 == 0 and n >= 256 * 5 * 32 + 2 * 256 * 4


@pytest.mark.parametrize("K,budget,a_p,r,V", [(6, 64, 0.8, 1.0, 152064), (4, 32, 0.75, 0.5, 128256),
                                               (3, 12, 0.5625, 1.0, 100), (8, 100, 0.6, 0.0, 10),
                                               (2, 100, 0.5, 1.0, 20), (1, 0, 0.3, 2.0, 5)])
def test_fanout_matches_oracle(ssd, K, budget, a_p, r, V):
    F, off = ssd.ssd_fanout(K, budget, a_p, r, V)
    Fo, offo, _ = oracle.fanout(K, budget, a_p, r, V)
    np.testing.assert_array_equal(F, Fo)
    np.testing.assert_array_equal(off, offo)


def test_fanout_random_parameters_match_oracle(ssd):
    rng = np.random.default_rng(0)
    for _ in range(300):
        K = int(rng.integers(1, 33))
        budget = int(rng.integers(0, 500))
        a_p = float(rng.uniform(0.01, 0.99))
        r = float(rng.uniform(-0.9, 4.0))
        V = int(rng.integers(1, 1000))
        F, off = ssd.ssd_fanout(K, budget, a_p, r, V)
        Fo, offo, x = oracle.fanout(K, budget, a_p, r, V)
        frac = np.sort(x - np.floor(x))
        if len(frac) > 1 and np.min(np.diff(frac)) < 1e-12:
            continue  # a remainder tie at rounding precision: either order is a valid reading
        np.testing.assert_array_equal(F, Fo)


def test_fanout_rejects_bad_arguments(ssd):
    for args in [(0, 10, 0.5, 1.0, 10), (33, 10, 0.5, 1.0, 10), (3, -1, 0.5, 1.0, 10),
                 (3, 10, 0.0, 1.0, 10), (3, 10, 1.0, 1.0, 10), (3, 10, 0.5, -1.0, 10),
                 (3, 10, 0.5, float("nan"), 10), (3, 10, 0.5, 1.0, 0)]:
        with pytest.raises(ssd.SSDError) as e:
            ssd.ssd_fanout(*args)
        assert e.value.status == ssd.SSD_ERR_INVALID_ARG


def test_fanout_uniform_matches_oracle(ssd):
    for K in range(1, 33):
        for budget in [0, 1, K, K + 1, 2 * K + 3, 32, 64, 255, 1000]:
            for V in [1, 3, 50, 128256]:
                F, off = ssd.ssd_fanout_uniform(K, budget, V)
                Fo, offo = oracle.fanout_uniform(K, budget, V)
                np.testing.assert_array_equal(F, Fo)
                np.testing.assert_array_equal(off, offo)
    for args in [(0, 10, 10), (33, 10, 10), (3, -1, 10), (3, 10, 0)]:
        with pytest.raises(ssd.SSDError) as e:
            ssd.ssd_fanout_uniform(*args)
        assert e.value.status == ssd.SSD_ERR_INVALID_ARG


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


def test_host_staging_size(ssd):
    bf, f32 = ssd.SSD_BF16, ssd.SSD_F32
    assert ssd.ssd_host_staging_size(bf, 0, 4, 100, 8) == 0
    assert ssd.ssd_host_staging_size(bf, 4, 0, 100, 8) == 0
    assert ssd.ssd_host_staging_size(bf, 4, 33, 100, 8) == 0
    assert ssd.ssd_host_staging_size(bf, 4, 2, 1, 8) == 0
    assert ssd.ssd_host_staging_size(bf, 4, 2, 100, -1) == 0
    assert ssd.ssd_host_staging_size(9, 4, 2, 100, 8) == 0
    for dt, s in ((bf, 2), (f32, 4)):
        B, K, V, budget = 256, 4, 128256, 32
        raw = B * (2 * K + 1) * V * s + B * K * 4 + B * (K + 1) * 4 + 4 * B * 4 + B * budget * 4 + B
        n = ssd.ssd_host_staging_size(dt, B, K, V, budget)
        assert raw <= n < raw + 10 * 256 and n % 256 == 0


def test_device_calls_validate_before_any_cuda_call(ssd):
    L = ssd.lib()
    p = _fake()
    ws_ok = ssd.ssd_workspace_size(4, 2)

    def verify(dtype=ssd.SSD_F32, B=4, K=2, V=100, drf_rows=2, ws=p, ws_bytes=ws_ok, tgt=p):
        return L.ssd_verify(tgt, p, dtype, B, K, V, drf_rows, p, p, p, None, p, p, None, None, ws,
                            ws_bytes, None, None)

    assert verify(dtype=7) == ssd.SSD_ERR_DTYPE
    assert verify(B=0) == ssd.SSD_ERR_INVALID_ARG
    assert verify(K=0) == ssd.SSD_ERR_INVALID_ARG
    assert verify(K=33, drf_rows=33) == ssd.SSD_ERR_INVALID_ARG
    assert verify(V=1) == ssd.SSD_ERR_INVALID_ARG
    assert verify(drf_rows=5) == ssd.SSD_ERR_INVALID_ARG
    assert verify(tgt=None) == ssd.SSD_ERR_INVALID_ARG
    assert verify(V=10 ** 6) == ssd.SSD_ERR_UNSUPPORTED
    assert verify(ws=None) == ssd.SSD_ERR_WORKSPACE
    assert verify(ws=_fake(0x10010)) == ssd.SSD_ERR_WORKSPACE
    assert verify(ws_bytes=ws_ok - 1) == ssd.SSD_ERR_WORKSPACE
    # p_tok without q_tok
    assert L.ssd_verify(p, p, 0, 4, 2, 100, 2, p, p, p, None, p, p, p, None, p, ws_ok, None,
                        None) == ssd.SSD_ERR_INVALID_ARG

    F = np.array([2, 1, 3], np.int32)
    Fp = F.ctypes.data_as(ctypes.c_void_p)
    Fbig = np.array([2, 300, 3], np.int32)
    Fneg = np.array([2, -1, 3], np.int32)
    cache = L.ssd_build_cache
    assert cache(p, p, 0, 4, 2, 100, 2, p, p, None, Fp, 5, p, p, ws_ok, None, None) == \
        ssd.SSD_ERR_INVALID_ARG  # budget < sum F
    assert cache(p, p, 0, 4, 2, 100, 2, p, p, None, Fbig.ctypes.data_as(ctypes.c_void_p), 400, p, p,
                 ws_ok, None, None) == ssd.SSD_ERR_INVALID_ARG  # F_k > SSD_MAX_F
    assert cache(p, p, 0, 4, 2, 100, 2, p, p, None, Fneg.ctypes.data_as(ctypes.c_void_p), 10, p, p,
                 ws_ok, None, None) == ssd.SSD_ERR_INVALID_ARG
    F3 = np.array([2, 1, 3], np.int32)
    assert cache(p, p, 0, 4, 2, 2, 2, p, p, None, F3.ctypes.data_as(ctypes.c_void_p), 6, p, p,
                 ws_ok, None, None) == ssd.SSD_ERR_INVALID_ARG  # F_k > V
    assert cache(p, p, 0, 4, 2, 100, 2, p, p, None, None, 6, p, p, ws_ok, None, None) == \
        ssd.SSD_ERR_INVALID_ARG
    assert L.ssd_round(p, p, 0, 4, 2, 100, 2, p, p, p, None, Fp, 6, p, p, None, None, p, None, p,
                       p, ws_ok, None, None) == ssd.SSD_ERR_INVALID_ARG  # hit missing
    assert L.ssd_cache_lookup(p, 4, 2, 5, Fp, p, p, p, p, None) == ssd.SSD_ERR_INVALID_ARG
    assert L.ssd_cache_lookup(p, 0, 2, 6, Fp, p, p, p, p, None) == ssd.SSD_ERR_INVALID_ARG
    dc = L.ssd_draft_cache
    Fz = np.array([2, 100, 3], np.int32).ctypes.data_as(ctypes.c_void_p)
    c = ctypes.c_float
    assert dc(p, 5, 4, 2, 100, p, Fp, 6, c(1), p, None, None, None) == ssd.SSD_ERR_DTYPE
    assert dc(p, 0, 4, 2, 100, p, Fp, 6, c(1), None, None, None, None) == \
        ssd.SSD_ERR_INVALID_ARG  # neither cache nor descriptors
    assert dc(p, 0, 4, 2, 100, p, Fp, 5, c(1), p, None, None, None) == \
        ssd.SSD_ERR_INVALID_ARG  # budget < sum F
    assert dc(p, 0, 4, 2, 100, p, None, 6, c(1), p, None, None, None) == ssd.SSD_ERR_INVALID_ARG
    assert dc(p, 0, 4, 2, 100, p, Fp, 6, c(1.5), None, p, None, None) == ssd.SSD_ERR_INVALID_ARG
    assert dc(p, 0, 4, 2, 100, p, Fz, 105, c(0), None, p, None, None) == \
        ssd.SSD_ERR_INVALID_ARG  # C == 0 with F_k = V: no weight left
    Fv = np.array([2, 101, 3], np.int32).ctypes.data_as(ctypes.c_void_p)
    assert dc(p, 0, 4, 2, 100, p, Fv, 106, c(1), p, None, None, None) == \
        ssd.SSD_ERR_INVALID_ARG  # F_k > V
    need = ssd.ssd_host_staging_size(0, 4, 2, 100, 6)

    def rhost(dtype=0, B=4, K=2, V=100, F=Fp, budget=6, tgt=p, staging=p, staging_bytes=need):
        return L.ssd_round_host(tgt, p, dtype, B, K, V, p, p, p, F, budget, p, p, p, p, p, staging,
                                staging_bytes, p, ws_ok, None, None, None)

    assert rhost(dtype=5) == ssd.SSD_ERR_DTYPE
    assert rhost(B=0) == ssd.SSD_ERR_INVALID_ARG
    assert rhost(tgt=None) == ssd.SSD_ERR_INVALID_ARG
    assert rhost(staging=None) == ssd.SSD_ERR_INVALID_ARG
    assert rhost(F=None) == ssd.SSD_ERR_INVALID_ARG
    assert rhost(budget=5) == ssd.SSD_ERR_INVALID_ARG  # budget < sum F
    assert rhost(F=Fneg.ctypes.data_as(ctypes.c_void_p), budget=10) == ssd.SSD_ERR_INVALID_ARG
    assert rhost(staging_bytes=need - 1) == ssd.SSD_ERR_INVALID_ARG
    assert L.ssd_check_wait_timeout(None, 20, None) == ssd.SSD_ERR_INVALID_ARG
    assert L.ssd_check_wait_timeout(p, 0, None) == ssd.SSD_ERR_INVALID_ARG
    assert L.ssd_check_wait_timeout(p, 10001, None) == ssd.SSD_ERR_INVALID_ARG
    assert L.ssd_verify_ld(p, p, 0, 4, 2, 100, 99, 2, p, p, p, None, p, p, None, None, p, ws_ok, None,
                           None) == ssd.SSD_ERR_INVALID_ARG  # ld < V
    assert L.ssd_round_ld(p, p, 0, 4, 2, 100, 99, 2, p, p, p, None, Fp, 6, p, p, None, None, p, p, p,
                          p, ws_ok, None, None) == ssd.SSD_ERR_INVALID_ARG
    bf = L.ssd_backup_fill
    assert bf(p, p, 0, 4, 100, p, None) == ssd.SSD_ERR_INVALID_ARG
    assert bf(p, p, 4, 0, 100, p, None) == ssd.SSD_ERR_INVALID_ARG
    assert bf(p, p, 4, 33, 100, p, None) == ssd.SSD_ERR_INVALID_ARG
    assert bf(p, p, 4, 2, 0, p, None) == ssd.SSD_ERR_INVALID_ARG
    assert bf(None, p, 4, 2, 100, p, None) == ssd.SSD_ERR_INVALID_ARG
    assert bf(p, p, 4, 2, 100, None, None) == ssd.SSD_ERR_INVALID_ARG
    rs = L.ssd_reshape_draft
    assert rs(p, 3, 4, 100, p, 8, ctypes.c_float(0.5), p, None, None, None) == ssd.SSD_ERR_DTYPE
    assert rs(p, 0, 4, 100, p, 300, ctypes.c_float(0.5), p, None, None, None) == ssd.SSD_ERR_INVALID_ARG
    assert rs(p, 0, 4, 100, p, 8, ctypes.c_float(1.5), p, None, None, None) == ssd.SSD_ERR_INVALID_ARG
    assert rs(p, 0, 4, 100, p, 8, ctypes.c_float(float("nan")), p, None, None, None) == \
        ssd.SSD_ERR_INVALID_ARG
    assert rs(p, 0, 4, 8, p, 8, ctypes.c_float(0.0), p, None, None, None) == ssd.SSD_ERR_INVALID_ARG
    assert rs(p, 0, 4, 100, None, 8, ctypes.c_float(0.5), p, p, None, None) == ssd.SSD_ERR_INVALID_ARG


def test_round_host_binding_validates_before_any_device_use(ssd):
    torch = pytest.importorskip("torch")
    B, K, V = 4, 2, 64
    tgt = torch.zeros((B, K + 1, V), dtype=torch.float32)
    drf = torch.zeros((B, K, V), dtype=torch.float32)
    tok = torch.zeros((B, K), dtype=torch.int32)
    u = torch.zeros((B, K + 1), dtype=torch.float32)
    tau = torch.ones(B, dtype=torch.float32)
    F = [1, 1, 1]
    with pytest.raises(ValueError):
        ssd.ssd_round_host(tgt, drf[:, :1], tok, u, tau, F, 3)  # drf not [B, K, V]
    with pytest.raises(TypeError):
        ssd.ssd_round_host(tgt, drf.to(torch.bfloat16), tok, u, tau, F, 3)  # dtypes differ
    with pytest.raises(TypeError):
        ssd.ssd_round_host(tgt, drf, tok.to(torch.int64), u, tau, F, 3)
    with pytest.raises(ValueError):
        ssd.ssd_round_host(tgt, drf, tok, u[:, :K], tau, F, 3)  # uniforms not [B, K+1]
    with pytest.raises(ValueError):
        ssd.ssd_round_host(tgt.transpose(0, 1), drf, tok, u, tau, F, 3)  # not contiguous
