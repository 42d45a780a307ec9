"""The sigma_{F,C} reshape kernel's selection paths against the float64 oracle:
rows on and off the 16-byte grid (slices with partial boundary vectors), F = 256
(the general block selection with every element a candidate), F = 0, tiny V,
rows of equal values (more than 32 keys reach the threshold), all-negative rows
(the threshold rounded down into bf16 from below) and quantised rows with ties."""
import numpy as np
import pytest

import oracle
import synth

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


def _rows(V, dtype, seed):
    rng = np.random.default_rng(seed)
    z = (rng.standard_normal((6, V)) * 2.5).astype(np.float32) + synth.zipf_log_bias(V, 1.1)
    z[1] = 0.75                                          # all equal
    z[2] = -np.abs(z[2]) - 3.0                           # all negative
    z[3] = np.round(z[3] * 2).astype(np.float32) / 2     # ties
    z[4, ::7] = z[4].max() + 1.0                         # many equal maxima
    return synth.store(z, dtype)


@pytest.mark.parametrize("dtype,V,F", [("bf16", 24000, 256), ("f32", 20011, 8), ("bf16", 20011, 255),
                                       ("f32", 300, 1), ("bf16", 128256, 64), ("f32", 24000, 0),
                                       ("bf16", 4099, 33)])
def test_reshape_descriptors_and_q_match_oracle(ssd, dtype, V, F):
    stored = _rows(V, dtype, 80 + F)
    rows = stored.shape[0]
    t = torch.from_numpy(np.ascontiguousarray(stored).view(np.int16) if dtype == "bf16" else stored)
    t = t.cuda()
    if dtype == "bf16":
        t = t.view(torch.bfloat16)
    tau = np.full(rows, 0.8, np.float32)
    C = 0.3
    desc, q = ssd.ssd_reshape_draft(t, F, C, torch.from_numpy(tau).cuda(), want_q=True)
    thr_val, thr_id, Fd, _ = [x.cpu().numpy() for x in ssd.desc_fields(desc)]
    z = synth.stored_to_f32(stored, dtype).astype(np.float64)
    ro = oracle.reshape_rows(stored, tau, dtype, F, C)
    for r in range(rows):
        assert Fd[r] == F
        if F == 0:
            assert thr_id[r] == -1 and np.isinf(thr_val[r])
        else:
            ids = oracle.topf(z[r], F)
            assert thr_id[r] == ids[-1] and thr_val[r] == z[r, ids[-1]], (r, thr_id[r], ids[-1])
    err = np.abs(q.cpu().numpy() - ro["q"]).max()
    assert err <= 1e-5, err
