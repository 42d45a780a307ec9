"""Seeded synthetic workloads for the verify-and-sample step and the Saguaro cache.

This module is the one piece shared by the CPU oracle's tests and the CUDA path's
tests and benchmark.  It draws inputs only: logits, draft tokens, uniforms and
temperatures.  It holds none of the method's arithmetic (no softmax, no accept
test, no residual, no fan-out, no top-F).  Random numbers the method consumes
(the accept/bonus uniforms) are drawn here and passed in as inputs.

Input recipe (one per workload, all drawn from ``numpy.random.default_rng(seed)``):

* draft logits   z_d[b, i, t] ~ N(0, sigma_d^2) - s * ln(t + 1)   (a Zipf(s) log-bias,
  token id 0 most frequent), drawn for i = 0..K (row K is never stored: it only
  seeds target row K);
* target logits  z_t[b, i, t] = z_d[b, i, t] + N(0, sigma_n^2), i = 0..K;
* both generated in fp32, then stored as fp32 or as bf16 (round to nearest even);
* draft tokens   x~[b, i] drawn from the draft's own sampling distribution at the
  sequence's temperature (Gumbel-max over the stored draft logits / tau, plus an
  optional additive log-bias supplied by the caller, e.g. the log C of a reshaped
  draft distribution); greedy sequences (tau = 0) draft the argmax;
* uniforms       u[b, i] ~ U[0, 1) fp32, shape [B, K+1];
* temperature    per sequence, fp32.

The parameters of the five named workloads follow the speculative-decoding pages'
problem statement (target logits [B, K+1, V], draft tokens [B, K], uniforms
[B, K+1]); the pages evaluate on HumanEval, UltraFeedback, Alpaca and GSM8k with
Llama / Qwen weights, which are not used here: these seeded synthetic logits
stand in for the verify-time logits such runs produce.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np

F32 = "f32"
BF16 = "bf16"


@dataclass(frozen=True)
class Workload:
    """One synthetic verify / cache workload (sizes and value distribution)."""

    name: str
    B: int
    K: int
    V: int
    dtype: str                 # "f32" or "bf16": storage type of the logits
    sigma_d: float             # std of the draft logits' Gaussian part
    zipf_s: float              # Zipf exponent of the log-bias over token id
    sigma_n: float             # std of the target-minus-draft noise
    tau: float                 # temperature of the sampled sequences
    greedy_first: int = 0      # sequences b < greedy_first use tau = 0 (argmax)
    reshape_F: int = 0         # sigma_{F,C} reshape of the draft (0 = none)
    reshape_C: float = 1.0
    budget: int = 0            # Saguaro cache budget per sequence (0 = no cache)
    a_p: float = 0.0           # fan-out acceptance-rate parameter
    r: float = 0.0             # fan-out power-law exponent
    mode: str = "verify"       # "verify" or "round" (verify + cache + lookup)
    description: str = ""

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == F32 else 2


WORKLOADS: dict[str, Workload] = {
    "c1": Workload(
        "c1", B=1, K=4, V=32000, dtype=F32, sigma_d=3.0, zipf_s=1.1, sigma_n=0.5,
        tau=1.0, mode="verify",
        description="B=1, K=4, V=32000 fp32 logits, tau=1, plain verify"),
    "c2": Workload(
        "c2", B=8, K=5, V=128256, dtype=BF16, sigma_d=3.0, zipf_s=1.1, sigma_n=0.7,
        tau=1.0, mode="verify",
        description="B=8, K=5, V=128256 bf16 logits, tau=1, verify + residual bonus"),
    "c3": Workload(
        "c3", B=64, K=8, V=128256, dtype=BF16, sigma_d=3.0, zipf_s=1.1, sigma_n=1.0,
        tau=0.7, reshape_F=8, reshape_C=0.5, mode="verify",
        description="B=64, K=8, V=128256 bf16, tau=0.7, sigma_{F,C} draft reshape "
                    "F=8 C=0.5 before drafting, verify on the reshaped q"),
    "c4": Workload(
        "c4", B=32, K=6, V=152064, dtype=F32, sigma_d=4.0, zipf_s=1.2, sigma_n=0.6,
        tau=1.0, budget=64, a_p=0.8, r=1.0, mode="round",
        description="B=32, K=6, V=152064 fp32, cache build (budget 64, a_p=0.8, r=1) "
                    "+ verify + lookup"),
    "c5": Workload(
        "c5", B=256, K=4, V=128256, dtype=BF16, sigma_d=3.0, zipf_s=1.1, sigma_n=0.8,
        tau=1.0, greedy_first=128, budget=32, a_p=0.75, r=0.5, mode="round",
        description="B=256, K=4, V=128256 bf16, half greedy (b<128) half tau=1, "
                    "verify + fan-out cache build (budget 32, a_p=0.75, r=0.5) + lookup"),
}

# Seeds: parity inputs use 1000 + index, benchmark inputs 2000 + index.
PARITY_SEED = {name: 1000 + i for i, name in enumerate(WORKLOADS, start=1)}
BENCH_SEED = {name: 2000 + i for i, name in enumerate(WORKLOADS, start=1)}


# ---------------------------------------------------------------------------
# Storage conversions (bit-level; no rounding other than fp32 -> bf16 RNE).
# ---------------------------------------------------------------------------

def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even.

    NaN inputs map to a quiet NaN."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounding = np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    out = ((u + rounding) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def f32_from_bf16_bits(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exactly equal fp32 values."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def stored_to_f32(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Stored logits (fp32 array or bf16 bit patterns) -> fp32 values (exact)."""
    if dtype == F32:
        return np.asarray(arr, dtype=np.float32)
    return f32_from_bf16_bits(arr)


def store(x_f32: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 values -> stored representation for ``dtype``."""
    if dtype == F32:
        return np.ascontiguousarray(x_f32, dtype=np.float32)
    return bf16_bits_from_f32(x_f32)


# ---------------------------------------------------------------------------
# Draws.
# ---------------------------------------------------------------------------

def zipf_log_bias(V: int, s: float) -> np.ndarray:
    """-s * ln(t + 1) for t = 0..V-1 (fp32): the log of a Zipf(s) pmf up to a constant."""
    return (-s * np.log1p(np.arange(V, dtype=np.float64))).astype(np.float32)


def temperatures(wl: Workload) -> np.ndarray:
    tau = np.full(wl.B, wl.tau, dtype=np.float32)
    tau[: min(wl.greedy_first, wl.B)] = 0.0
    return tau


def sample_draft_tokens(rng: np.random.Generator, drf_f32: np.ndarray, tau: np.ndarray,
                        log_bias: np.ndarray | None = None) -> np.ndarray:
    """Simulates the draft model's own sampling (the drafting step upstream of
    verification): x~ = argmax_t (z_t / tau + log_bias_t + G_t), G ~ Gumbel(0, 1),
    which draws x~ from the distribution proportional to exp(z / tau + log_bias).
    tau = 0 drafts the argmax of the stored draft row (lowest id on ties)."""
    B, K, V = drf_f32.shape
    out = np.empty((B, K), dtype=np.int32)
    for b in range(B):
        if tau[b] == 0.0:
            out[b] = np.argmax(drf_f32[b], axis=-1)
            continue
        u = rng.random((K, V))
        u = np.maximum(u, np.finfo(np.float64).tiny)
        g = -np.log(-np.log(u))
        score = drf_f32[b].astype(np.float64) / float(tau[b]) + g
        if log_bias is not None:
            score = score + log_bias[b]
        out[b] = np.argmax(score, axis=-1)
    return out


def make_logits(wl: Workload, rng: np.random.Generator, draft_rows: int | None = None):
    """Draws the stored target logits [B, K+1, V] and draft logits [B, draft_rows, V]
    (draft_rows K by default; K+1 keeps the draft row of position K, which a cache
    built from draft logits alone needs for the all-accepted outcome).  The random
    stream is the same for either choice."""
    B, K, V = wl.B, wl.K, wl.V
    R = K if draft_rows is None else int(draft_rows)
    assert R in (K, K + 1)
    bias = zipf_log_bias(V, wl.zipf_s)
    tgt = np.empty((B, K + 1, V), dtype=np.float32 if wl.dtype == F32 else np.uint16)
    drf = np.empty((B, R, V), dtype=tgt.dtype)
    for b in range(B):
        zd = rng.standard_normal((K + 1, V), dtype=np.float32) * np.float32(wl.sigma_d) + bias
        zt = zd + rng.standard_normal((K + 1, V), dtype=np.float32) * np.float32(wl.sigma_n)
        tgt[b] = store(zt, wl.dtype)
        drf[b] = store(zd[:R], wl.dtype)
    return tgt, drf


def make_inputs(wl: Workload, seed: int, draft_log_bias=None) -> dict:
    """All inputs of one round of ``wl``.

    ``draft_log_bias``: optional callable (drf_f32 [B,K,V]) -> additive log-weights
    [B,K,V] of the draft's sampling distribution (used when the draft samples
    from a reshaped distribution)."""
    rng = np.random.default_rng(seed)
    tgt, drf = make_logits(wl, rng)
    tau = temperatures(wl)
    drf_f32 = stored_to_f32(drf, wl.dtype)
    bias = draft_log_bias(drf_f32) if draft_log_bias is not None else None
    tokens = sample_draft_tokens(rng, drf_f32, tau, bias)
    uniforms = rng.random((wl.B, wl.K + 1), dtype=np.float32)
    return {"tgt": tgt, "drf": drf, "tokens": tokens, "uniforms": uniforms,
            "temperature": tau, "workload": wl, "seed": seed}


def make_rows(rng: np.random.Generator, rows: int, V: int, dtype: str, sigma: float = 3.0,
              zipf_s: float = 1.1) -> np.ndarray:
    """Independent logit rows [rows, V] (stored), same value distribution as the draft."""
    bias = zipf_log_bias(V, zipf_s)
    z = rng.standard_normal((rows, V), dtype=np.float32) * np.float32(sigma) + bias
    return store(z, dtype)


def algorithmic_bytes(wl: Workload, tau: np.ndarray, accept_len: np.ndarray | None = None) -> int:
    """Distinct logit bytes the method must read for one round.

    round mode: every row is needed (each k's residual feeds the cache):
      sampled sequences (2K+1) rows, greedy sequences K+1 target rows.
    verify mode: rows after the first rejection are not needed:
      sampled: 2(a+1) rows if a < K else 2K+1; greedy: a+1 target rows (a<K) else K+1.
    """
    s = wl.elem_bytes
    V, K = wl.V, wl.K
    total = 0
    for b in range(wl.B):
        greedy = tau[b] == 0.0
        if wl.mode == "round" or accept_len is None:
            rows = (K + 1) if greedy else (2 * K + 1)
        else:
            a = int(accept_len[b])
            if greedy:
                rows = a + 1 if a < K else K + 1
            else:
                rows = 2 * (a + 1) if a < K else 2 * K + 1
        total += rows * V * s
    if wl.reshape_F > 0:
        # the reshape reads every draft row of the sampled sequences once more
        total += int(np.count_nonzero(tau > 0)) * K * V * s
    return total
