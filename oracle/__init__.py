"""Float64 CPU oracle for the verify-and-sample step and the Saguaro cache side.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  It shares
no code with the CUDA library (``speculative_decoding_verification_ssd_gb300``)
and never imports it.

The arithmetic lives in ``oracle.c`` (plain C, double precision, sequential
loops in token-id order, one function per step of the pages, each citing its
passage).  This module only marshals numpy arrays into it and splits a batch
across host threads (sequences are independent).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(worked table, closed forms, exact enumeration, Monte Carlo, brute force,
library routines).  Where the pages are silent -- which uniform draws the
bonus, the CDF order and boundary, the Z == 0 fallback -- they fix only the
law of the draw.  The chi-square and exact-enumeration pins check that law;
the chosen readings are pinned token by token against numpy's inverse CDF
(``searchsorted`` over the cumulative weights of scipy's softmax, ascending
token id) on the same uniforms.
"""
from __future__ import annotations

import ctypes
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import build as _build

F32, BF16 = 0, 1
_DTYPES = {"f32": F32, "bf16": BF16}

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i, d = ctypes.c_int, ctypes.c_double
        L.oracle_softmax.argtypes = [P, i, d, P]
        L.oracle_softmax.restype = None
        L.oracle_topf.argtypes = [P, i, i, P]
        L.oracle_topf.restype = None
        L.oracle_sigma.argtypes = [P, i, d, i, d, P, P]
        L.oracle_sigma.restype = i
        L.oracle_fanout.argtypes = [i, i, d, d, i, P, P, P]
        L.oracle_fanout.restype = i
        L.oracle_fanout_uniform.argtypes = [i, i, i, P, P]
        L.oracle_fanout_uniform.restype = i
        L.oracle_backup_fill.argtypes = [P, P, i, i, i, P]
        L.oracle_backup_fill.restype = None
        L.oracle_verify.argtypes = [i, i, i, i, i, i, P, P, i, P, P, P, i, P, d,
                                    P, P, P, P, P, P, P]
        L.oracle_verify.restype = i
        L.oracle_build_cache.argtypes = [i, i, i, i, i, i, P, P, i, P, P, i, P, d, P, i, P, P, P]
        L.oracle_draft_cache.argtypes = [i, i, i, i, P, P, P, i, P]
        L.oracle_draft_cache.restype = i
        L.oracle_p_hit.argtypes = [i, i, i, i, i, i, P, P, i, P, P, i, P, d, P, i, P, P]
        L.oracle_p_hit.restype = i
        L.oracle_build_cache.restype = i
        L.oracle_lookup.argtypes = [i, i, P, P, P, P, P, P]
        L.oracle_lookup.restype = None
        L.oracle_reshape_rows.argtypes = [i, i, i, i, P, P, i, d, P, P]
        L.oracle_reshape_rows.restype = i
        _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(dtype) -> int:
    return _DTYPES[dtype] if isinstance(dtype, str) else int(dtype)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _split(n: int, parts: int):
    parts = max(1, min(parts, n)) if n > 0 else 1
    bounds = np.linspace(0, n, parts + 1).astype(int)
    return [(int(bounds[j]), int(bounds[j + 1])) for j in range(parts) if bounds[j + 1] > bounds[j]]


# ---------------------------------------------------------------------------
# Single-row primitives.
# ---------------------------------------------------------------------------

def softmax(z, tau: float) -> np.ndarray:
    z = np.ascontiguousarray(z, dtype=np.float64)
    p = np.empty_like(z)
    lib().oracle_softmax(_ptr(z), z.size, float(tau), _ptr(p))
    return p


def topf(z, F: int) -> np.ndarray:
    z = np.ascontiguousarray(z, dtype=np.float64)
    out = np.empty(min(F, z.size), dtype=np.int32)
    lib().oracle_topf(_ptr(z), z.size, int(F), _ptr(out))
    return out


def sigma(z, tau: float, F: int, C: float):
    """sigma_{F,C} reshape of one draft row; returns (q', member flags) or raises."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    q = np.empty_like(z)
    mem = np.empty(z.size, dtype=np.uint8)
    rc = lib().oracle_sigma(_ptr(z), z.size, float(tau), int(F), float(C), _ptr(q), _ptr(mem))
    if rc != 0:
        raise ValueError("sigma_{F,C}: every token has zero weight")
    return q, mem.astype(bool)


def fanout(K: int, budget: int, a_p: float, r: float, V: int = 1 << 30):
    """Geometric fan-out: returns (F [K+1], off [K+2], x [K+1] real-valued)."""
    F = np.empty(K + 1, dtype=np.int32)
    off = np.empty(K + 2, dtype=np.int32)
    x = np.empty(K + 1, dtype=np.float64)
    rc = lib().oracle_fanout(int(K), int(budget), float(a_p), float(r), int(V), _ptr(F),
                             _ptr(off), _ptr(x))
    if rc != 0:
        raise ValueError("invalid fan-out parameters")
    return F, off, x


def fanout_uniform(K: int, budget: int, V: int = 1 << 30):
    """Uniform fan-out: returns (F [K+1], off [K+2])."""
    F = np.empty(K + 1, dtype=np.int32)
    off = np.empty(K + 2, dtype=np.int32)
    if lib().oracle_fanout_uniform(int(K), int(budget), int(V), _ptr(F), _ptr(off)) != 0:
        raise ValueError("invalid fan-out parameters")
    return F, off


def backup_fill(hit, uniforms, V: int, next_tokens):
    """Random-token backup: fills next_tokens [B, K] (int32, in place) for hit == 0."""
    hit = np.ascontiguousarray(hit, dtype=np.uint8)
    u = np.ascontiguousarray(uniforms, dtype=np.float32)
    assert next_tokens.dtype == np.int32 and next_tokens.flags.c_contiguous
    B, K = u.shape
    lib().oracle_backup_fill(_ptr(hit), _ptr(u), int(B), int(K), int(V), _ptr(next_tokens))
    return next_tokens


# ---------------------------------------------------------------------------
# Batched steps.
# ---------------------------------------------------------------------------

def _problem(tgt, drf, tokens, dtype):
    tgt = np.ascontiguousarray(tgt)
    drf = np.ascontiguousarray(drf)
    B, K1, V = tgt.shape
    K = K1 - 1
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, K)
    return tgt, drf, tokens, B, K, V, _dtype_code(dtype), drf.shape[1]


def _reshape_arg(reshape_F, K):
    """reshape_F: one F for every position, or a sequence of K per-position F_k."""
    if np.ndim(reshape_F) == 0:
        return int(reshape_F), None
    Fk = np.ascontiguousarray(np.asarray(reshape_F, dtype=np.int32).reshape(-1)[:K])
    assert Fk.size == K
    return 0, Fk


def verify(tgt, drf, tokens, uniforms, temperature, dtype, reshape_F=0,
           reshape_C: float = 1.0, threads: int | None = None) -> dict:
    tgt, drf, tokens, B, K, V, dt, drf_rows = _problem(tgt, drf, tokens, dtype)
    F1, Fk = _reshape_arg(reshape_F, K)
    u = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, K + 1)
    tau = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    out = {
        "accept_len": np.empty(B, np.int32), "bonus": np.empty(B, np.int32),
        "p_tok": np.empty((B, K), np.float64), "q_tok": np.empty((B, K), np.float64),
        "acc_margin": np.empty((B, K), np.float64), "bonus_margin": np.empty(B, np.float64),
        "Z": np.empty(B, np.float64),
    }

    def run(rng):
        return lib().oracle_verify(
            rng[0], rng[1], B, K, V, dt, _ptr(tgt), _ptr(drf), drf_rows, _ptr(tokens), _ptr(u),
            _ptr(tau), F1, _ptr(Fk), float(reshape_C), _ptr(out["accept_len"]),
            _ptr(out["bonus"]), _ptr(out["p_tok"]), _ptr(out["q_tok"]), _ptr(out["acc_margin"]),
            _ptr(out["bonus_margin"]), _ptr(out["Z"]))

    out["invalid"] = _parallel(run, B, threads)
    return out


def build_cache(tgt, drf, tokens, temperature, dtype, off, budget: int, reshape_F=0,
                reshape_C: float = 1.0, threads: int | None = None) -> dict:
    tgt, drf, tokens, B, K, V, dt, drf_rows = _problem(tgt, drf, tokens, dtype)
    F1, Fk = _reshape_arg(reshape_F, K)
    tau = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    off = np.ascontiguousarray(off, dtype=np.int32)
    out = {"cache_tok": np.empty((B, budget), np.int32),
           "cache_score": np.empty((B, budget), np.float64),
           "cache_margin": np.empty((B, K + 1), np.float64)}

    def run(rng):
        return lib().oracle_build_cache(
            rng[0], rng[1], B, K, V, dt, _ptr(tgt), _ptr(drf), drf_rows, _ptr(tokens), _ptr(tau),
            F1, _ptr(Fk), float(reshape_C), _ptr(off), int(budget), _ptr(out["cache_tok"]),
            _ptr(out["cache_score"]), _ptr(out["cache_margin"]))

    out["invalid"] = _parallel(run, B, threads)
    out["temperature"] = tau.copy()      # which scores are raw logits (tau == 0)
    return out


def draft_cache(drf, tokens, dtype, off, budget: int) -> np.ndarray:
    """Cache keys from the draft logits drf [B, K+1, V]: cache_tok [B, budget] int32
    (columns past off[K+1] are -2); tokens [B, K] (left out of their segment) or None."""
    drf = np.ascontiguousarray(drf)
    B, K1, V = drf.shape
    K = K1 - 1
    tok = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, K)
    off = np.ascontiguousarray(off, dtype=np.int32)
    cache = np.full((B, budget), -2, np.int32)
    if lib().oracle_draft_cache(B, K, V, _dtype_code(dtype), _ptr(drf), _ptr(tok), _ptr(off),
                                int(budget), _ptr(cache)) != 0:
        raise MemoryError("oracle_draft_cache")
    return cache


def p_hit(tgt, drf, tokens, temperature, dtype, off, budget: int, cache_tok, reshape_F=0,
          reshape_C: float = 1.0, threads: int | None = None) -> np.ndarray:
    """Per-sequence probability [B] that the round's outcome (a, t*) is in cache_tok,
    given the drafted tokens (the law of (a, t*) over the round's uniforms)."""
    tgt, drf, tokens, B, K, V, dt, drf_rows = _problem(tgt, drf, tokens, dtype)
    F1, Fk = _reshape_arg(reshape_F, K)
    tau = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    off = np.ascontiguousarray(off, dtype=np.int32)
    cache = np.ascontiguousarray(cache_tok, dtype=np.int32).reshape(B, budget)
    out = np.empty(B, np.float64)

    def run(rng):
        return lib().oracle_p_hit(rng[0], rng[1], B, K, V, dt, _ptr(tgt), _ptr(drf), drf_rows,
                                  _ptr(tokens), _ptr(tau), F1, _ptr(Fk), float(reshape_C),
                                  _ptr(off), int(budget), _ptr(cache), _ptr(out))

    if _parallel(run, B, threads):
        raise ValueError("invalid sequence")
    return out


def lookup(cache_tok, off, accept_len, bonus) -> dict:
    cache_tok = np.ascontiguousarray(cache_tok, dtype=np.int32)
    B, budget = cache_tok.shape
    off = np.ascontiguousarray(off, dtype=np.int32)
    a = np.ascontiguousarray(accept_len, dtype=np.int32)
    t = np.ascontiguousarray(bonus, dtype=np.int32)
    hit = np.empty(B, np.uint8)
    slot = np.empty(B, np.int32)
    lib().oracle_lookup(B, budget, _ptr(off), _ptr(cache_tok), _ptr(a), _ptr(t), _ptr(hit),
                        _ptr(slot))
    return {"hit": hit, "slot": slot}


def round_(tgt, drf, tokens, uniforms, temperature, dtype, off, budget: int,
           reshape_F: int = 0, reshape_C: float = 1.0, threads: int | None = None) -> dict:
    """One SSD round: verify + cache build + hit lookup of the true outcome."""
    v = verify(tgt, drf, tokens, uniforms, temperature, dtype, reshape_F, reshape_C, threads)
    c = build_cache(tgt, drf, tokens, temperature, dtype, off, budget, reshape_F, reshape_C,
                    threads)
    h = lookup(c["cache_tok"], off, v["accept_len"], v["bonus"])
    out = dict(v)
    out.update({k: c[k] for k in ("cache_tok", "cache_score", "cache_margin", "temperature")})
    out.update(h)
    out["invalid"] = v["invalid"] + c["invalid"]
    return out


def reshape_rows(logits, temperature, dtype, F: int, C: float, want_q: bool = True,
                 threads: int | None = None) -> dict:
    logits = np.ascontiguousarray(logits)
    V = logits.shape[-1]
    rows = logits.size // V
    tau = np.ascontiguousarray(temperature, dtype=np.float32).reshape(rows)
    q = np.empty((rows, V), np.float64) if want_q else None
    mem = np.empty((rows, V), np.uint8)

    def run(rng):
        return lib().oracle_reshape_rows(rng[0], rng[1], V, _dtype_code(dtype), _ptr(logits),
                                         _ptr(tau), int(F), float(C), _ptr(q), _ptr(mem))

    bad = _parallel(run, rows, threads)
    return {"q": q, "member": mem.astype(bool), "invalid": bad}


def _parallel(fn, n: int, threads: int | None) -> int:
    threads = default_threads() if threads is None else max(1, int(threads))
    chunks = _split(n, threads)
    if len(chunks) <= 1:
        return int(sum(fn(c) for c in chunks))
    with ThreadPoolExecutor(max_workers=len(chunks)) as ex:
        return int(sum(ex.map(fn, chunks)))
