"""Helpers for GPU-vs-oracle parity tests (test infrastructure).

Tolerance rule (the stated parity bar for this path):
* accepted lengths, bonus tokens, top-F sets and cache hits must match the
  float64 oracle exactly, except decisions whose oracle margin (|u - p/q| for an
  accept test, the normalised CDF gap for a bonus draw, the score gap at the
  top-F boundary) is below 1e-6; such mismatches are counted and must be at
  most 1e-5 of all decisions;
* probabilities (p_tok, q_tok, reshaped q') must agree within 1e-5 absolute.
"""
from __future__ import annotations

from contextlib import contextmanager
from dataclasses import dataclass, field

import numpy as np
import torch

import synth

MARGIN = 1e-6
PROB_ATOL = 1e-5
EXEMPT_RATIO = 1e-5


@dataclass
class Tally:
    decisions: int = 0
    exempt: int = 0
    near_margin: int = 0
    hard: list = field(default_factory=list)

    def check(self):
        """Hard mismatches fail the test at once; near-tie mismatches are added to the
        suite-wide count, whose ratio to all decisions is checked after the parity tests
        (tests/test_zy_parity_ratio.py)."""
        assert not self.hard, "hard mismatches:\n" + "\n".join(self.hard[:20])
        SESSION.decisions += self.decisions
        SESSION.exempt += self.exempt
        SESSION.near_margin += self.near_margin


SESSION = Tally()


def to_device(inp: dict, device="cuda") -> dict:
    """numpy inputs (stored fp32 or bf16 bits) -> torch CUDA tensors."""
    wl = inp["workload"]

    def logits(a):
        if wl.dtype == synth.F32:
            return torch.from_numpy(np.ascontiguousarray(a)).to(device)
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)

    return {"tgt": logits(inp["tgt"]), "drf": logits(inp["drf"]),
            "tokens": torch.from_numpy(np.ascontiguousarray(inp["tokens"], dtype=np.int32)).to(device),
            "uniforms": torch.from_numpy(np.ascontiguousarray(inp["uniforms"], dtype=np.float32)).to(device),
            "temperature": torch.from_numpy(np.ascontiguousarray(inp["temperature"], dtype=np.float32)).to(device)}


def np_out(d: dict) -> dict:
    return {k: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def compare_verify(g: dict, o: dict, K: int, tally: Tally, probs: bool = True):
    """Accepted lengths, bonus tokens and p/q of the drafted tokens (vectorised)."""
    ga, gb = np.asarray(g["accept_len"]), np.asarray(g["bonus"])
    oa, ob = np.asarray(o["accept_len"]), np.asarray(o["bonus"])
    am, bm = np.asarray(o["acc_margin"]), np.asarray(o["bonus_margin"])

    def hard(mask, fmt):
        for b in np.nonzero(mask)[0][:20]:
            tally.hard.append(fmt(int(b)))

    inv = oa < 0
    tally.decisions += int(inv.sum())
    hard(inv & (ga != -1), lambda b: f"b={b}: oracle invalid, gpu accept_len={ga[b]}")
    hard(~inv & (ga < 0), lambda b: f"b={b}: gpu flagged the sequence invalid, oracle a={oa[b]}")
    ok = ~inv & (ga >= 0)
    n = np.minimum(ga, oa)
    cnt = np.where(ok, np.minimum(n + 1, K), 0)
    tally.decisions += int(cnt.sum())
    cols = np.arange(K)[None, :]
    tally.near_margin += int(((cols < cnt[:, None]) & (am < MARGIN)).sum())
    diff = ok & (ga != oa)
    if diff.any():
        m = am[np.nonzero(diff)[0], n[diff]]
        tally.exempt += int((m < MARGIN).sum())
        bad = np.zeros_like(diff)
        bad[np.nonzero(diff)[0][m >= MARGIN]] = True
        hard(bad, lambda b: f"b={b}: accept_len gpu={ga[b]} oracle={oa[b]} "
                            f"(margin {am[b, n[b]]:.3g} at i={n[b]})")
    same = ok & (ga == oa)
    tally.decisions += int(same.sum())
    tally.near_margin += int((same & (bm < MARGIN)).sum())
    bdiff = same & (gb != ob)
    tally.exempt += int((bdiff & (bm < MARGIN)).sum())
    hard(bdiff & (bm >= MARGIN), lambda b: f"b={b}: bonus gpu={gb[b]} oracle={ob[b]} a={oa[b]} "
                                           f"(margin {bm[b]:.3g})")
    if probs and "p_tok" in g:
        gp, gq = np.asarray(g["p_tok"], np.float64), np.asarray(g["q_tok"], np.float64)
        op, oq = np.asarray(o["p_tok"]), np.asarray(o["q_tok"])
        inside = same[:, None] & (cols <= oa[:, None])
        past = same[:, None] & (cols > oa[:, None])
        err = inside & ~((np.abs(gp - op) <= PROB_ATOL) & (np.abs(gq - oq) <= PROB_ATOL))
        hard(err.any(axis=1), lambda b: f"b={b}: p/q gpu=({gp[b].tolist()},{gq[b].tolist()}) "
                                        f"oracle=({op[b].tolist()},{oq[b].tolist()})")
        nn = past & ~(np.isnan(gp) & np.isnan(gq))
        hard(nn.any(axis=1), lambda b: f"b={b}: p/q past a must be NaN, got ({gp[b].tolist()})")


def compare_cache(g_cache: np.ndarray, o: dict, off, K: int, tally: Tally, skip_rows=()):
    """Cache segments in rank order.  A segment is a near-tie decision when the oracle's
    boundary margin or a gap between consecutive kept scores lies in (0, 1e-6).  Exact
    ties (gap 0) are decided by the lowest id on both sides, so they must match bit for
    bit; the one exception is a sampled sequence whose kept scores reach 0, the clamp of
    (p - q)^+, which hides how close the clamped residuals are to 0 (the order among
    them, and the boundary, then counts as near)."""
    oc = o["cache_tok"]
    tau = np.asarray(o.get("temperature", np.ones(oc.shape[0], np.float32)))
    for b in range(oc.shape[0]):
        if b in skip_rows:
            continue
        for k in range(K + 1):
            lo, hi = int(off[k]), int(off[k + 1])
            if hi == lo:
                continue
            tally.decisions += 1
            sg, so = g_cache[b, lo:hi], oc[b, lo:hi]
            sc = o["cache_score"][b, lo:hi]
            gaps = -np.diff(sc) if hi - lo > 1 else np.array([np.inf])
            near = (o["cache_margin"][b, k] < MARGIN or bool(np.any((gaps > 0) & (gaps < MARGIN)))
                    or (tau[b] > 0 and sc[-1] == 0.0))
            if near:
                tally.near_margin += 1
            if np.array_equal(sg, so):
                continue
            if near:
                tally.exempt += 1
            else:
                tally.hard.append(f"b={b} k={k}: cache gpu={sg.tolist()} oracle={so.tolist()} "
                                  f"(margin {o['cache_margin'][b, k]:.3g})")


def lookup_from(cache: np.ndarray, off, a: np.ndarray, t: np.ndarray):
    """Reference hit test (integer only) on the given cache / outcomes."""
    B = cache.shape[0]
    hit = np.zeros(B, np.uint8)
    slot = np.full(B, -1, np.int32)
    for b in range(B):
        if a[b] < 0:
            continue
        seg = cache[b, off[a[b]]:off[a[b] + 1]]
        w = np.nonzero(seg == t[b])[0]
        if len(w):
            hit[b] = 1
            slot[b] = off[a[b]] + w[0]
    return hit, slot


@contextmanager
def use_dispatch(ssd, policy):
    """Runs the block with the library's kernel choice forced to `policy`."""
    prev = ssd.ssd_set_dispatch(policy)
    try:
        yield
    finally:
        ssd.ssd_set_dispatch(prev)
