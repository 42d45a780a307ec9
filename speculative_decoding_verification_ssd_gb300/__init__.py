"""Python binding of libssd: batched speculative-decoding verification and the
Saguaro speculation-cache kernels for GB300 (sm_103a).

The functions here carry the names of the C ABI in ``include/ssd.h`` and only
marshal arguments: torch tensors provide device memory and the CUDA stream,
every step of the computation runs in libssd's kernels.  If ``libssd.so`` has
not been built (``__graft_entry__.build()`` or ``python -m
speculative_decoding_verification_ssd_gb300._build``), every call raises:
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import _build

SSD_OK = 0
SSD_ERR_INVALID_ARG = 1
SSD_ERR_DTYPE = 2
SSD_ERR_CUDA = 3
SSD_ERR_WORKSPACE = 4
SSD_ERR_UNSUPPORTED = 5

SSD_F32 = 0
SSD_BF16 = 1

SSD_DEV_BAD_TOKEN = 1
SSD_DEV_BAD_TEMPERATURE = 2
SSD_DEV_NONFINITE = 4
SSD_DEV_TIMEOUT = 8

SSD_MAX_K = 32
SSD_MAX_F = 256

LIB_PATH = _build.LIB

# Symbols declared in include/ssd.h.
ABI_SYMBOLS = ("ssd_strerror", "ssd_version", "ssd_workspace_size", "ssd_verify", "ssd_fanout",
               "ssd_reshape_draft", "ssd_build_cache", "ssd_cache_lookup", "ssd_round",
               "ssd_noalloc_max_scratch", "ssd_round_noalloc", "ssd_fanout_uniform",
               "ssd_backup_fill", "ssd_draft_cache", "ssd_verify_sigma", "ssd_round_sigma",
               "ssd_set_dispatch", "ssd_check_wait_timeout", "ssd_verify_ld", "ssd_round_ld",
               "ssd_host_staging_size", "ssd_round_host", "ssd_last_kernel", "ssd_workspace_size_v")


class SSDError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {strerror(status)}")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libssd (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libssd is not built ({LIB_PATH} missing); run "
                               "`python -m speculative_decoding_verification_ssd_gb300._build`")
        L = ctypes.CDLL(LIB_PATH)
        P, i, d, z = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_size_t
        f = ctypes.c_float
        L.ssd_strerror.argtypes = [i]
        L.ssd_strerror.restype = ctypes.c_char_p
        L.ssd_version.argtypes = []
        L.ssd_version.restype = ctypes.c_char_p
        L.ssd_last_kernel.argtypes = []
        L.ssd_last_kernel.restype = ctypes.c_char_p
        L.ssd_workspace_size.argtypes = [i, i]
        L.ssd_workspace_size.restype = z
        L.ssd_workspace_size_v.argtypes = [i, i, i, i, i]
        L.ssd_workspace_size_v.restype = z
        L.ssd_verify.argtypes = [P, P, i, i, i, i, i, P, P, P, P, P, P, P, P, P, z, P, P]
        L.ssd_verify.restype = i
        L.ssd_fanout.argtypes = [i, i, d, d, i, P, P]
        L.ssd_fanout.restype = i
        L.ssd_reshape_draft.argtypes = [P, i, i, i, P, i, f, P, P, P, P]
        L.ssd_reshape_draft.restype = i
        L.ssd_build_cache.argtypes = [P, P, i, i, i, i, i, P, P, P, P, i, P, P, z, P, P]
        L.ssd_build_cache.restype = i
        L.ssd_cache_lookup.argtypes = [P, i, i, i, P, P, P, P, P, P]
        L.ssd_cache_lookup.restype = i
        L.ssd_round.argtypes = [P, P, i, i, i, i, i, P, P, P, P, P, i, P, P, P, P, P, P, P, P, z,
                                P, P]
        L.ssd_round.restype = i
        L.ssd_noalloc_max_scratch.argtypes = []
        L.ssd_noalloc_max_scratch.restype = z
        L.ssd_round_noalloc.argtypes = [P, P, i, i, i, i, i, P, P, P, P, P, i, P, P, P, P, P, P, P, P,
                                        P]
        L.ssd_round_noalloc.restype = i
        L.ssd_fanout_uniform.argtypes = [i, i, i, P, P]
        L.ssd_fanout_uniform.restype = i
        L.ssd_backup_fill.argtypes = [P, P, i, i, i, P, P]
        L.ssd_backup_fill.restype = i
        L.ssd_draft_cache.argtypes = [P, i, i, i, i, P, P, i, f, P, P, P, P]
        L.ssd_draft_cache.restype = i
        L.ssd_verify_sigma.argtypes = [P, P, i, i, i, i, i, P, P, P, P, f, P, P, P, P, P, P, z, P, P]
        L.ssd_verify_sigma.restype = i
        L.ssd_round_sigma.argtypes = [P, P, i, i, i, i, i, P, P, P, P, f, P, P, i, P, P, P, P, P, P,
                                      P, P, z, P, P]
        L.ssd_round_sigma.restype = i
        L.ssd_set_dispatch.argtypes = [i]
        L.ssd_set_dispatch.restype = i
        L.ssd_check_wait_timeout.argtypes = [P, i, P]
        L.ssd_check_wait_timeout.restype = i
        L.ssd_verify_ld.argtypes = [P, P, i, i, i, i, i, i, P, P, P, P, P, P, P, P, P, z, P, P]
        L.ssd_verify_ld.restype = i
        L.ssd_round_ld.argtypes = [P, P, i, i, i, i, i, i, P, P, P, P, P, i, P, P, P, P, P, P, P, P,
                                   z, P, P]
        L.ssd_round_ld.restype = i
        L.ssd_host_staging_size.argtypes = [i, i, i, i, i]
        L.ssd_host_staging_size.restype = z
        L.ssd_round_host.argtypes = [P, P, i, i, i, i, P, P, P, P, i, P, P, P, P, P, P, z, P, z, P, P,
                                     P]
        L.ssd_round_host.restype = i
        _lib = L
    return _lib


SSD_DISPATCH_AUTO, SSD_DISPATCH_STREAM, SSD_DISPATCH_CLUSTER, SSD_DISPATCH_SLICE, SSD_DISPATCH_WIDE = 0, 1, 2, 3, 4


def ssd_set_dispatch(policy: int) -> int:
    """Kernel choice for aligned rows (process-wide); returns the previous policy."""
    prev = int(lib().ssd_set_dispatch(int(policy)))
    if prev < 0:
        raise ValueError(f"unknown dispatch policy {policy}")
    return prev


def ssd_check_wait_timeout(dev_status, limit_ms: int, *, stream=None):
    """Runs the bounded-wait check: a wait nothing completes gives up after limit_ms
    and ORs SSD_DEV_TIMEOUT into dev_status (a device int32 tensor)."""
    _dev(dev_status, "dev_status", torch.int32)
    _check(lib().ssd_check_wait_timeout(_ptr(dev_status), int(limit_ms), _stream(stream)),
           "ssd_check_wait_timeout")
    return dev_status


def strerror(status: int) -> str:
    try:
        return lib().ssd_strerror(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def ssd_last_kernel() -> str:
    """The kernel the calling thread's last verify / cache / round call launched."""
    return lib().ssd_last_kernel().decode()


def version() -> str:
    return lib().ssd_version().decode()


def _check(status: int, where: str):
    if status != SSD_OK:
        raise SSDError(status, where)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data_as(ctypes.c_void_p)
    return ctypes.c_void_p(t.data_ptr())


def _dev(t: torch.Tensor, name: str, dtype=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _logit_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SSD_F32
    if t.dtype == torch.bfloat16:
        return SSD_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


# ---------------------------------------------------------------------------
# Host-only calls.
# ---------------------------------------------------------------------------

def ssd_workspace_size(B: int, K: int) -> int:
    return int(lib().ssd_workspace_size(int(B), int(K)))


def ssd_workspace_size_v(B: int, K: int, V: int, dtype: int, budget: int = 0) -> int:
    return int(lib().ssd_workspace_size_v(int(B), int(K), int(V), int(dtype), int(budget)))


def ssd_fanout(K: int, budget: int, a_p: float, r: float, V: int):
    """Geometric fan-out: (F [K+1], off [K+2]) as numpy int32 arrays."""
    F = np.empty(K + 1, np.int32)
    off = np.empty(K + 2, np.int32)
    _check(lib().ssd_fanout(int(K), int(budget), float(a_p), float(r), int(V), _ptr(F), _ptr(off)),
           "ssd_fanout")
    return F, off


def ssd_fanout_uniform(K: int, budget: int, V: int):
    """Uniform fan-out: (F [K+1], off [K+2]) as numpy int32 arrays."""
    F = np.empty(K + 1, np.int32)
    off = np.empty(K + 2, np.int32)
    _check(lib().ssd_fanout_uniform(int(K), int(budget), int(V), _ptr(F), _ptr(off)),
           "ssd_fanout_uniform")
    return F, off


def workspace(B: int, K: int, device=None, V: int | None = None, dtype: int | None = None,
              budget: int = 0) -> torch.Tensor:
    """A zero-filled workspace for B sequences of K drafted tokens; with V and dtype
    (and the cache budget) it also holds the slice kernel's regions."""
    if V is not None and dtype is not None:
        n = ssd_workspace_size_v(B, K, V, dtype, budget)
    else:
        n = ssd_workspace_size(B, K)
    if n == 0:
        raise ValueError("invalid workspace arguments")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def _workspace(ws, B, K, device, V=None, dtype=None, budget=0):
    if ws is None:
        ws = workspace(B, K, device, V, dtype, budget)
    _dev(ws, "workspace", torch.uint8)
    return ws


def _row_stride(t, name):
    """Elements between consecutive rows of a [B, R, V] logit tensor whose rows are
    contiguous and evenly spaced (a contiguous tensor, or a [..., :V] view of one
    with a longer row); raises for any other layout."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dim() != 3:
        raise ValueError(f"{name} must be [B, rows, V]")
    B, R, V = t.shape
    ld = t.stride(1) if R > 1 else (t.stride(0) if B > 1 else V)
    if t.stride(2) != 1 or ld < V or (R > 1 and B > 1 and t.stride(0) != R * ld):
        raise ValueError(f"{name} rows must be contiguous and evenly spaced")
    return int(ld)


def _shapes(tgt, drf, tokens, allow_ld=False):
    if tgt.dim() != 3 or drf.dim() != 3:
        raise ValueError("tgt must be [B, K+1, V] and drf [B, K or K+1, V]")
    if allow_ld:
        ld_t, ld_d = _row_stride(tgt, "tgt"), _row_stride(drf, "drf")
        if tgt.shape[1] == 1 and tgt.shape[0] == 1:
            ld_t = ld_d
        if drf.shape[1] == 1 and drf.shape[0] == 1:
            ld_d = ld_t
        if ld_t != ld_d:
            raise ValueError("tgt and drf must share one row stride")
    else:
        _dev(tgt, "tgt")
        _dev(drf, "drf")
        ld_t = int(tgt.shape[2])
    B, K1, V = tgt.shape
    K = K1 - 1
    if drf.shape[0] != B or drf.shape[2] != V or drf.dtype != tgt.dtype:
        raise ValueError("drf must match tgt in batch, vocabulary and dtype")
    _dev(tokens, "tokens", torch.int32)
    if tuple(tokens.shape) != (B, K):
        raise ValueError("tokens must be [B, K]")
    if allow_ld:
        return B, K, V, int(drf.shape[1]), ld_t
    return B, K, V, int(drf.shape[1])


def _opt(t, name, dtype):
    return None if t is None else _dev(t, name, dtype)


def _F_host(F):
    return np.ascontiguousarray(np.asarray(F, dtype=np.int32))


# ---------------------------------------------------------------------------
# Device calls.
# ---------------------------------------------------------------------------

def ssd_verify(tgt, drf, tokens, uniforms, temperature, reshape=None, *, accept_len=None,
               bonus=None, p_tok=None, q_tok=None, probs=True, workspace=None, dev_status=None,
               stream=None):
    """Verify one batch: returns dict(accept_len, bonus[, p_tok, q_tok]).  The logit
    tensors may be [..., :V] views of rows with a longer stride (same for both)."""
    B, K, V, drf_rows, ld = _shapes(tgt, drf, tokens, allow_ld=True)
    dev = tgt.device
    _dev(uniforms, "uniforms", torch.float32)
    _dev(temperature, "temperature", torch.float32)
    accept_len = accept_len if accept_len is not None else torch.empty(B, dtype=torch.int32, device=dev)
    bonus = bonus if bonus is not None else torch.empty(B, dtype=torch.int32, device=dev)
    if probs:
        p_tok = p_tok if p_tok is not None else torch.empty((B, K), dtype=torch.float32, device=dev)
        q_tok = q_tok if q_tok is not None else torch.empty((B, K), dtype=torch.float32, device=dev)
    ws = _workspace(workspace, B, K, dev, V, _logit_dtype(tgt))
    _opt(reshape, "reshape", torch.int32)
    _check(lib().ssd_verify_ld(
        _ptr(tgt), _ptr(drf), _logit_dtype(tgt), B, K, V, ld, drf_rows, _ptr(tokens), _ptr(uniforms),
        _ptr(temperature), _ptr(reshape), _ptr(accept_len), _ptr(bonus), _ptr(p_tok), _ptr(q_tok),
        _ptr(ws), ws.numel(), _ptr(_opt(dev_status, "dev_status", torch.int32)), _stream(stream)),
        "ssd_verify_ld")
    out = {"accept_len": accept_len, "bonus": bonus}
    if probs:
        out.update(p_tok=p_tok, q_tok=q_tok)
    return out


def ssd_build_cache(tgt, drf, tokens, temperature, F, budget, reshape=None, *, cache_tok=None,
                    workspace=None, dev_status=None, stream=None):
    """Speculation-cache keys: cache_tok [B, budget] int32 (segment k = top-F_k)."""
    B, K, V, drf_rows = _shapes(tgt, drf, tokens)
    dev = tgt.device
    _dev(temperature, "temperature", torch.float32)
    Fh = _F_host(F)
    cache_tok = cache_tok if cache_tok is not None else torch.full((B, budget), -1, dtype=torch.int32, device=dev)
    ws = _workspace(workspace, B, K, dev, V, _logit_dtype(tgt), int(budget))
    _check(lib().ssd_build_cache(
        _ptr(tgt), _ptr(drf), _logit_dtype(tgt), B, K, V, drf_rows, _ptr(tokens),
        _ptr(temperature), _ptr(_opt(reshape, "reshape", torch.int32)), _ptr(Fh), int(budget),
        _ptr(cache_tok), _ptr(ws), ws.numel(), _ptr(_opt(dev_status, "dev_status", torch.int32)),
        _stream(stream)), "ssd_build_cache")
    return cache_tok


def ssd_cache_lookup(cache_tok, F, accept_len, bonus, *, hit=None, slot=None, stream=None):
    """Hit test of the true outcome (a, t*): (hit [B] uint8, slot [B] int32)."""
    _dev(cache_tok, "cache_tok", torch.int32)
    B, budget = cache_tok.shape
    Fh = _F_host(F)
    K = len(Fh) - 1
    dev = cache_tok.device
    hit = hit if hit is not None else torch.empty(B, dtype=torch.uint8, device=dev)
    slot = slot if slot is not None else torch.empty(B, dtype=torch.int32, device=dev)
    _check(lib().ssd_cache_lookup(
        _ptr(cache_tok), B, K, budget, _ptr(Fh), _ptr(_dev(accept_len, "accept_len", torch.int32)),
        _ptr(_dev(bonus, "bonus", torch.int32)), _ptr(hit), _ptr(slot), _stream(stream)),
        "ssd_cache_lookup")
    return hit, slot


def ssd_backup_fill(hit, uniforms, V: int, next_tokens, *, stream=None):
    """Random-token backup for the sequences that missed: next_tokens [B, K] int32 is
    written in place where hit[b] == 0 (token floor(u * V)); returns next_tokens."""
    _dev(hit, "hit", torch.uint8)
    _dev(uniforms, "uniforms", torch.float32)
    _dev(next_tokens, "next_tokens", torch.int32)
    if uniforms.dim() != 2 or tuple(next_tokens.shape) != tuple(uniforms.shape) \
            or hit.shape != (uniforms.shape[0],):
        raise ValueError("uniforms and next_tokens must be [B, K] and hit [B]")
    B, K = uniforms.shape
    _check(lib().ssd_backup_fill(_ptr(hit), _ptr(uniforms), B, K, int(V), _ptr(next_tokens),
                                 _stream(stream)), "ssd_backup_fill")
    return next_tokens


def ssd_round(tgt, drf, tokens, uniforms, temperature, F, budget, reshape=None, *, out=None,
              probs=True, workspace=None, dev_status=None, stream=None):
    """One fused SSD round: verify + cache build + lookup.  Returns a dict of outputs.
    The logit tensors may be [..., :V] views of rows with a longer stride."""
    B, K, V, drf_rows, ld = _shapes(tgt, drf, tokens, allow_ld=True)
    dev = tgt.device
    _dev(uniforms, "uniforms", torch.float32)
    _dev(temperature, "temperature", torch.float32)
    Fh = _F_host(F)
    o = dict(out) if out is not None else {}
    if not probs:
        o.pop("p_tok", None)
        o.pop("q_tok", None)
    # allocate only what the caller did not supply (no work is enqueued otherwise)
    if "accept_len" not in o:
        o["accept_len"] = torch.empty(B, dtype=torch.int32, device=dev)
    if "bonus" not in o:
        o["bonus"] = torch.empty(B, dtype=torch.int32, device=dev)
    if probs and "p_tok" not in o:
        o["p_tok"] = torch.empty((B, K), dtype=torch.float32, device=dev)
    if probs and "q_tok" not in o:
        o["q_tok"] = torch.empty((B, K), dtype=torch.float32, device=dev)
    if "cache_tok" not in o:
        o["cache_tok"] = torch.full((B, budget), -1, dtype=torch.int32, device=dev)
    if "hit" not in o:
        o["hit"] = torch.empty(B, dtype=torch.uint8, device=dev)
    if "slot" not in o:
        o["slot"] = torch.empty(B, dtype=torch.int32, device=dev)
    ws = _workspace(workspace, B, K, dev, V, _logit_dtype(tgt), int(budget))
    _check(lib().ssd_round_ld(
        _ptr(tgt), _ptr(drf), _logit_dtype(tgt), B, K, V, ld, drf_rows, _ptr(tokens), _ptr(uniforms),
        _ptr(temperature), _ptr(_opt(reshape, "reshape", torch.int32)), _ptr(Fh), int(budget),
        _ptr(o["accept_len"]), _ptr(o["bonus"]), _ptr(o.get("p_tok")), _ptr(o.get("q_tok")),
        _ptr(o["cache_tok"]), _ptr(o["hit"]), _ptr(o["slot"]), _ptr(ws), ws.numel(),
        _ptr(_opt(dev_status, "dev_status", torch.int32)), _stream(stream)), "ssd_round_ld")
    return o


def _host(t, name: str, dtype=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise TypeError(f"{name} must be a host (CPU) tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def ssd_host_staging_size(dtype: int, B: int, K: int, V: int, budget: int) -> int:
    """Device bytes ssd_round_host needs for its copies of one round's inputs and outputs."""
    return int(lib().ssd_host_staging_size(int(dtype), int(B), int(K), int(V), int(budget)))


def ssd_round_host(tgt, drf, tokens, uniforms, temperature, F, budget, *, out=None, staging=None,
                   workspace=None, dev_status=None, stream=None, device=None):
    """ssd_round on host tensors (page-locked ones copy asynchronously): the inputs
    are copied to the device (the draft rows of sampled sequences only), the round
    runs and its results are copied back, all on `stream`.  Returns (outputs, h2d):
    a dict of host tensors accept_len, bonus, cache_tok, hit, slot -- valid once the
    stream has completed -- and the bytes copied to the device."""
    _host(tgt, "tgt")
    _host(drf, "drf", tgt.dtype)
    if tgt.dim() != 3 or drf.dim() != 3:
        raise ValueError("tgt must be [B, K+1, V] and drf [B, K, V]")
    B, K1, V = tgt.shape
    K = K1 - 1
    if tuple(drf.shape) != (B, K, V):
        raise ValueError("drf must be [B, K, V]")
    _host(tokens, "tokens", torch.int32)
    _host(uniforms, "uniforms", torch.float32)
    _host(temperature, "temperature", torch.float32)
    if tuple(tokens.shape) != (B, K) or tuple(uniforms.shape) != (B, K + 1) or tuple(temperature.shape) != (B,):
        raise ValueError("tokens [B, K], uniforms [B, K+1] and temperature [B] expected")
    dt = _logit_dtype(tgt)
    Fh = _F_host(F)
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    o = dict(out) if out is not None else {}
    shapes = {"accept_len": ((B,), torch.int32), "bonus": ((B,), torch.int32),
              "cache_tok": ((B, int(budget)), torch.int32), "hit": ((B,), torch.uint8),
              "slot": ((B,), torch.int32)}
    for k, (shp, dty) in shapes.items():
        if k not in o:
            o[k] = torch.empty(shp, dtype=dty).pin_memory()
        _host(o[k], k, dty)
    need = ssd_host_staging_size(dt, B, K, V, budget)
    if need == 0:
        raise ValueError("invalid sizes for ssd_round_host")
    if staging is None:
        staging = torch.empty(need, dtype=torch.uint8, device=dev)
    _dev(staging, "staging", torch.uint8)
    ws = _workspace(workspace, B, K, dev, V, dt, int(budget))
    moved = ctypes.c_size_t(0)
    _check(lib().ssd_round_host(
        _ptr(tgt), _ptr(drf), dt, B, K, V, _ptr(tokens), _ptr(uniforms), _ptr(temperature), _ptr(Fh),
        int(budget), _ptr(o["accept_len"]), _ptr(o["bonus"]), _ptr(o["cache_tok"]), _ptr(o["hit"]),
        _ptr(o["slot"]), _ptr(staging), staging.numel(), _ptr(ws), ws.numel(),
        _ptr(_opt(dev_status, "dev_status", torch.int32)), ctypes.c_void_p(ctypes.addressof(moved)),
        _stream(stream)), "ssd_round_host")
    return o, int(moved.value)


def _sigma_args(sigma_F, K, B, desc_out, dev):
    Fs = _F_host(sigma_F)
    if Fs.shape != (K,):
        raise ValueError("sigma_F must have K entries")
    desc_out = desc_out if desc_out is not None else torch.zeros((B * K, 4), dtype=torch.int32,
                                                                 device=dev)
    _dev(desc_out, "desc_out", torch.int32)
    if desc_out.numel() != B * K * 4:
        raise ValueError("desc_out must hold B*K descriptors")
    return Fs, desc_out


def ssd_verify_sigma(tgt, drf, tokens, uniforms, temperature, sigma_F, sigma_C, *, desc_out=None,
                     probs=True, workspace=None, dev_status=None, stream=None):
    """ssd_verify on sigma_{F_k,C} with the descriptors found in the same pass:
    returns dict(accept_len, bonus[, p_tok, q_tok], desc)."""
    B, K, V, drf_rows = _shapes(tgt, drf, tokens)
    dev = tgt.device
    _dev(uniforms, "uniforms", torch.float32)
    _dev(temperature, "temperature", torch.float32)
    Fs, desc_out = _sigma_args(sigma_F, K, B, desc_out, dev)
    accept_len = torch.empty(B, dtype=torch.int32, device=dev)
    bonus = torch.empty(B, dtype=torch.int32, device=dev)
    p_tok = torch.empty((B, K), dtype=torch.float32, device=dev) if probs else None
    q_tok = torch.empty((B, K), dtype=torch.float32, device=dev) if probs else None
    ws = _workspace(workspace, B, K, dev)
    _check(lib().ssd_verify_sigma(
        _ptr(tgt), _ptr(drf), _logit_dtype(tgt), B, K, V, drf_rows, _ptr(tokens), _ptr(uniforms),
        _ptr(temperature), _ptr(Fs), float(sigma_C), _ptr(desc_out), _ptr(accept_len), _ptr(bonus),
        _ptr(p_tok), _ptr(q_tok), _ptr(ws), ws.numel(),
        _ptr(_opt(dev_status, "dev_status", torch.int32)), _stream(stream)), "ssd_verify_sigma")
    out = {"accept_len": accept_len, "bonus": bonus, "desc": desc_out}
    if probs:
        out.update(p_tok=p_tok, q_tok=q_tok)
    return out


def ssd_round_sigma(tgt, drf, tokens, uniforms, temperature, sigma_F, sigma_C, F, budget, *,
                    desc_out=None, probs=True, workspace=None, dev_status=None, stream=None):
    """ssd_round on sigma_{F_k,C} with the descriptors found in the same pass: returns the
    outputs of ssd_round plus desc."""
    B, K, V, drf_rows = _shapes(tgt, drf, tokens)
    dev = tgt.device
    _dev(uniforms, "uniforms", torch.float32)
    _dev(temperature, "temperature", torch.float32)
    Fs, desc_out = _sigma_args(sigma_F, K, B, desc_out, dev)
    Fh = _F_host(F)
    o = {"accept_len": torch.empty(B, dtype=torch.int32, device=dev),
         "bonus": torch.empty(B, dtype=torch.int32, device=dev),
         "cache_tok": torch.full((B, budget), -1, dtype=torch.int32, device=dev),
         "hit": torch.empty(B, dtype=torch.uint8, device=dev),
         "slot": torch.empty(B, dtype=torch.int32, device=dev), "desc": desc_out}
    if probs:
        o["p_tok"] = torch.empty((B, K), dtype=torch.float32, device=dev)
        o["q_tok"] = torch.empty((B, K), dtype=torch.float32, device=dev)
    ws = _workspace(workspace, B, K, dev)
    _check(lib().ssd_round_sigma(
        _ptr(tgt), _ptr(drf), _logit_dtype(tgt), B, K, V, drf_rows, _ptr(tokens), _ptr(uniforms),
        _ptr(temperature), _ptr(Fs), float(sigma_C), _ptr(desc_out), _ptr(Fh), int(budget),
        _ptr(o["accept_len"]), _ptr(o["bonus"]), _ptr(o.get("p_tok")), _ptr(o.get("q_tok")),
        _ptr(o["cache_tok"]), _ptr(o["hit"]), _ptr(o["slot"]), _ptr(ws), ws.numel(),
        _ptr(_opt(dev_status, "dev_status", torch.int32)), _stream(stream)), "ssd_round_sigma")
    return o


def ssd_reshape_draft(drf, F, C, temperature_rows=None, *, want_q=False, desc=None, q_out=None,
                      dev_status=None, stream=None):
    """sigma_{F,C} descriptors of every draft row (drf [..., V] viewed as [rows, V]).

    Returns (desc [rows, 4] int32 holding {thr_val (fp32 bits), thr_id, F, C (fp32 bits)},
    q' [rows, V] fp32 or None)."""
    _dev(drf, "drf")
    V = int(drf.shape[-1])
    rows = drf.numel() // V
    dev = drf.device
    desc = desc if desc is not None else torch.empty((rows, 4), dtype=torch.int32, device=dev)
    if want_q:
        q_out = q_out if q_out is not None else torch.empty((rows, V), dtype=torch.float32, device=dev)
        _dev(temperature_rows, "temperature_rows", torch.float32)
    _check(lib().ssd_reshape_draft(
        _ptr(drf), _logit_dtype(drf), rows, V, _ptr(temperature_rows), int(F), float(C), _ptr(desc),
        _ptr(q_out if want_q else None), _ptr(_opt(dev_status, "dev_status", torch.int32)),
        _stream(stream)), "ssd_reshape_draft")
    return desc, (q_out if want_q else None)


def ssd_draft_cache(drf, tokens, F, budget, C=1.0, *, cache=True, reshape=False, cache_tok=None,
                    desc=None, dev_status=None, stream=None):
    """Draft-side cache keys and sigma_{F_k,C} descriptors from drf [B, K+1, V].

    Returns (cache_tok [B, budget] int32 or None, desc [B*K, 4] int32 or None); tokens
    [B, K] int32 (the drafted tokens left out of their segment) may be None."""
    _dev(drf, "drf")
    if drf.dim() != 3:
        raise ValueError("drf must be [B, K+1, V]")
    B, K1, V = drf.shape
    K = K1 - 1
    Fh = _F_host(F)
    if len(Fh) != K + 1:
        raise ValueError("F must have K+1 entries")
    dev = drf.device
    if tokens is not None:
        _dev(tokens, "tokens", torch.int32)
        if tuple(tokens.shape) != (B, K):
            raise ValueError("tokens must be [B, K]")
    if cache:
        cache_tok = cache_tok if cache_tok is not None else torch.empty(
            (B, budget), dtype=torch.int32, device=dev)
        _dev(cache_tok, "cache_tok", torch.int32)
        if tuple(cache_tok.shape) != (B, budget):
            raise ValueError("cache_tok must be [B, budget]")
    else:
        cache_tok = None
    if reshape:
        desc = desc if desc is not None else torch.empty((B * K, 4), dtype=torch.int32, device=dev)
        _dev(desc, "desc", torch.int32)
        if desc.numel() != B * K * 4:
            raise ValueError("desc must hold B*K descriptors")
    else:
        desc = None
    _check(lib().ssd_draft_cache(
        _ptr(drf), _logit_dtype(drf), B, K, V, _ptr(tokens), _ptr(Fh), int(budget), float(C),
        _ptr(cache_tok), _ptr(desc), _ptr(_opt(dev_status, "dev_status", torch.int32)),
        _stream(stream)), "ssd_draft_cache")
    return cache_tok, desc


def desc_fields(desc: torch.Tensor):
    """Decodes reshape descriptors: (thr_val fp32, thr_id int32, F int32, C fp32) tensors."""
    return desc[:, 0].view(torch.float32), desc[:, 1], desc[:, 2], desc[:, 3].view(torch.float32)
