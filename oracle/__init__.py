"""CPU oracle for query-aware page selection + masked sparse attention (fp64).

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
benchmark's CPU-baseline leg, never by the library.  The arithmetic lives in
``oracle.c`` (plain C, fp64); this module only compiles it with gcc, loads it
with ctypes and marshals numpy arrays.  It shares no code with the CUDA path.

All functions work on logical token order for ONE (sequence, KV head) unless
stated otherwise; inputs are widened to float64 before the call.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain gcc, -O2, no CUDA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_page_bounds.argtypes = [ctypes.c_int] * 3 + [_D, _D, _D]
            lib.oracle_page_bounds_by_appends.argtypes = [ctypes.c_int] * 3 + [
                _D, ctypes.c_int, _I, _D, _D]
            lib.oracle_page_scores.argtypes = [ctypes.c_int] * 3 + [_D, _D, _D, _D]
            lib.oracle_select_pages.argtypes = [ctypes.c_int, _D, ctypes.c_int, _I]
            lib.oracle_select_pages.restype = ctypes.c_int
            lib.oracle_attention.argtypes = [ctypes.c_int] * 4 + [
                _D, _D, _D, ctypes.c_int, _I, ctypes.c_double, _D]
            lib.oracle_decode_unit.argtypes = [ctypes.c_int] * 4 + [
                _D, _D, _D, _D, _D, ctypes.c_int, ctypes.c_double, _D, _I, _D]
            lib.oracle_decode_unit.restype = ctypes.c_int
            lib.oracle_page_attention_mass.argtypes = [ctypes.c_int] * 4 + [_D, _D, ctypes.c_double, _D]
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_ubyte]
            lib.oracle_e4m3_decode.restype = ctypes.c_float
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_encode.restype = ctypes.c_ubyte
            _F = ctypes.POINTER(ctypes.c_float)
            _U = ctypes.POINTER(ctypes.c_ubyte)
            lib.oracle_fp8_append_replay.argtypes = [ctypes.c_int] * 3 + [_F, ctypes.c_int, _I, _U, _F, _U, _U]
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float64)


def _i32(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.int32)


def _dp(a: np.ndarray):
    return a.ctypes.data_as(_D)


def _ip(a: np.ndarray):
    return a.ctypes.data_as(_I)


def num_pages(L: int, P: int) -> int:
    return (int(L) + int(P) - 1) // int(P)


def page_bounds(K, P: int) -> Tuple[np.ndarray, np.ndarray]:
    """Per-page per-channel (min, max) of the keys K [L, d]; returns lo, hi [N, d]."""
    K = _f64(K)
    L, d = K.shape
    N = num_pages(L, P)
    lo = np.empty((N, d))
    hi = np.empty((N, d))
    if N:
        _load().oracle_page_bounds(L, d, P, _dp(K), _dp(lo), _dp(hi))
    return lo, hi


def page_bounds_by_appends(K, P: int, chunk_lens: Sequence[int]) -> Tuple[np.ndarray, np.ndarray]:
    """Boxes maintained chunk by chunk as an append-time builder would."""
    K = _f64(K)
    L, d = K.shape
    N = num_pages(L, P)
    lo = np.full((N, d), np.nan)
    hi = np.full((N, d), np.nan)
    ch = _i32(chunk_lens)
    if N:
        _load().oracle_page_bounds_by_appends(L, d, P, _dp(K), len(ch), _ip(ch), _dp(lo), _dp(hi))
    return lo, hi


def page_scores(q, lo, hi) -> np.ndarray:
    """Score of every page: max_g sum_c max(q[g,c]*lo[p,c], q[g,c]*hi[p,c])."""
    q, lo, hi = _f64(q), _f64(lo), _f64(hi)
    if q.ndim == 1:
        q = q[None]
    G, d = q.shape
    N = lo.shape[0]
    s = np.empty(N)
    if N:
        _load().oracle_page_scores(G, d, N, _dp(q), _dp(lo), _dp(hi), _dp(s))
    return s


def select_pages(scores, k: int) -> np.ndarray:
    """Kept logical page ids (ascending) for a budget of k pages."""
    s = _f64(scores)
    N = s.shape[0]
    out = np.empty(max(N, 1), dtype=np.int32)
    n = _load().oracle_select_pages(N, _dp(s), int(k), _ip(out))
    return out[:n].copy()


def attention(q, K, V, L: int, P: int, pages, scale: Optional[float] = None) -> np.ndarray:
    """Masked softmax attention of q [G, d] over the tokens of ``pages`` below L."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    if q.ndim == 1:
        q = q[None]
    G, d = q.shape
    pg = _i32(pages)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.empty((G, d))
    _load().oracle_attention(G, d, int(L), int(P), _dp(q), _dp(K), _dp(V), len(pg),
                             _ip(pg if len(pg) else np.zeros(1, np.int32)), float(scale),
                             _dp(out))
    return out


def dense_attention(q, K, V, L: int, P: int, scale: Optional[float] = None) -> np.ndarray:
    return attention(q, K, V, L, P, np.arange(num_pages(L, P)), scale)


def decode_unit(q, K, V, lo, hi, L: int, P: int, k: int, scale: Optional[float] = None):
    """One decode step of one (sequence, KV head): scores, kept ids, output [G, d]."""
    q, K, V, lo, hi = _f64(q), _f64(K), _f64(V), _f64(lo), _f64(hi)
    if q.ndim == 1:
        q = q[None]
    G, d = q.shape
    N = num_pages(L, P)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    scores = np.empty(max(N, 1))
    sel = np.empty(max(N, 1), dtype=np.int32)
    out = np.empty((G, d))
    n = _load().oracle_decode_unit(G, d, int(L), int(P), _dp(q), _dp(K), _dp(V), _dp(lo),
                                   _dp(hi), int(k), float(scale), _dp(scores), _ip(sel),
                                   _dp(out))
    return scores[:N].copy(), sel[:n].copy(), out


def page_attention_mass(q, K, L: int, P: int, scale: Optional[float] = None) -> np.ndarray:
    """Per-page share of the dense attention mass (mean over the G heads)."""
    q, K = _f64(q), _f64(K)
    if q.ndim == 1:
        q = q[None]
    G, d = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    N = num_pages(L, P)
    mass = np.zeros(max(N, 1))
    _load().oracle_page_attention_mass(G, d, int(L), int(P), _dp(q), _dp(K), float(scale), _dp(mass))
    return mass[:N].copy()


def page_hit_rate(mass, selected, k: int) -> Tuple[int, float, float]:
    """Compare a selection with the page mass of one (sequence, KV head).

    T = the k pages of largest mass, equal masses taken in page order (a stable
    sort of the negated masses).  Returns (|first k selected ids ∩ T|, mass of
    the selected pages, mass of T).
    """
    mass = _f64(mass)
    top = np.argsort(-mass, kind="stable")[:k]
    sel = np.asarray(selected, dtype=np.int64)[:k]
    in_top = np.zeros(len(mass), dtype=bool)
    in_top[top] = True
    return int(in_top[sel].sum()), float(mass[sel].sum()), float(mass[top].sum())


# ------------------------------------------------------------------ FP8 KV

def e4m3_decode(codes) -> np.ndarray:
    """Values (float32) of E4M3 codes."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    table = np.array([lib.oracle_e4m3_decode(i) for i in range(256)], dtype=np.float32)
    return table[c]


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 codes (ties to even, finite overflow saturates, -0 -> +0)."""
    lib = _load()
    x = np.asarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    flat, of = x.reshape(-1), out.reshape(-1)
    for i in range(flat.size):
        of[i] = lib.oracle_e4m3_encode(float(flat[i]))
    return out


def fp8_append_replay(X, P: int, chunk_lens: Sequence[int]):
    """Quantized appends of one (sequence, KV head) tensor X [L, d] (fp32
    values), chunk by chunk.  Returns (codes [L, d] uint8, amax [N] float32,
    lo [N, d] uint8, hi [N, d] uint8)."""
    X = np.ascontiguousarray(X, dtype=np.float32)
    L, d = X.shape
    N = num_pages(L, P)
    ch = _i32(chunk_lens)
    codes = np.zeros((max(L, 1), d), dtype=np.uint8)
    amax = np.zeros(max(N, 1), dtype=np.float32)
    lo = np.zeros((max(N, 1), d), dtype=np.uint8)
    hi = np.zeros((max(N, 1), d), dtype=np.uint8)
    F = ctypes.POINTER(ctypes.c_float)
    U = ctypes.POINTER(ctypes.c_ubyte)
    _load().oracle_fp8_append_replay(int(L), int(d), int(P), X.ctypes.data_as(F), len(ch),
                                     _ip(ch if len(ch) else np.zeros(1, np.int32)),
                                     codes.ctypes.data_as(U), amax.ctypes.data_as(F),
                                     lo.ctypes.data_as(U), hi.ctypes.data_as(U))
    return codes[:L].copy(), amax[:N].copy(), lo[:N].copy(), hi[:N].copy()


def fp8_scale(amax) -> np.ndarray:
    """Per-page scale amax / 448 as the fp32 division computes it."""
    return (np.asarray(amax, dtype=np.float32) / np.float32(448.0)).astype(np.float32)


def fp8_dequant(codes, scale_per_row) -> np.ndarray:
    """Exact values code * s (float64: a 4-bit times a 24-bit significand)."""
    return e4m3_decode(codes).astype(np.float64) * np.asarray(scale_per_row, dtype=np.float64)[..., None]


def run_units(fn, items, threads: int = 1):
    """Map ``fn`` over independent (sequence, KV head) units; ctypes drops the GIL
    during each C call, so threads run the C code in parallel."""
    if threads <= 1:
        return [fn(it) for it in items]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(fn, items))
