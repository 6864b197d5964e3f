"""Shared helpers of the GPU parity tests.

A `Case` holds one seeded workload twice: as logical host arrays (what the
oracle reads, widened to float64) and as a device paged cache filled through
the library's own append kernel (what the CUDA path reads).  Nothing here
computes any part of the method; comparisons and tolerances live in the tests.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np
import torch

import oracle
from query_aware_sparse_append_gb300 import paged
from query_aware_sparse_append_gb300 import workloads as W

TORCH_DTYPE = paged.TORCH_DTYPE

# attention outputs: |gpu - oracle| <= ATOL + RTOL * |oracle|
ATOL, RTOL = 2e-3, 1e-2
# two scores closer than this (relative) are a tie for the selection check
TIE_REL = 1e-5


to_torch = paged.to_torch




def from_torch(t: torch.Tensor, dtype: str) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


class Case(paged.DeviceWorkload):
    """A DeviceWorkload plus the oracle's view of it (logical float64 arrays)."""

    @property
    def G(self):
        return self.cfg.group

    @property
    def bt(self):
        return self.block_table

    def k64(self, b, h):
        return W.widen(self.seqs[b].k[:, h], self.cfg.dtype)

    def v64(self, b, h):
        return W.widen(self.seqs[b].v[:, h], self.cfg.dtype)

    def q64(self, b, h):
        G = self.G
        return W.widen(self.seqs[b].q[h * G:(h + 1) * G], self.cfg.dtype)


def make_case(cfg: W.Workload, seed: int = 0, batch: Optional[int] = None, lens=None,
              budgets=None, shuffle: bool = True, reserve_tokens: int = 0, device: bool = True,
              append_chunks: Optional[List[int]] = None, poison: bool = True) -> Case:
    """Generate the workload and (optionally) load it into a device cache.

    poison (default on): pools and boxes start as NaN, so any read of a slot or
    box that the method must not use shows up in the results.
    """
    wl = paged.generate(cfg, seed=seed, batch=batch, lens=lens, budgets=budgets,
                        shuffle=shuffle, reserve_tokens=reserve_tokens)
    case = Case(**{f.name: getattr(wl, f.name) for f in dataclasses.fields(wl)})
    if device:
        paged.load(case, poison=poison, append_chunks=append_chunks)
    return case


def chunk_lens(L: int, append_chunks: Optional[List[int]]) -> List[int]:
    """The append sizes paged.load uses for a sequence of L tokens."""
    out, done = [], 0
    for c in (append_chunks or [L]):
        t = min(L - done, c)
        if t > 0:
            out.append(t)
            done += t
    return out


def fp8_unit(case: Case, b: int, h: int, append_chunks: Optional[List[int]] = None):
    """The oracle's FP8 cache of one (sequence, KV head), replaying the appends:
    codes, amax and boxes of K and V, and the exact dequantized values."""
    P = case.cfg.page_size
    L = int(case.lens[b])
    ch = chunk_lens(L, append_chunks)
    kc, ka, lo, hi = oracle.fp8_append_replay(case.k64(b, h).astype(np.float32), P, ch)
    vc, va, _, _ = oracle.fp8_append_replay(case.v64(b, h).astype(np.float32), P, ch)
    sk, sv = oracle.fp8_scale(ka), oracle.fp8_scale(va)
    tok_page = np.arange(L) // P
    return dict(k_codes=kc, k_amax=ka, lo=lo, hi=hi, v_codes=vc, v_amax=va,
                K=oracle.fp8_dequant(kc, sk[tok_page]), V=oracle.fp8_dequant(vc, sv[tok_page]),
                LO=oracle.fp8_dequant(lo, sk), HI=oracle.fp8_dequant(hi, sk))


def build_device(case: Case, append_chunks=None, poison=True):
    return paged.load(case, poison=poison, append_chunks=append_chunks)


def score_tolerance(q64: np.ndarray, lo: np.ndarray, hi: np.ndarray) -> np.ndarray:
    """Bound on |fp32 score - exact score| per page.

    Every product of two stored 16-bit values is exact in fp32 (and the fp32
    path rounds each product once), so the error is the fp32 summation error of
    2d terms: at most 2d * 2^-23 * sum_c |term| (twice the textbook gamma_n
    bound, allowing for an accumulator that truncates instead of rounding).
    """
    terms = np.maximum(q64[:, None, :] * lo[None], q64[:, None, :] * hi[None])  # [G, N, d]
    mag = np.abs(terms).sum(axis=-1).max(axis=0)
    d = q64.shape[-1]
    return 2 * d * 2.0 ** -23 * mag + 1e-30


# Tally of the selection checks of this process, printed at the end of the
# test session: how many units had identical sets, how many differed only
# inside the 1e-5 relative tie band, and how many differed by more than that
# but within the fp32 summation bound of the pages involved.
SEL_STATS = {"units": 0, "identical": 0, "tie_band": 0, "fp32_band": 0}


def check_selection(gpu_sel: np.ndarray, gpu_scores: Optional[np.ndarray], o_scores: np.ndarray,
                    o_sel: np.ndarray, k: int, tol: np.ndarray):
    """Assert the GPU's kept set equals the oracle's outside the tie band.

    The kept sets must be identical unless the pages that differ are tied.
    For every page a the oracle keeps and the GPU drops, and every page b the
    GPU keeps and the oracle drops, the oracle's fp64 scores must satisfy
        s_a - s_b <= 1e-5 * |s_k|            (the tie rule; s_k = the k-th
                                              best candidate's score), or
        s_a - s_b <= tol[a] + tol[b]         (the fp32 summation bounds of
                                              those two pages: their fp32
                                              scores can order them either way).
    Units decided by the second clause are counted in SEL_STATS["fp32_band"].

    Returns True when the two sets are identical."""
    N = len(o_scores)
    kept = gpu_sel[gpu_sel >= 0]
    assert np.all(np.diff(kept) > 0), "ids not strictly ascending"
    assert len(kept) == len(o_sel), (len(kept), len(o_sel))
    assert np.all(gpu_sel[len(kept):] == -1)
    assert kept.min() >= 0 and kept.max() < N
    if N >= 1:
        assert 0 in kept and (N - 1) in kept
    SEL_STATS["units"] += 1
    if np.array_equal(kept, o_sel):
        SEL_STATS["identical"] += 1
        return True
    cand = np.arange(1, N - 1)
    kc = len(o_sel) - 2
    order = cand[np.lexsort((cand, -o_scores[cand]))]
    s_k = o_scores[order[kc - 1]]
    rel = TIE_REL * abs(s_k)
    dropped = sorted(set(o_sel.tolist()) - set(kept.tolist()))
    added = sorted(set(kept.tolist()) - set(o_sel.tolist()))
    widened = False
    for a in dropped:
        for b in added:
            gap = o_scores[a] - o_scores[b]
            if gap <= rel:
                continue
            assert gap <= tol[a] + tol[b], (
                "kept sets differ outside the tie band: oracle keeps page %d (score %r), GPU keeps "
                "page %d (score %r); gap %g > max(%g, %g)" % (a, o_scores[a], b, o_scores[b], gap, rel,
                                                              tol[a] + tol[b]))
            widened = True
    SEL_STATS["fp32_band" if widened else "tie_band"] += 1
    if gpu_scores is not None:
        # the GPU's own ranking must produce exactly its set
        g_order = cand[np.lexsort((cand, -gpu_scores[cand]))]
        assert np.array_equal(np.sort(np.concatenate([[0, N - 1], g_order[:kc]])), kept)
    return False


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str = "output"):
    err = np.abs(gpu - ref)
    lim = ATOL + RTOL * np.abs(ref)
    bad = err > lim
    assert not bad.any(), "%s: %d of %d elements outside tolerance; worst %g at %s (gpu %g, ref %g)" % (
        what, int(bad.sum()), bad.size, float((err - lim).max()), np.unravel_index(np.argmax(err - lim), err.shape),
        float(gpu.flat[np.argmax(err - lim)]), float(ref.flat[np.argmax(err - lim)]))


def gpu_out64(out: torch.Tensor, dtype: str) -> np.ndarray:
    return W.widen(from_torch(out, dtype), dtype)


def all_units(case):
    return [(b, h) for b in range(case.cfg.batch) for h in range(case.cfg.num_kv_heads)]


def check_units(case, out, sel, scores, units, check_bounds=True):
    """Compare the GPU's decode step with the oracle on the given (sequence,
    KV head) units: page boxes exactly, scores within the fp32 bound (when the
    GPU wrote them), kept sets with check_selection, outputs with assert_close
    (on the GPU's own set when a tie let the two sets differ).  Returns the
    number of units whose kept sets were identical."""
    cfg = case.cfg
    P = cfg.page_size
    out64 = gpu_out64(out, cfg.dtype)
    sel = sel.cpu().numpy()
    scores = scores.cpu().numpy() if scores is not None else None
    bounds = from_torch(case.cache.page_bounds, cfg.dtype) if check_bounds else None
    n_equal = 0
    for b, h in units:
        L = int(case.lens[b])
        N = -(-L // P)
        K = case.k64(b, h)
        lo, hi = oracle.page_bounds(K, P)
        if check_bounds and N:
            phys = case.plan.block_table[b, :N]
            glo = W.widen(bounds[phys, h, 0], cfg.dtype)
            ghi = W.widen(bounds[phys, h, 1], cfg.dtype)
            assert np.array_equal(glo, lo) and np.array_equal(ghi, hi), (b, h)
        q64 = case.q64(b, h)
        o_s, o_sel, o_out = oracle.decode_unit(q64, K, case.v64(b, h), lo, hi, L, P,
                                               int(case.budgets[b]))
        if N == 0:
            assert np.all(sel[b, h] == -1)
            assert np.all(out64[b, h * case.G:(h + 1) * case.G] == 0)
            continue
        k_eff = len(o_sel)
        tol = score_tolerance(q64, lo, hi)
        g_s = None
        if scores is not None:
            g_s = scores[b, h, :N].astype(np.float64)
            if k_eff < N:
                assert np.all(np.abs(g_s - o_s) <= tol), (b, h, np.max(np.abs(g_s - o_s) - tol))
        same = check_selection(sel[b, h], g_s if k_eff < N else None, o_s, o_sel, k_eff, tol)
        ref = o_out if same else oracle.attention(q64, K, case.v64(b, h), L, P,
                                                  sel[b, h][sel[b, h] >= 0])
        n_equal += same
        assert_close(out64[b, h * case.G:(h + 1) * case.G], ref, "out b=%d h=%d" % (b, h))
    return n_equal
