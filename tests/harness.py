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


def check_selection(gpu_sel: np.ndarray, gpu_scores: Optional[np.ndarray], o_scores: np.ndarray,
                    o_sel: np.ndarray, k: int, tol: np.ndarray):
    """Assert the GPU's kept set equals the oracle's outside the tie band.

    Returns True when the two sets are identical."""
    N = len(o_scores)
    kept = gpu_sel[gpu_sel >= 0]
    assert np.all(np.diff(kept) > 0), "ids not strictly ascending"
    assert len(kept) == len(o_sel), (len(kept), len(o_sel))
    assert np.all(gpu_sel[len(kept):] == -1)
    assert kept.min() >= 0 and kept.max() < N
    if N >= 1:
        assert 0 in kept and (N - 1) in kept
    if np.array_equal(kept, o_sel):
        return True
    # sets differ: only allowed inside the band of scores tied with the boundary
    cand = np.arange(1, N - 1)
    kc = len(o_sel) - 2
    order = cand[np.lexsort((cand, -o_scores[cand]))]
    s_k = o_scores[order[kc - 1]]
    s_k1 = o_scores[order[kc]] if kc < len(order) else -np.inf
    band = np.maximum(TIE_REL * abs(s_k), 2 * tol.max())
    assert s_k - s_k1 <= band, "boundary scores %r, %r are not tied but sets differ" % (s_k, s_k1)
    for p in set(kept.tolist()) ^ set(o_sel.tolist()):
        assert abs(o_scores[p] - s_k) <= band + abs(s_k - s_k1), p
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
