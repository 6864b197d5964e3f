"""CPU model of the selection kernel's top-k (the digit narrowing of
select_from_scores), checked against a plain sort.

The kernel finds tau, the key of the (k-2)-th best candidate, from 1024-bin
histograms of 10-bit digits; in each pass one warp finds the bin holding the
wanted rank: every lane sums 32 consecutive bins (descending digits), a warp
scan over the lane totals names the holding lane, and that lane walks its 32
bins from the top.  This file restates those steps in Python, with the lane
arithmetic of the kernel, and checks that the two-level search agrees with a
walk over all bins and that the selection it leads to is the top-k of a sort
(ties to the lower page index).

The kept set is what "TinyServe: Query-Aware Cache Selection for Efficient
LLM Serving", 方法详解 / 关键设计, asks for: the pages whose bounding-box
scores are highest.
"""
import struct

import numpy as np
import pytest

BINS = 1024
LANES = 32
BPL = BINS // LANES


def rank_key(f: float) -> int:
    """Order-preserving uint32 image of an fp32 score (larger first; -0 == +0; NaN lowest)."""
    if f != f:
        return 0
    if f == 0.0:
        f = 0.0
    u = struct.unpack("<I", struct.pack("<f", f))[0]
    return (~u & 0xFFFFFFFF) if (u & 0x80000000) else (u | 0x80000000)


def digit_by_walk(hist, need):
    """Bin holding rank `need` (1 = largest digit first): a walk from the top."""
    run = 0
    for b in range(BINS - 1, -1, -1):
        if run + hist[b] >= need:
            return b, run, hist[b]
        run += hist[b]
    return None


def digit_by_lanes(hist, need):
    """The same bin found as the kernel's warp does: lane totals and their scan
    name the holding lane, which walks its own 32 bins."""
    tot = [sum(hist[BINS - BPL * (l + 1):BINS - BPL * l]) for l in range(LANES)]
    incl = list(np.cumsum(tot))
    excl = [incl[l] - tot[l] for l in range(LANES)]
    for lane in range(LANES):
        if excl[lane] < need <= incl[lane]:
            top = BINS - BPL * lane
            run = excl[lane]
            for j in range(1, BPL + 1):
                c = hist[top - j]
                if run + c >= need:
                    return top - j, run, c
                run += c
    return None


def model_tau(cand_keys, kc, nt=128, passes=None):
    """tau as the kernel narrows it down (histogram passes, then a gather of <= nt keys).
    `passes`, if a list, receives the number of histogram passes."""
    kmin, kmax = min(cand_keys), max(cand_keys)
    if kmin == kmax:
        return kmax
    hb = (kmin ^ kmax).bit_length() - 1
    pmask = 0 if hb == 31 else (~((2 << hb) - 1)) & 0xFFFFFFFF
    prefix = kmax & pmask
    need, low = kc, hb + 1
    while True:
        shift = low - 10 if low > 10 else 0
        dmask = (1 << (low - shift)) - 1
        hist = [0] * BINS
        for key in cand_keys:
            if key & pmask == prefix:
                hist[(key >> shift) & dmask] += 1
        found = digit_by_lanes(hist, need)
        assert found == digit_by_walk(hist, need)
        digit, above, cnt = found
        need -= above
        prefix |= digit << shift
        pmask |= dmask << shift
        low = shift
        if passes is not None:
            passes.append(1)
        if low == 0 or cnt <= nt:
            break
    if low == 0:
        return prefix
    gathered = [key for key in cand_keys if key & pmask == prefix]
    assert len(gathered) == cnt
    for v in gathered:
        gt = sum(w > v for w in gathered)
        eq = sum(w == v for w in gathered)
        if gt < need <= gt + eq:
            return v
    raise AssertionError("no key of the wanted rank")


def model_select(scores, k, nt=128, passes=None):
    """Kept page ids (ascending) of one unit as the kernel chooses them."""
    n = len(scores)
    if k >= n:
        return list(range(n))
    kc = k - 2
    if kc == 0:
        return [0, n - 1]
    keys = [rank_key(float(s)) for s in scores]
    tau = model_tau(keys[1:n - 1], kc, nt, passes)
    above = sum(key > tau for key in keys[1:n - 1])
    quota = kc - above
    kept, eq = [0], 0
    for i in range(1, n - 1):
        if keys[i] > tau:
            kept.append(i)
        elif keys[i] == tau:
            if eq < quota:
                kept.append(i)
            eq += 1
    kept.append(n - 1)
    return kept


def sort_select(scores, k):
    """Top-k by a stable sort: forced pages 0 and N-1, the rest by score, ties to the lower index."""
    n = len(scores)
    if k >= n:
        return list(range(n))
    keys = [rank_key(float(s)) for s in scores]
    cand = sorted(range(1, n - 1), key=lambda i: (-keys[i], i))
    return sorted([0, n - 1] + cand[:k - 2])


@pytest.mark.parametrize("seed", range(6))
def test_lane_search_matches_the_walk(seed):
    rng = np.random.default_rng(seed)
    for _ in range(200):
        hist = [0] * BINS
        nz = rng.integers(1, 60)
        for b in rng.integers(0, BINS, size=nz):
            hist[int(b)] += int(rng.integers(1, 40))
        total = sum(hist)
        for need in {1, total, int(rng.integers(1, total + 1)), int(rng.integers(1, total + 1))}:
            assert digit_by_lanes(hist, need) == digit_by_walk(hist, need)


def test_lane_search_single_bin_and_lane_edges():
    for b in (0, 31, 32, 511, 992, 1023):
        hist = [0] * BINS
        hist[b] = 5
        for need in (1, 3, 5):
            assert digit_by_lanes(hist, need) == (b, 0, 5)
    hist = [1] * BINS
    for need in (1, 32, 33, 1000, 1024):
        assert digit_by_lanes(hist, need) == digit_by_walk(hist, need) == (BINS - need, need - 1, 1)


@pytest.mark.parametrize("kind", ["normal", "integers", "few_values", "signed"])
def test_model_selection_equals_sort(kind):
    rng = np.random.default_rng(7)
    for trial in range(40):
        n = int(rng.integers(3, 700))
        k = int(rng.integers(2, n + 2))
        if kind == "normal":
            s = rng.normal(20.0, 3.0, n)
        elif kind == "integers":
            s = np.round(rng.normal(20.0, 3.0, n))
        elif kind == "few_values":
            s = rng.choice([-1.5, 0.0, -0.0, 2.25, 7.0], n)
        else:
            s = rng.normal(0.0, 1e-3, n) * rng.choice([1.0, 1e6], n)
        s = s.astype(np.float32)
        assert model_select(list(s), k) == sort_select(list(s), k), (kind, trial, n, k)


def test_model_selection_needs_a_second_pass():
    # keys that differ up to bit 13: the first pass takes bits 4-13, and 400
    # keys share one such digit (more than the 128 threads gather), so a second
    # pass over bits 0-3 decides; the other keys spread over other digits
    rng = np.random.default_rng(3)
    one = struct.unpack("<I", struct.pack("<f", 20.0))[0]
    offs = [0x2A0 + int(v) for v in rng.integers(0, 16, 400)] + [int(v) for v in rng.integers(0, 1 << 14, 300)]
    rng.shuffle(offs)
    s = [struct.unpack("<f", struct.pack("<I", one + o))[0] for o in offs]
    keys = [rank_key(v) for v in s]
    assert (min(keys) ^ max(keys)).bit_length() == 14
    most = 0
    for k in (3, 50, 200, 350, 500, 698, 702):
        passes = []
        assert model_select(s, k, passes=passes) == sort_select(s, k)
        most = max(most, len(passes))
    assert most == 2
