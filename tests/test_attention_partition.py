"""CPU model of the attention kernel's work split, checked for every grid size
the library launches (1 .. SM count; small batches get fewer CTAs than SMs).

The kernel flattens all kept (unit, page) pairs unit-major (unit = sequence b,
KV head h; sequence b contributes Hkv units of cnt_b pages each), gives CTA c of
C the pages whose weighted position g + W0*(u+1) lies in [c*V/C, (c+1)*V/C),
V = T + W0*U (every unit adds W0 page-equivalents of work), walks it rotated (first the part of its last
unit that starts inside the range, then the rest), writes whole units directly
and, for a unit cut by a range boundary, a partial to slot unit + c plus a page
ticket; the CTA whose ticket completes the unit merges the partials of CTAs
cta_of(first page) .. cta_of(last page).  The single-launch form also lets the
CTA holding a unit's first page select that unit.  This model restates that
index arithmetic (range_start, cta_of, locate, the rotation) and checks:

* the segments of all CTAs tile [0, T) exactly, each inside one unit;
* a CTA has at most one segment per unit, and a unit handled whole by one CTA
  is written directly (no ticket, no slot);
* partial slots unit + c are distinct and below U + C (the workspace holds
  U + SM-count slots);
* every split unit's tickets add up to its page count, so exactly one CTA
  completes it, and the merge range is exactly the CTAs that wrote partials;
* every unit with pages has exactly one selecting CTA, which holds its first
  page;
* the grid for small batches is at least 1 and at most the SM count.
"""
import random

import pytest


class Split:
    def __init__(self, cnts, Hkv, C, W0=0):
        self.B, self.Hkv, self.C, self.cnts, self.W0 = len(cnts), Hkv, C, cnts, W0
        self.prefix = [0]
        for x in cnts:
            self.prefix.append(self.prefix[-1] + x)
        self.T = Hkv * self.prefix[-1]
        self.U = self.B * Hkv
        self.V = self.T + W0 * self.U   # weighted work: pages + W0 per unit

    def unit_bounds(self, u):
        b, h = divmod(u, self.Hkv)
        cnt = self.cnts[b]
        us = self.Hkv * self.prefix[b] + h * cnt
        return us, us + cnt

    def range_start(self, c):
        """First page whose weighted position g + W0*(u+1) reaches c*V/C."""
        if c >= self.C:
            return self.T
        V = c * self.V // self.C
        lo, hi = 0, self.U
        while lo < hi:          # first unit u with ue(u) + W0*(u+1) > V
            mid = (lo + hi) >> 1
            if self.unit_bounds(mid)[1] + self.W0 * (mid + 1) > V:
                hi = mid
            else:
                lo = mid + 1
        if lo >= self.U:
            return self.T
        return max(self.unit_bounds(lo)[0], V - self.W0 * (lo + 1))

    def cta_of(self, g):
        b, h, _, _ = self.locate(g)
        v = g + self.W0 * (b * self.Hkv + h + 1)
        return ((v + 1) * self.C - 1) // self.V

    def locate(self, g):
        lo, hi = 0, self.B - 1
        while lo < hi:   # largest b with Hkv * prefix[b] <= g
            mid = (lo + hi + 1) >> 1
            if self.Hkv * self.prefix[mid] <= g:
                lo = mid
            else:
                hi = mid - 1
        b = lo
        cnt = self.prefix[b + 1] - self.prefix[b]
        off = g - self.Hkv * self.prefix[b]
        h = off // cnt
        return b, h, self.Hkv * self.prefix[b] + h * cnt, cnt

    def segments(self, c):
        """(g, s1, unit, unit start, unit end) in the order CTA c walks them."""
        g0, g1 = self.range_start(c), self.range_start(c + 1)
        n_loc = g1 - g0
        gL = g0
        if n_loc > 0:
            _, _, us, _ = self.locate(g1 - 1)
            if us > g0:
                gL = us
        nL = g1 - gL

        def rot(pos):
            return gL + pos if pos < nL else g0 + (pos - nL)

        def run_end(pos):
            return g1 if pos < nL else gL

        out, pos = [], 0
        while pos < n_loc:
            g = rot(pos)
            b, h, us, cnt = self.locate(g)
            ue = us + cnt
            s1 = min(run_end(pos), ue)
            out.append((g, s1, b * self.Hkv + h, us, ue))
            pos += s1 - g
        return out

    def selected_units(self, c):
        """Units the single-launch CTA c selects (its last unit first)."""
        g0, g1 = self.range_start(c), self.range_start(c + 1)
        if g1 <= g0:
            return []
        b, h, us, _ = self.locate(g1 - 1)
        u_last = b * self.Hkv + h
        sel = [u_last] if us >= g0 else []
        b, h, us, _ = self.locate(g0)
        u = b * self.Hkv + h + (1 if us < g0 else 0)
        while u < u_last:
            ub = u // self.Hkv
            if self.prefix[ub + 1] != self.prefix[ub]:
                sel.append(u)
            u += 1
        return sel


def check(cnts, Hkv, C, W0=0):
    m = Split(cnts, Hkv, C, W0)
    if m.T == 0:
        return
    segs = []
    partial_writers = {}          # unit -> CTAs that wrote a partial
    ticket = {}                   # unit -> pages ticketed
    slots = set()
    for c in range(C):
        seen = set()
        for g, s1, u, us, ue in m.segments(c):
            assert us <= g < s1 <= ue, (g, s1, us, ue)
            assert m.range_start(c) <= g and s1 <= m.range_start(c + 1)
            assert u not in seen, ("two segments of one unit in a CTA", u, c)
            seen.add(u)
            segs.append((g, s1))
            if g == us and s1 == ue:
                continue                              # whole unit: written directly
            slot = u + c
            assert slot not in slots and slot < m.B * Hkv + C, (slot, u, c)
            slots.add(slot)
            partial_writers.setdefault(u, set()).add(c)
            ticket[u] = ticket.get(u, 0) + (s1 - g)
    segs.sort()
    assert segs[0][0] == 0 and segs[-1][1] == m.T
    for (a0, a1), (b0, b1) in zip(segs, segs[1:]):
        assert a1 == b0, "segments must tile the flattened pages"
    for u, writers in partial_writers.items():
        b = u // Hkv
        cnt = cnts[b]
        us = Hkv * m.prefix[b] + (u % Hkv) * cnt
        assert ticket[u] == cnt                       # exactly one CTA completes it
        merged = {x for x in range(m.cta_of(us), m.cta_of(us + cnt - 1) + 1)
                  if m.range_start(x) != m.range_start(x + 1)}
        assert merged == writers, (u, merged, writers)
    owner = {}
    for c in range(C):
        for u in m.selected_units(c):
            assert u not in owner, ("unit selected twice", u)
            owner[u] = c
    for u in range(m.B * Hkv):
        b = u // Hkv
        if cnts[b] == 0:
            assert u not in owner
            continue
        us = Hkv * m.prefix[b] + (u % Hkv) * cnts[b]
        assert m.range_start(owner[u]) <= us < m.range_start(owner[u] + 1)


def attention_grid(units, most_pages_per_unit, sms, min_pages_per_cta=8):
    """The host's grid: one CTA per SM, fewer when the batch's most pages give
    fewer than min_pages_per_cta per CTA."""
    want = -(-units * most_pages_per_unit // min_pages_per_cta)
    return max(1, min(sms, want))


@pytest.mark.parametrize("seed", range(4))
def test_work_split_invariants_for_every_grid(seed):
    rng = random.Random(seed)
    for _ in range(1500):
        B = rng.randint(1, 24)
        Hkv = rng.choice([1, 2, 4, 8])
        cnts = [rng.choice([0, 1, 2, 3, 5, 6, 16, 64, 128, 200]) for _ in range(B)]
        most = max(cnts) if max(cnts) else 2
        C = rng.choice([1, 2, 3, 5, 8, 37, 64, 151, 152,
                        attention_grid(B * Hkv, most, 152)])
        check(cnts, Hkv, C, W0=rng.choice([0, 1, 4, 4, 9, 256]))


@pytest.mark.parametrize("W0", [0, 4])
def test_headline_and_small_batch_shapes(W0):
    check([64] * 128, 4, 152, W0)                       # the 8K / 12.5 % headline
    check([16], 4, attention_grid(4, 16, 152), W0)      # one sequence: 8 CTAs
    check([64, 64], 4, attention_grid(8, 64, 152), W0)  # two sequences: 64 CTAs
    check([0, 40, 0, 3, 2, 128], 4, 152, W0)            # empty sequences and ragged budgets


def test_unit_weight_moves_pages_away_from_ranges_of_short_units():
    # a batch of one long sequence then many short ones: with a weight per
    # unit, the CTAs holding the short units get fewer pages, and every CTA's
    # pages + W0 * (units it starts) stay within one unit's worth of the mean
    cnts = [512] + [4] * 127
    for W0 in (0, 4):
        m = Split(cnts, 4, 152, W0)
        work = []
        for c in range(152):
            segs = m.segments(c)
            pages = sum(s1 - g for g, s1, _, _, _ in segs)
            starts = sum(1 for g, _, _, us, _ in segs if g == us)
            work.append(pages + W0 * starts)
        if W0:
            assert max(work) - min(work) <= 512 // 152 + W0 + 2, (min(work), max(work))
    m0, m4 = Split(cnts, 4, 152, 0), Split(cnts, 4, 152, 4)
    last0 = sum(s1 - g for g, s1, _, _, _ in m0.segments(151))
    last4 = sum(s1 - g for g, s1, _, _, _ in m4.segments(151))
    assert last4 < last0   # the last CTA (all short units) gets fewer pages


def test_small_batch_grid_bounds():
    assert attention_grid(4, 16, 152) == 8
    assert attention_grid(512, 64, 152) == 152
    assert attention_grid(1, 2, 152) == 1
    for units in range(1, 60):
        for most in (2, 3, 7, 8, 9, 64):
            C = attention_grid(units, most, 152)
            assert 1 <= C <= 152
            assert C == 152 or units * most <= 8 * C


def range_start_by_sequence(m, c):
    """The kernel's form of range_start: a search over the sequences (their
    last units end at weighted positions Hkv*(prefix[b+1] + W0*(b+1))), then
    the unit inside the sequence by one division, then the page."""
    if c >= m.C:
        return m.T
    V = c * m.V // m.C
    lo, hi = 0, m.B
    while lo < hi:
        mid = (lo + hi) >> 1
        if m.Hkv * (m.prefix[mid + 1] + m.W0 * (mid + 1)) > V:
            hi = mid
        else:
            lo = mid + 1
    if lo >= m.B:
        return m.T
    cn = m.cnts[lo]
    base, step = m.Hkv * (m.prefix[lo] + m.W0 * lo), cn + m.W0
    hh = min(max((V - base) // step, 0), m.Hkv - 1)
    us = m.Hkv * m.prefix[lo] + hh * cn
    return max(us, V - m.W0 * (lo * m.Hkv + hh + 1))


@pytest.mark.parametrize("seed", range(3))
def test_sequence_search_matches_the_unit_search(seed):
    rng = random.Random(100 + seed)
    for _ in range(1500):
        B = rng.randint(1, 40)
        Hkv = rng.choice([1, 2, 4, 8])
        cnts = [rng.choice([0, 0, 1, 2, 5, 16, 64, 129, 1000]) for _ in range(B)]
        C = rng.choice([1, 2, 7, 64, 152])
        m = Split(cnts, Hkv, C, rng.choice([0, 1, 4, 8, 256]))
        if m.T == 0:
            continue
        for c in range(C + 1):
            assert range_start_by_sequence(m, c) == m.range_start(c), (cnts, Hkv, C, m.W0, c)
