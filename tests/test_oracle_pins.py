"""Pins of the CPU oracle against facts fixed outside it (no GPU).

The pages print no worked example, so every pin is a closed form, an
invariant, a brute-force enumeration on tiny inputs, or a reduction to a
library routine (numpy min/max, a matmul, scipy's softmax).  Each is chosen so
that a plausible slip in the oracle -- a swapped lo/hi, a dropped head in the
group maximum, an off-by-one page range, an inverted tie rule, a missing
softmax scale or mask -- fails at least one of them.
"""
import itertools
import math

import numpy as np
import pytest
import scipy.special

import oracle


def rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------- page boxes

@pytest.mark.parametrize("L,P", [(1, 16), (16, 16), (37, 16), (100, 32), (64, 8)])
def test_bounds_equal_numpy_minmax(L, P):
    K = rng(L).standard_normal((L, 12))
    lo, hi = oracle.page_bounds(K, P)
    N = -(-L // P)
    assert lo.shape == (N, 12)
    for p in range(N):
        rows = K[p * P:min((p + 1) * P, L)]
        assert np.array_equal(lo[p], rows.min(axis=0))
        assert np.array_equal(hi[p], rows.max(axis=0))


@pytest.mark.parametrize("chunks", [[1] * 50, [7, 9, 1, 33], [16, 16, 18], [50], [3, 13, 2, 2, 30]])
def test_bounds_by_appends_equal_from_scratch(chunks):
    L = sum(chunks)
    K = rng(L).standard_normal((L, 8))
    a = oracle.page_bounds(K, 16)
    b = oracle.page_bounds_by_appends(K, 16, chunks)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ------------------------------------------------------------------- scores

def _brute_max_qk(q, K, L, P):
    N = -(-L // P)
    out = np.empty(N)
    for p in range(N):
        rows = K[p * P:min((p + 1) * P, L)]
        out[p] = np.max(q @ rows.T)
    return out


@pytest.mark.parametrize("G,d,L,P", [(1, 16, 70, 16), (4, 32, 129, 16), (8, 64, 256, 32)])
def test_score_upper_bounds_every_true_logit(G, d, L, P):
    r = rng(G * 1000 + d)
    q = r.standard_normal((G, d))
    K = r.standard_normal((L, d)) * r.lognormal(0, 0.5, size=d)
    lo, hi = oracle.page_bounds(K, P)
    s = oracle.page_scores(q, lo, hi)
    true = _brute_max_qk(q, K, L, P)
    assert np.all(s >= true - 1e-12 * np.abs(true).max())


@pytest.mark.parametrize("G", [1, 3, 8])
def test_score_tight_when_all_keys_equal(G):
    r = rng(G)
    d, P = 48, 16
    q = r.standard_normal((G, d))
    K = r.standard_normal((4 * P, d))
    K[P:2 * P] = K[P]                       # page 1: every key identical
    lo, hi = oracle.page_bounds(K, P)
    s = oracle.page_scores(q, lo, hi)
    expect = max(float(np.dot(q[g], K[P])) for g in range(G))
    assert s[1] == pytest.approx(expect, rel=1e-13, abs=1e-13)


def test_score_equals_sign_split_matmul():
    # sum_c max(q lo, q hi) == q+ . hi + q- . lo when lo <= hi (a different formula)
    r = rng(7)
    G, d, N = 8, 64, 40
    q = r.standard_normal((G, d))
    a, b = r.standard_normal((N, d)), r.standard_normal((N, d))
    lo, hi = np.minimum(a, b), np.maximum(a, b)
    qp, qm = np.maximum(q, 0), np.minimum(q, 0)
    expect = (qp @ hi.T + qm @ lo.T).max(axis=0)
    assert np.allclose(oracle.page_scores(q, lo, hi), expect, rtol=1e-13, atol=1e-13)


def test_score_orientation_closed_form():
    lo = np.array([[-1.0, 0.0]])
    hi = np.array([[2.0, 0.0]])
    assert oracle.page_scores(np.array([1.0, 0.0]), lo, hi)[0] == 2.0
    assert oracle.page_scores(np.array([-1.0, 0.0]), lo, hi)[0] == 1.0
    # group maximum, not sum or mean, over the heads sharing the KV head
    q = np.array([[1.0, 0.0], [-3.0, 0.0]])
    assert oracle.page_scores(q, lo, hi)[0] == 3.0


def test_score_negative_group_max_is_not_clamped_at_zero():
    lo = np.array([[1.0, 1.0]])
    hi = np.array([[2.0, 2.0]])
    q = np.array([[-1.0, -1.0], [-2.0, -0.5]])
    assert oracle.page_scores(q, lo, hi)[0] == -2.0


# ---------------------------------------------------------------- selection

def _brute_select(s, k):
    N = len(s)
    if k >= N:
        return list(range(N))
    forced = [0, N - 1] if N >= 2 else [0]
    cand = [p for p in range(N) if p not in forced]
    take = max(k - len(forced), 0)
    best = None
    for sub in itertools.combinations(cand, take):
        tot = sum(s[p] for p in sub)
        key = (-tot, tuple(sorted(sub)))
        if best is None or key < best[0]:
            best = (key, sub)
    return sorted(forced + list(best[1]))


@pytest.mark.parametrize("N", [1, 2, 3, 5, 8, 11])
def test_select_matches_bruteforce_with_ties(N):
    r = rng(N)
    for trial in range(6):
        s = r.integers(-3, 4, size=N).astype(np.float64)   # many exact ties
        for k in range(1, N + 2):
            got = oracle.select_pages(s, k).tolist()
            assert got == _brute_select(s.tolist(), k), (s, k)


def test_select_ties_go_to_lower_index():
    s = np.zeros(10)
    assert oracle.select_pages(s, 5).tolist() == [0, 1, 2, 3, 9]
    s[7] = 1.0
    assert oracle.select_pages(s, 4).tolist() == [0, 1, 7, 9]


def test_select_forced_pages_and_budget_floor():
    s = np.arange(10, dtype=np.float64)[::-1].copy()  # page 0 best, page 9 worst
    s[0], s[9] = -100.0, -100.0
    assert oracle.select_pages(s, 1).tolist() == [0, 9]      # forced even over budget
    assert oracle.select_pages(s, 3).tolist() == [0, 1, 9]
    assert oracle.select_pages(np.array([5.0]), 1).tolist() == [0]
    assert oracle.select_pages(np.array([5.0, 1.0]), 1).tolist() == [0, 1]
    assert oracle.select_pages(s, 10).tolist() == list(range(10))
    assert oracle.select_pages(s, 99).tolist() == list(range(10))


def test_select_nan_ranks_last():
    s = np.array([0.0, np.nan, 1.0, np.nan, 0.5, 0.0])
    assert oracle.select_pages(s, 3).tolist() == [0, 2, 5]


# ---------------------------------------------------------------- attention

def _textbook(q, K, V, L, scale):
    z = scale * (q @ K[:L].T)
    return scipy.special.softmax(z, axis=-1) @ V[:L]


@pytest.mark.parametrize("G,d,L,P", [(1, 8, 1, 16), (2, 16, 33, 16), (8, 64, 300, 32)])
def test_dense_attention_equals_scipy_softmax(G, d, L, P):
    r = rng(L)
    q, K, V = r.standard_normal((G, d)), r.standard_normal((L + 5, d)), r.standard_normal((L + 5, d))
    got = oracle.dense_attention(q, K, V, L, P)
    assert np.allclose(got, _textbook(q, K, V, L, 1 / math.sqrt(d)), rtol=1e-12, atol=1e-13)


def test_attention_over_pages_equals_dense_over_their_tokens():
    r = rng(11)
    G, d, P, L = 4, 16, 16, 150
    q, K, V = r.standard_normal((G, d)), r.standard_normal((L, d)), r.standard_normal((L, d))
    pages = [0, 3, 5, 9]                              # 9 is the partial newest page
    toks = np.concatenate([np.arange(p * P, min((p + 1) * P, L)) for p in pages])
    got = oracle.attention(q, K, V, L, P, pages)
    expect = _textbook(q, K[toks], V[toks], len(toks), 1 / math.sqrt(d))
    assert np.allclose(got, expect, rtol=1e-12, atol=1e-13)


def test_attention_single_token_returns_v():
    r = rng(3)
    q, K, V = r.standard_normal((3, 8)), r.standard_normal((1, 8)), r.standard_normal((1, 8))
    assert np.allclose(oracle.dense_attention(q, K, V, 1, 16), np.repeat(V, 3, 0), rtol=0, atol=1e-15)


def test_attention_equal_logits_give_mean_of_valid_values():
    r = rng(4)
    K, V = r.standard_normal((40, 8)), r.standard_normal((40, 8))
    out = oracle.dense_attention(np.zeros((2, 8)), K, V, 37, 16)
    assert np.allclose(out, V[:37].mean(axis=0)[None], rtol=1e-13, atol=1e-14)


def test_attention_ignores_tokens_at_or_beyond_length():
    r = rng(5)
    q, K, V = r.standard_normal((2, 8)), r.standard_normal((48, 8)), r.standard_normal((48, 8))
    a = oracle.dense_attention(q, K, V, 37, 16)
    K2, V2 = K.copy(), V.copy()
    K2[37:] = 1e3
    V2[37:] = -1e3
    assert np.array_equal(a, oracle.dense_attention(q, K2, V2, 37, 16))


def test_attention_scale_is_inverse_sqrt_d():
    # two tokens, logits differ by 1 before scaling: weights are sigmoid(+-1/sqrt(d))
    d = 16
    q = np.zeros((1, d)); q[0, 0] = 1.0
    K = np.zeros((2, d)); K[1, 0] = 1.0
    V = np.zeros((2, d)); V[1, 1] = 1.0
    out = oracle.dense_attention(q, K, V, 2, 16)
    assert out[0, 1] == pytest.approx(1 / (1 + math.exp(-1 / math.sqrt(d))), rel=1e-14)


# --------------------------------------------------- full step (decode unit)

def test_full_budget_equals_dense():
    r = rng(12)
    G, d, P, L = 4, 32, 16, 200
    q, K, V = r.standard_normal((G, d)), r.standard_normal((L, d)), r.standard_normal((L, d))
    lo, hi = oracle.page_bounds(K, P)
    N = -(-L // P)
    dense = oracle.dense_attention(q, K, V, L, P)
    for k in (N, N + 5):
        s, sel, out = oracle.decode_unit(q, K, V, lo, hi, L, P, k)
        assert sel.tolist() == list(range(N))
        assert np.array_equal(out, dense)


def test_decode_unit_composes_the_three_steps():
    r = rng(13)
    G, d, P, L, k = 2, 16, 16, 333, 6
    q, K, V = r.standard_normal((G, d)), r.standard_normal((L, d)), r.standard_normal((L, d))
    lo, hi = oracle.page_bounds(K, P)
    s, sel, out = oracle.decode_unit(q, K, V, lo, hi, L, P, k)
    assert np.array_equal(s, oracle.page_scores(q, lo, hi))
    assert np.array_equal(sel, oracle.select_pages(s, k))
    assert np.array_equal(out, oracle.attention(q, K, V, L, P, sel))


def test_empty_sequence_gives_zeros():
    s, sel, out = oracle.decode_unit(np.ones((2, 4)), np.zeros((0, 4)), np.zeros((0, 4)),
                                     np.zeros((0, 4)), np.zeros((0, 4)), 0, 16, 4)
    assert len(sel) == 0 and np.all(out == 0)


# ------------------------------------------- page attention mass and hit rate
# The TinyServe abstract names the page hit rate without a definition; the
# oracle measures it against the dense softmax mass on each page.

def test_page_mass_equals_dense_attention_over_page_indicator_values():
    # with V[t] = one-hot of t's page, the dense attention output of head g is
    # exactly head g's mass per page; the mass is the mean over the heads
    r = rng(30)
    G, P, L = 3, 16, 70
    N = -(-L // P)
    d = 8
    q, K = r.standard_normal((G, d)), r.standard_normal((L, d))
    V = np.zeros((L, d))
    V[np.arange(L), np.arange(L) // P] = 1.0
    want = oracle.dense_attention(q, K, V, L, P)[:, :N].mean(axis=0)
    got = oracle.page_attention_mass(q, K, L, P)
    assert got.shape == (N,)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-16)


def test_page_mass_of_equal_keys_is_token_share_with_ragged_tail():
    G, d, P, L = 2, 8, 16, 53
    K = np.tile(np.linspace(-1, 1, d), (L, 1))
    q = rng(31).standard_normal((G, d))
    got = oracle.page_attention_mass(q, K, L, P)
    assert got.tolist() == pytest.approx([16 / 53, 16 / 53, 16 / 53, 5 / 53], rel=1e-14)


def test_page_mass_closed_form_for_one_raised_page():
    # tokens of page 2 have logit a*scale, all others 0
    d, P, L, a = 4, 16, 64, 3.0
    q = np.array([[2.0, 0, 0, 0]])
    K = np.zeros((L, d))
    K[32:48, 0] = a / 2.0
    e = math.exp(a / math.sqrt(d))
    got = oracle.page_attention_mass(q, K, L, P)
    den = 16 * e + 48
    assert got.tolist() == pytest.approx([16 / den, 16 / den, 16 * e / den, 16 / den], rel=1e-14)


def test_page_mass_averages_heads_not_logits():
    # two heads that each put all their weight on a different page
    d, P, L = 2, 16, 32
    K = np.zeros((L, d)); K[:16, 0] = 1.0; K[16:, 1] = 1.0
    q = np.array([[800.0, 0.0], [0.0, 800.0]])
    got = oracle.page_attention_mass(q, K, L, P)
    assert got.tolist() == pytest.approx([0.5, 0.5], abs=1e-15)


def test_page_mass_of_empty_sequence():
    assert oracle.page_attention_mass(np.ones((1, 4)), np.zeros((0, 4)), 0, 16).shape == (0,)


def test_hit_rate_hand_example():
    mass = [0.1, 0.4, 0.2, 0.3]
    assert oracle.page_hit_rate(mass, [0, 3], 2) == (1, pytest.approx(0.4), pytest.approx(0.7))
    assert oracle.page_hit_rate(mass, [1, 3], 2) == (2, pytest.approx(0.7), pytest.approx(0.7))
    # equal masses: the lower page ids are the top ones
    assert oracle.page_hit_rate([0.25] * 4, [2, 3], 2) == (0, 0.5, 0.5)
    assert oracle.page_hit_rate([0.25] * 4, [0, 3], 2)[0] == 1


def test_hit_rate_against_brute_force_subsets():
    import itertools
    r = rng(32)
    for trial in range(40):
        N = int(r.integers(2, 9))
        mass = r.integers(0, 4, size=N).astype(float)   # many ties
        mass /= max(mass.sum(), 1.0)
        k = int(r.integers(1, N + 1))
        sel = np.sort(r.choice(N, size=k, replace=False))
        hits, cov, best = oracle.page_hit_rate(mass, sel, k)
        subsets = list(itertools.combinations(range(N), k))
        best_sum = max(sum(mass[list(s)]) for s in subsets)
        assert best == pytest.approx(best_sum, abs=1e-15)
        assert cov == pytest.approx(sum(mass[sel]), abs=1e-15)
        # the top set: largest sum, and among those the lexicographically
        # smallest list of (-mass, page) pairs
        top = min((s for s in subsets if abs(sum(mass[list(s)]) - best_sum) < 1e-15),
                  key=lambda s: sorted((-mass[i], i) for i in s))
        assert hits == len(set(top) & set(sel.tolist()))


# ------------------------------------------------------------- FP8 KV (E4M3)
# Format: OCP 8-bit floating point, E4M3 variant (bias 7, 3 mantissa bits,
# subnormals, no infinities, S.1111.111 = NaN, largest finite 448).

def test_e4m3_decode_known_codes_and_order():
    d = oracle.e4m3_decode(np.arange(256))
    known = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x39: 1.125,
             0x3F: 1.875, 0x40: 2.0, 0x77: 240.0, 0x78: 256.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    for c, v in known.items():
        assert d[c] == v, hex(c)
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF])
    pos = d[:0x7F]
    assert np.all(np.diff(pos) > 0), "codes 0..126 must increase"
    assert np.array_equal(d[0x80:0xFF], -pos)


def test_e4m3_encode_is_the_nearest_code_with_ties_to_even():
    d = oracle.e4m3_decode(np.arange(256)).astype(np.float64)
    finite = [c for c in range(256) if not np.isnan(d[c]) and c != 0x80]
    r = rng(40)
    xs = np.concatenate([r.standard_normal(3000) * 10.0 ** r.uniform(-4, 3, 3000),
                         (d[1:0x7E] + d[2:0x7F]) / 2,          # midpoints between neighbours
                         -(d[1:0x7E] + d[2:0x7F]) / 2])
    xs = xs.astype(np.float32)
    got = oracle.e4m3_encode(xs)
    for x, c in zip(xs.astype(np.float64), got):
        if abs(x) > 448:
            assert d[c] == np.sign(x) * 448
            continue
        err = np.abs(d[finite] - x)
        best = err.min()
        cands = [finite[i] for i in np.flatnonzero(err == best)]
        if len(cands) > 1:      # a tie: the code with the even mantissa (a zero result is +0)
            cands = [k for k in cands if (k & 1) == 0 or d[k] == 0]
        assert c in cands, (x, c, cands)


def test_e4m3_round_trip_saturation_and_zero():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF, 0x80)], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes)), codes)
    assert oracle.e4m3_encode(np.float32([-0.0, -1e-30, 1e30, -1e30, 449.0]))[:5].tolist() == [0, 0, 0x7E, 0xFE, 0x7E]


def test_fp8_scale_closed_forms():
    # scale = amax / 448 in fp32: exact for amax = 448 * 2^k, zero for a zero
    # page, monotone in amax, and within half an fp32 ulp of the real quotient
    k = np.arange(-20, 21)
    amax = np.float32(448.0) * np.exp2(k).astype(np.float32)
    assert np.array_equal(oracle.fp8_scale(amax), np.exp2(k).astype(np.float32))
    assert oracle.fp8_scale(np.float32([0.0]))[0] == 0.0
    a = np.sort(rng(43).random(2000).astype(np.float32) * 1000)
    s = oracle.fp8_scale(a)
    assert s.dtype == np.float32 and np.all(np.diff(s) >= 0)
    exact = a.astype(np.float64) / 448.0
    assert np.all(np.abs(s - exact) <= 0.5 * np.spacing(s.astype(np.float32)).astype(np.float64))


def _round_to_f32(fr):
    """The float32 nearest to the exact rational fr (ties to the even significand)."""
    from fractions import Fraction
    f = np.float32(float(fr))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    return min(cands, key=lambda c: (abs(Fraction(float(c)) - fr), int(np.float32(c).view(np.uint32)) & 1))


def test_fp8_scale_is_the_correctly_rounded_quotient():
    # fp32 division rounds the exact quotient to nearest: compare the oracle's
    # scale with amax / 448 computed exactly in rational arithmetic and rounded
    # once, on random magnitudes, powers of two and values next to them
    from fractions import Fraction
    r = rng(45)
    a = np.concatenate([r.random(300).astype(np.float32) * np.float32(500.0),
                        np.exp2(np.arange(-30, 12)).astype(np.float32),
                        np.nextafter(np.exp2(np.arange(-10, 10)).astype(np.float32), np.float32(np.inf)),
                        np.float32([448.0, 447.99997, 1e-38, 3.4e38])])
    got = oracle.fp8_scale(a)
    for x, g in zip(a, got):
        want = _round_to_f32(Fraction(float(x)) / 448)
        assert np.float32(g).view(np.uint32) == np.float32(want).view(np.uint32), (x, g, want)


def test_fp8_dequant_closed_forms():
    # code * scale per row: 1.0 (0x38) and -1.0 (0xB8) give +-scale, the
    # largest finite code (0x7E = 448) gives 448 * scale, zero gives 0; and a
    # value quantized under its row's scale comes back within half a code step
    sc = np.array([0.5, 3.0, 1e-3], dtype=np.float32)
    codes = np.tile(np.uint8([0x38, 0xB8, 0x7E, 0x00]), (3, 1))
    v = oracle.fp8_dequant(codes, sc)
    assert v.dtype == np.float64
    assert np.array_equal(v[:, 0], sc.astype(np.float64)) and np.array_equal(v[:, 1], -sc.astype(np.float64))
    assert np.array_equal(v[:, 2], 448.0 * sc.astype(np.float64)) and not v[:, 3].any()
    x = rng(44).standard_normal((3, 64)).astype(np.float32) * np.float32(100.0) * sc[:, None]
    q = oracle.e4m3_encode(x / sc[:, None])
    back = oracle.fp8_dequant(q, sc)
    mag = np.abs(oracle.e4m3_decode(q)).astype(np.float64)
    # E4M3 step at a value of magnitude m: 2^(floor(log2 m) - 3) (normals), 2^-9 below 2^-6
    step = np.where(mag >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(mag, 2.0 ** -6))) - 3), 2.0 ** -9)
    assert np.all(np.abs(back - x) <= 0.5 * step * sc[:, None] * (1 + 1e-6) + 1e-30)


def _fp8_page_check(X, P, codes, amax, lo, hi):
    L, d = X.shape
    for p in range(-(-L // P)):
        rows = slice(p * P, min(L, (p + 1) * P))
        assert amax[p] == np.abs(X[rows]).max()
        v = oracle.e4m3_decode(codes[rows])
        assert np.array_equal(oracle.e4m3_decode(lo[p]), v.min(axis=0))
        assert np.array_equal(oracle.e4m3_decode(hi[p]), v.max(axis=0))


def test_fp8_append_single_chunk_is_direct_quantization():
    r = rng(41)
    P, L, d = 16, 75, 8
    X = (r.standard_normal((L, d)) * 3).astype(np.float32)
    codes, amax, lo, hi = oracle.fp8_append_replay(X, P, [L])
    for p in range(-(-L // P)):
        rows = slice(p * P, min(L, (p + 1) * P))
        s = np.float32(np.abs(X[rows]).max()) / np.float32(448.0)
        assert np.array_equal(codes[rows], oracle.e4m3_encode(X[rows] / s))
    _fp8_page_check(X, P, codes, amax, lo, hi)


def test_fp8_append_without_amax_growth_matches_one_chunk():
    # the first token of every page holds the page's largest |x|: later chunks
    # never change a scale, so the chunking cannot matter
    r = rng(42)
    P, L, d = 16, 64, 8
    X = (r.standard_normal((L, d))).astype(np.float32)
    X[::P, 0] = 100.0
    one = oracle.fp8_append_replay(X, P, [L])
    many = oracle.fp8_append_replay(X, P, [1] * L)
    for a, b in zip(one, many):
        assert np.array_equal(a, b)


def test_fp8_append_requantizes_when_amax_grows():
    # token by token with growing magnitudes: the old codes are re-scaled, so
    # the error of every value stays within two rounding steps of the final
    # scale (one for its own quantization, one per re-scaling is bounded by the
    # geometric growth here); leaving the old codes alone would be off by the
    # ratio of the scales
    r = rng(43)
    P, L, d = 16, 48, 4
    X = (r.standard_normal((L, d)) * np.linspace(1, 40, L)[:, None]).astype(np.float32)
    codes, amax, lo, hi = oracle.fp8_append_replay(X, P, [1] * L)
    _fp8_page_check(X, P, codes, amax, lo, hi)
    for p in range(L // P):
        rows = slice(p * P, (p + 1) * P)
        s = np.float64(np.float32(amax[p]) / np.float32(448.0))
        deq = oracle.e4m3_decode(codes[rows]).astype(np.float64) * s
        x = X[rows].astype(np.float64)
        # half an E4M3 step at |x| is at most |x| / 16 (normal) or s * 2^-10 (subnormal)
        step = np.maximum(np.abs(x) / 16.0, s * 2.0 ** -10)
        assert np.all(np.abs(deq - x) <= 4 * step + 1e-12), np.max(np.abs(deq - x) / step)


def test_fp8_append_zero_page():
    X = np.zeros((20, 4), np.float32)
    codes, amax, lo, hi = oracle.fp8_append_replay(X, 16, [3, 17])
    assert not codes.any() and not amax.any() and not lo.any() and not hi.any()


def test_stored_oracle_values_are_reproduced():
    # tests/golden/tiny_decode.txt is written by tests/golden/make_golden.py from
    # the oracle alone; any change of the oracle's arithmetic must show up here
    import importlib.util
    import os
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(here, "make_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    stored = [ln for ln in open(os.path.join(here, "tiny_decode.txt")).read().splitlines() if ln]
    fresh = mod.golden_lines()
    assert len(stored) == len(fresh)
    for a, b in zip(stored, fresh):
        if a.startswith("#") or " kept " in a:
            assert a == b
        else:
            xa = [float(x) for x in a.split()[3:]]
            xb = [float(x) for x in b.split()[3:]]
            assert np.allclose(xa, xb, rtol=1e-12, atol=0.0), (a, b)
