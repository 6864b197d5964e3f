"""GPU parity of the FP8 (E4M3) KV cache.

The workloads draw float16 K/V; the append kernel quantizes them with a
per-(page, KV head) amax and re-quantizes a page's codes when an append raises
its amax.  The oracle replays the same appends (fp32 steps, its own E4M3
codec), so codes, amax and boxes must agree bit for bit.  Scores and outputs
are compared with the oracle on the exactly dequantized values (code * scale):
scores within the fp32 summation bound plus one rounding for the scale,
selections exact outside the tie band, outputs within the output tolerance.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from query_aware_sparse_append_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from query_aware_sparse_append_gb300 import build
    build.build()


def _qasa():
    from query_aware_sparse_append_gb300 import binding
    return binding


def _fp8(name):
    return dataclasses.replace(W.CONFIGS[name], dtype="e4m3")


def _gpu_cache(case):
    c = case.cache
    return (c.k_pool.cpu().numpy(), c.v_pool.cpu().numpy(), c.page_bounds.cpu().numpy(),
            c.page_scales.cpu().numpy())


def _check_cache(case, chunks, units):
    kp, vp, bd, sc = _gpu_cache(case)
    P = case.cfg.page_size
    for b, h in units:
        L = int(case.lens[b])
        if L == 0:
            continue
        N = -(-L // P)
        ref = H.fp8_unit(case, b, h, chunks)
        phys = case.plan.block_table[b, :N]
        tok = np.arange(L)
        g_k = kp[phys[tok // P], h, tok % P]
        g_v = vp[phys[tok // P], h, tok % P]
        assert np.array_equal(g_k, ref["k_codes"]), (b, h, "K codes")
        assert np.array_equal(g_v, ref["v_codes"]), (b, h, "V codes")
        assert np.array_equal(sc[phys, h, 0], ref["k_amax"]), (b, h, "K amax")
        assert np.array_equal(sc[phys, h, 1], ref["v_amax"]), (b, h, "V amax")
        assert np.array_equal(bd[phys, h, 0], ref["lo"]), (b, h, "box lo")
        assert np.array_equal(bd[phys, h, 1], ref["hi"]), (b, h, "box hi")


def _check_decode(case, chunks, units, out, sel, scores):
    P = case.cfg.page_size
    out64 = H.gpu_out64(out, "e4m3")
    sel, scores = sel.cpu().numpy(), scores.cpu().numpy()
    for b, h in units:
        L = int(case.lens[b])
        N = -(-L // P)
        if N == 0:
            assert np.all(sel[b, h] == -1)
            continue
        ref = H.fp8_unit(case, b, h, chunks)
        q64 = case.q64(b, h)
        o_s, o_sel, o_out = oracle.decode_unit(q64, ref["K"], ref["V"], ref["LO"], ref["HI"], L, P,
                                               int(case.budgets[b]))
        k_eff = len(o_sel)
        tol = H.score_tolerance(q64, ref["LO"], ref["HI"]) + 2.0 ** -23 * np.abs(o_s)
        g_s = scores[b, h, :N].astype(np.float64)
        if k_eff < N:
            assert np.all(np.abs(g_s - o_s) <= tol), (b, h, np.max(np.abs(g_s - o_s) - tol))
        same = H.check_selection(sel[b, h], g_s if k_eff < N else None, o_s, o_sel, k_eff, tol)
        kept = sel[b, h][sel[b, h] >= 0]
        want = o_out if same else oracle.attention(q64, ref["K"], ref["V"], L, P, kept)
        H.assert_close(out64[b, h * case.G:(h + 1) * case.G], want, "fp8 out b=%d h=%d" % (b, h))


def _decode(case):
    qasa = _qasa()
    maxp = case.bt.shape[1]
    scores = torch.full((case.cfg.batch, case.cfg.num_kv_heads, maxp), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, sel = qasa.sparse_decode_attention(case.cache, case.q_dev, case.bt, case.lens_dev, case.budget_dev,
                                            max_budget=case.max_budget, scores=scores, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, qasa.decode_device_errors(int(status.item()))
    return out, sel, scores


def _units(case):
    return [(b, h) for b in range(case.cfg.batch) for h in range(case.cfg.num_kv_heads)]


@pytest.mark.parametrize("name,batch,seed,chunks", [
    ("tinyllama", 3, 61, None),                   # d64, P16, G8: one append per sequence
    ("tinyllama", 2, 62, [1] * 40 + [10 ** 6]),   # token-by-token appends first: re-quantization
    ("headline_8k", 2, 63, [7, 9, 1, 33, 10 ** 6]),   # d128, P16, mid-page starts
    ("llama_1b3_32k", 1, 64, [5, 40, 10 ** 6]),   # d128, P32, outlier channels
    ("gpt2_345m", 6, 65, None),                   # G = 1: FFMA scoring and consumers
])
def test_fp8_append_and_decode_match_the_oracle(name, batch, seed, chunks):
    lens = None
    if name == "llama_1b3_32k":
        lens = [6000]
    case = H.make_case(_fp8(name), seed=seed, batch=batch, lens=lens, append_chunks=chunks)
    units = _units(case)
    _check_cache(case, chunks, units)
    out, sel, scores = _decode(case)
    _check_decode(case, chunks, units, out, sel, scores)


def test_fp8_dense_matches_the_oracle_and_full_budget():
    qasa = _qasa()
    case = H.make_case(_fp8("serving_mix"), seed=66, batch=3, lens=[700, 16, 2049])
    out = qasa.dense_decode_attention(case.cache, case.q_dev, case.bt, case.lens_dev)
    torch.cuda.synchronize()
    g = H.gpu_out64(out, "e4m3")
    P = case.cfg.page_size
    for b, h in _units(case):
        ref = H.fp8_unit(case, b, h)
        want = oracle.dense_attention(case.q64(b, h), ref["K"], ref["V"], int(case.lens[b]), P)
        H.assert_close(g[b, h * case.G:(h + 1) * case.G], want, "fp8 dense b=%d h=%d" % (b, h))


def test_fp8_rebuilt_boxes_equal_the_append_boxes():
    qasa = _qasa()
    case = H.make_case(_fp8("headline_8k"), seed=67, batch=2, lens=[8192, 1001], append_chunks=[3, 10 ** 6])
    ref = case.cache.page_bounds.clone()
    case.cache.page_bounds.fill_(0x7F)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qasa.rebuild_page_bounds(case.cache, case.bt, case.lens_dev, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    P = case.cfg.page_size
    used = torch.tensor(sorted(set(int(x) for b, L in enumerate(case.lens)
                                   for x in case.plan.block_table[b, :-(-int(L) // P)])), device="cuda")
    assert torch.equal(case.cache.page_bounds[used], ref[used])


def test_fp8_zero_pages_and_empty_sequences():
    # all-zero keys give amax 0, scale 0 and zero codes; an empty sequence
    # gets -1 ids and a zero output
    qasa = _qasa()
    cfg = _fp8("tinyllama")
    case = H.make_case(cfg, seed=68, batch=3, lens=[0, 40, 300])
    for s in case.seqs[1:2]:
        s.k[:] = 0
        s.v[:] = 0
    H.build_device(case)
    kp, vp, bd, sc = _gpu_cache(case)
    phys = case.plan.block_table[1, :3]           # 40 tokens: pages of 16, 16 and 8 valid rows
    assert np.all(sc[phys, :, :2] == 0) and not bd[phys].any()
    assert not kp[phys[:2]].any() and not kp[phys[2], :, :8].any() and not vp[phys[2], :, :8].any()
    out, sel, scores = _decode(case)
    _check_decode(case, None, _units(case), out, sel, scores)
    assert np.all(H.gpu_out64(out, "e4m3")[0] == 0)


def test_fp8_through_the_other_entry_points(monkeypatch):
    # the single-launch request falls back to two launches for FP8 caches; the
    # workspace-free and host-buffer calls give the same bits; the page-mass
    # instrumentation refuses FP8 caches with QASA_ERR_DTYPE
    qasa = _qasa()
    case = H.make_case(_fp8("headline_8k"), seed=69, batch=4)
    ref_out, ref_sel, _ = _decode(case)
    monkeypatch.setenv("QASA_SINGLE_LAUNCH", "1")
    o1, s1, _ = _decode(case)
    monkeypatch.delenv("QASA_SINGLE_LAUNCH")
    assert torch.equal(s1, ref_sel) and torch.equal(o1.view(torch.int16), ref_out.view(torch.int16))

    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(ref_out)
    sel = torch.empty_like(ref_sel)
    assert qasa.sparse_decode_attention_noalloc(case.cache, case.q_dev, case.bt, case.lens_dev, case.budget_dev,
                                                case.max_budget, out, sel, status=status) == 0
    out_h = torch.empty(tuple(ref_out.shape), dtype=ref_out.dtype).pin_memory()
    sel_h = torch.empty(tuple(ref_sel.shape), dtype=torch.int32).pin_memory()
    qasa.sparse_decode_attention_host(case.cache, case.q_dev.cpu().pin_memory(), case.bt.cpu().pin_memory(),
                                      case.lens_dev.cpu().pin_memory(), case.budget_dev.cpu().pin_memory(),
                                      case.max_budget, out_h, sel_h, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(sel, ref_sel) and torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(sel_h, ref_sel.cpu()) and torch.equal(out_h.view(torch.int16), ref_out.cpu().view(torch.int16))

    with pytest.raises(qasa.QasaError) as err:
        qasa.page_attention_mass(case.cache, case.q_dev, case.bt, case.lens_dev)
    assert "dtype" in str(err.value)


def test_fp8_full_size_sampled_units():
    # the benchmark's FP8 workload at full size (B = 128, 8K, 12.5 %), in its
    # launch configuration: cache state and decode checked on sampled units
    cfg = _fp8("headline_8k")
    case = H.make_case(cfg, seed=0, poison=False)
    units = _units(case)
    rng = np.random.default_rng(0)
    pick = [units[i] for i in rng.choice(len(units), size=6, replace=False)] + [units[0], units[-1]]
    _check_cache(case, None, pick)
    out, sel, scores = _decode(case)
    _check_decode(case, None, pick, out, sel, scores)
    assert torch.isfinite(out.float()).all()
