"""GPU parity of the page hit-rate instrumentation.

qasa_page_attention_mass (the share of the dense attention of each
(sequence, KV head) on each page) is compared element by element with the fp64
oracle; qasa_page_hit_rate (hits against the k pages of largest mass, the mass
the selection covers, the best mass any k pages cover) is compared with the
oracle's page_hit_rate on the oracle's mass and the GPU's own selection.

Tolerances.  The GPU forms each logit in fp32 (d fused multiply-adds of
exactly representable products, then a butterfly over at most 32 lanes) and
sums at most a few thousand exp2 terms per row group in fp32; the relative
error of a page mass stays far below MASS_RTOL.  Hit counts are exact unless
the oracle's k-th and (k+1)-th largest masses lie within the mass tolerance of
each other: then the two sides may order that boundary differently, and the
counts may differ by at most the number of pages inside that band.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from query_aware_sparse_append_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu

MASS_RTOL, MASS_ATOL = 2e-4, 1e-7
SUM_ATOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from query_aware_sparse_append_gb300 import build
    build.build()


def _qasa():
    from query_aware_sparse_append_gb300 import binding
    return binding


def _kept(N, budget, max_budget):
    if N <= 0:
        return 0
    k = N if budget >= N else max(budget, min(N, 2))
    return min(k, max_budget)


def _check_unit(case, b, h, gmass, sel_row, hits, cov, best):
    P = case.cfg.page_size
    L = int(case.lens[b])
    N = -(-L // P)
    k = _kept(N, int(case.budgets[b]), case.max_budget)
    om = oracle.page_attention_mass(case.q64(b, h), case.k64(b, h), L, P)
    np.testing.assert_allclose(gmass[:N], om, rtol=MASS_RTOL, atol=MASS_ATOL,
                               err_msg="page mass of sequence %d head %d" % (b, h))
    if N:
        assert abs(float(gmass[:N].astype(np.float64).sum()) - 1.0) < SUM_ATOL
    o_hits, o_cov, o_best = oracle.page_hit_rate(om, sel_row[:k], k)
    assert cov == pytest.approx(o_cov, abs=SUM_ATOL), (b, h)
    assert best == pytest.approx(o_best, abs=SUM_ATOL), (b, h)
    assert best >= cov - SUM_ATOL
    if hits != o_hits:
        srt = np.sort(om)[::-1]
        m_k, m_k1 = srt[k - 1], (srt[k] if k < N else -np.inf)
        band = MASS_RTOL * m_k + MASS_ATOL
        assert m_k - m_k1 <= 2 * band, "hits %d vs oracle %d with untied boundary %r / %r" % (
            hits, o_hits, m_k, m_k1)
        in_band = int(np.sum(np.abs(om - m_k) <= 2 * band))
        assert abs(hits - o_hits) <= in_band
    return k


def _variant(name, dtype=None):
    cfg = W.CONFIGS[name]
    return dataclasses.replace(cfg, dtype=dtype) if dtype else cfg


@pytest.mark.parametrize("name,dtype,batch,seed,lens", [
    ("tiny", None, 1, 31, None),                          # f32, d=64, 4 planted pages
    ("tinyllama", None, 3, 32, [4096, 1000, 17]),         # f16, d=64, G=8, planted
    ("gpt2_345m", None, 7, 33, None),                     # f16, d=64, G=1, ragged
    ("gpt2_345m", "bf16", 5, 34, None),                   # bf16, d=64
    ("llama_1b3_32k", None, 1, 35, [9000]),               # bf16, d=128, P=32, outlier channels
    ("serving_mix", None, 4, 36, None),                   # f16, d=128, ragged long mix
    ("headline_8k", "f32", 2, 37, [8192, 3001]),          # f32, d=128
])
def test_page_mass_and_hit_rate_match_the_oracle(name, dtype, batch, seed, lens):
    qasa = _qasa()
    case = H.make_case(_variant(name, dtype), seed=seed, batch=batch, lens=lens)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    maxp = case.bt.shape[1]
    Hkv = case.cfg.num_kv_heads
    sentinel = -7.0
    mass = torch.full((batch, Hkv, maxp), sentinel, dtype=torch.float32, device="cuda")
    qasa.page_attention_mass(case.cache, case.q_dev, case.bt, case.lens_dev, mass=mass, status=status)
    _, sel = qasa.sparse_decode_attention(case.cache, case.q_dev, case.bt, case.lens_dev, case.budget_dev,
                                          max_budget=case.max_budget, status=status)
    hits, cov, best = qasa.page_hit_rate(case.cache, mass, case.lens_dev, case.budget_dev, sel,
                                         status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    gm, gs = mass.cpu().numpy(), sel.cpu().numpy()
    gh, gc, gb = hits.cpu().numpy(), cov.cpu().numpy(), best.cpu().numpy()
    P = case.cfg.page_size
    for b in range(batch):
        N = -(-int(case.lens[b]) // P)
        assert np.all(gm[b, :, N:] == sentinel), "entries beyond the page count were written"
        for h in range(Hkv):
            _check_unit(case, b, h, gm[b, h], gs[b, h], int(gh[b, h]), float(gc[b, h]), float(gb[b, h]))


def test_selection_of_the_top_mass_pages_hits_every_page():
    # feed the GPU's own top-k by mass back as the selection: every kept page is a hit
    qasa = _qasa()
    case = H.make_case(W.CONFIGS["tinyllama"], seed=38, batch=2, lens=[4096, 2500])
    mass = qasa.page_attention_mass(case.cache, case.q_dev, case.bt, case.lens_dev)
    gm = mass.cpu().numpy()
    P, mb = case.cfg.page_size, case.max_budget
    Hkv = case.cfg.num_kv_heads
    sel = np.full((2, Hkv, mb), -1, dtype=np.int32)
    ks = []
    for b in range(2):
        N = -(-int(case.lens[b]) // P)
        k = _kept(N, int(case.budgets[b]), mb)
        ks.append(k)
        for h in range(Hkv):
            sel[b, h, :k] = np.sort(np.argsort(-gm[b, h, :N], kind="stable")[:k])
    hits, cov, best = qasa.page_hit_rate(case.cache, mass, case.lens_dev, case.budget_dev,
                                         torch.from_numpy(sel).cuda())
    torch.cuda.synchronize()
    for b in range(2):
        assert np.all(hits[b].cpu().numpy() == ks[b])
    np.testing.assert_allclose(cov.cpu().numpy(), best.cpu().numpy(), rtol=0, atol=1e-6)


def test_hit_rate_edge_cases():
    # empty sequence, a one-token sequence, a budget covering every page, and an
    # invalid block-table entry (its page gets zero mass and a device flag)
    qasa = _qasa()
    cfg = W.CONFIGS["gpt2_345m"]
    case = H.make_case(cfg, seed=39, batch=4, lens=[0, 1, 300, 640], budgets=[8, 8, 1000, 8])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mass = qasa.page_attention_mass(case.cache, case.q_dev, case.bt, case.lens_dev, status=status)
    _, sel = qasa.sparse_decode_attention(case.cache, case.q_dev, case.bt, case.lens_dev, case.budget_dev,
                                          max_budget=case.max_budget, status=status)
    hits, cov, best = qasa.page_hit_rate(case.cache, mass, case.lens_dev, case.budget_dev, sel,
                                         status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    h, c, bst = hits.cpu().numpy(), cov.cpu().numpy(), best.cpu().numpy()
    assert np.all(h[0] == 0) and np.all(c[0] == 0) and np.all(bst[0] == 0)
    assert np.all(h[1] == 1) and np.allclose(c[1], 1.0, atol=1e-6) and np.allclose(bst[1], 1.0, atol=1e-6)
    assert np.all(h[2] == 19)                       # 300 tokens: 19 pages, all kept
    assert np.allclose(c[2], 1.0, atol=1e-4) and np.allclose(bst[2], 1.0, atol=1e-4)

    bt = case.bt.clone()
    bt[3, 5] = case.cache.num_phys_pages + 3
    status.zero_()
    mass2 = qasa.page_attention_mass(case.cache, case.q_dev, bt, case.lens_dev, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x1
    assert torch.all(mass2[3, :, 5] == 0)
    assert abs(float(mass2[3, :, :40].sum(dim=-1).max()) - 1.0) < 1e-4
