"""Seeded workload generator: determinism, shapes, block tables (no GPU)."""
import numpy as np
import pytest

import oracle
from query_aware_sparse_append_gb300 import workloads as W


def test_sequence_regenerates_bit_identically():
    cfg = W.CONFIGS["tinyllama"]
    a = W.sequence(cfg, 3, 4096, seed=0)
    b = W.sequence(cfg, 3, 4096, seed=0)
    c = W.sequence(cfg, 3, 4096, seed=1)
    assert a.k.dtype == np.float16 and a.k.shape == (4096, 4, 64) and a.q.shape == (32, 64)
    assert np.array_equal(a.k.view(np.uint16), b.k.view(np.uint16))
    assert np.array_equal(a.q.view(np.uint16), b.q.view(np.uint16))
    assert not np.array_equal(a.k.view(np.uint16), c.k.view(np.uint16))


def test_bf16_storage_roundtrip_is_exact_for_representable_values():
    x = np.array([1.0, -2.5, 0.15625, 2.0 ** 100, -0.0], dtype=np.float32)
    bits = W.to_storage(x, "bf16")
    assert bits.dtype == np.uint16
    assert np.array_equal(W.widen(bits, "bf16"), x.astype(np.float64))


@pytest.mark.parametrize("name", list(W.CONFIGS))
def test_lengths_budgets_and_block_tables(name):
    cfg = W.CONFIGS[name]
    lens = W.seq_lens(cfg, 0)
    assert lens.shape == (cfg.batch,)
    assert lens.min() >= cfg.ctx_min and lens.max() <= cfg.ctx_max
    k = W.budgets(cfg, lens)
    assert np.all(k >= 1)
    plan = W.page_plan(cfg, lens, 0, reserve_tokens=1)
    bt = plan.block_table
    used = bt[bt >= 0]
    assert len(np.unique(used)) == len(used) == plan.num_phys_pages
    need = W.num_pages(lens + 1, cfg.page_size)
    for b in range(cfg.batch):
        assert np.all(bt[b, :need[b]] >= 0) and np.all(bt[b, need[b]:] == -1)


def test_budget_rules_of_the_configs():
    cfg = W.CONFIGS["tinyllama"]
    assert W.budgets(cfg, np.array([4096]))[0] == 64           # 25% of 256 pages
    cfg = W.CONFIGS["headline_8k"]
    assert W.budgets(cfg, np.array([8192]))[0] == 64           # 12.5% of 512 pages
    cfg = W.CONFIGS["serving_mix"].with_budget("permille", 50)
    assert W.budgets(cfg, np.array([16 * 21]))[0] == 2         # ceil(0.05 * 21)


def test_planted_pages_are_selected_by_the_oracle_tiny_config():
    # sanity pin: the planted pages' keys point along q, so the oracle's
    # bounding-box ranking must keep all of them within the 16-page budget
    cfg = W.CONFIGS["tiny"]
    seq = W.sequence(cfg, 0, 2048, seed=0)
    assert len(seq.planted) == 4
    for h in range(cfg.num_kv_heads):
        K = W.widen(seq.k[:, h], cfg.dtype)
        lo, hi = oracle.page_bounds(K, cfg.page_size)
        q = W.widen(seq.q[h:h + 1], cfg.dtype)
        sel = oracle.select_pages(oracle.page_scores(q, lo, hi), 16)
        assert set(seq.planted.tolist()) <= set(sel.tolist())
