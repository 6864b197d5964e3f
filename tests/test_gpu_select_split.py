"""Page selection by one CTA per unit against a cluster of CTAs per unit.

For small batches qasa_select_pages runs every (sequence, KV head) on a
cluster of four CTAs that score a quarter of its 16-page tiles each into the
first CTA's shared memory, which then selects; for large batches one CTA
scores and selects a unit.  QASA_SELECT_SPLIT forces either form.  Every page
score is computed by the same code whichever CTA runs it, so scores and kept
ids must agree bit for bit, and the decode step's output too (the attention
kernel is the same).  The other GPU tests check both forms against the oracle:
their small batches take the cluster form, the bench-sized ones the other.
"""
import dataclasses

import pytest
import torch

from query_aware_sparse_append_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from query_aware_sparse_append_gb300 import build
    build.build()


def _select(case, split, monkeypatch):
    from query_aware_sparse_append_gb300 import binding as qasa
    monkeypatch.setenv("QASA_SELECT_SPLIT", str(split))
    maxp = case.bt.shape[1]
    sc = torch.full((case.cfg.batch, case.cfg.num_kv_heads, maxp), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sel = qasa.select_pages(case.cache, case.q_dev, case.bt, case.lens_dev, case.budget_dev, case.max_budget,
                            scores=sc, status=status)
    out, sel2 = qasa.sparse_decode_attention(case.cache, case.q_dev, case.bt, case.lens_dev, case.budget_dev,
                                             max_budget=case.max_budget, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, qasa.decode_device_errors(int(status.item()))
    assert torch.equal(sel, sel2)
    return sel, sc, out


def _bits(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32)


@pytest.mark.parametrize("name,dtype,batch,lens,budgets", [
    ("tiny", None, None, None, None),                        # fp32 boxes: FFMA scoring
    ("tinyllama", None, 3, None, None),                      # d64, G8
    ("llama_1b3_32k", None, 2, [32768, 20000], None),        # bf16, P32, 1024 pages
    ("headline_8k", "e4m3", 4, None, None),                  # FP8 boxes
    ("gpt2_345m", None, 2, None, None),                      # G = 1, 16 KV heads
    ("serving_mix", None, 7, [0, 700, 16384, 17, 513, 9000, 33], [5, 1000, 100, 3, 2, 1, 40]),
])
def test_cluster_selection_equals_one_cta_per_unit(name, dtype, batch, lens, budgets, monkeypatch):
    cfg = W.CONFIGS[name]
    if dtype:
        cfg = dataclasses.replace(cfg, dtype=dtype)
    case = H.make_case(cfg, seed=81, batch=batch, lens=lens, budgets=budgets)
    s1, c1, o1 = _select(case, 1, monkeypatch)
    s4, c4, o4 = _select(case, 4, monkeypatch)
    assert torch.equal(s1, s4), "kept ids differ between the two forms"
    assert torch.equal(_bits(c1), _bits(c4)), "scores differ between the two forms"
    assert torch.equal(_bits(o1), _bits(o4))
