"""Page selection is independent of how its work is split over the grid.

The selection kernel splits the flattened 16-page tiles of all units over the
warps of its grid; a unit's tiles may be scored by several warps of several
CTAs, and the warp whose tile count completes the unit's ticket selects it.
QASA_SELECT_CTAS forces the grid size, which moves every split point and
every ticket winner.  Every page score is computed by the same code whichever
warp runs its tile, so scores and kept ids must agree bit for bit across grid
sizes, and the decode step's output too (the attention kernel is the same).
The other GPU tests check the selection against the oracle.
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


def _select(case, ctas, monkeypatch):
    from query_aware_sparse_append_gb300 import binding as qasa
    if ctas:
        monkeypatch.setenv("QASA_SELECT_CTAS", str(ctas))
    else:
        monkeypatch.delenv("QASA_SELECT_CTAS", raising=False)
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
def test_selection_does_not_depend_on_the_grid(name, dtype, batch, lens, budgets, monkeypatch):
    cfg = W.CONFIGS[name]
    if dtype:
        cfg = dataclasses.replace(cfg, dtype=dtype)
    case = H.make_case(cfg, seed=81, batch=batch, lens=lens, budgets=budgets)
    s0, c0, o0 = _select(case, None, monkeypatch)
    for ctas in (1, 3, 37, 304):
        s1, c1, o1 = _select(case, ctas, monkeypatch)
        assert torch.equal(s0, s1), "kept ids differ with %d CTAs" % ctas
        assert torch.equal(_bits(c0), _bits(c1)), "scores differ with %d CTAs" % ctas
        assert torch.equal(_bits(o0), _bits(o1))
