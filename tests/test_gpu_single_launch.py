"""The decode step as one launch against the same step as two kernels.

qasa_sparse_decode_attention runs scoring, selection and attention in one
cooperative persistent kernel; with QASA_SINGLE_LAUNCH=0 it runs the selection
kernel and then the attention kernel.  Both use the same scoring and selection
code, so kept ids and scores must agree bit for bit; the attention outputs may
differ in summation order (a different number of consumer warps) and must
agree within the output tolerance.  The one-launch form has its own selector
code path (selector warps, bulk-copy box staging, ready flags), so its kept
ids, scores and outputs are also checked against the oracle at every unit.
"""
import os

import numpy as np
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


def _run(case, single, scores=True):
    from query_aware_sparse_append_gb300 import binding as qasa
    old = os.environ.get("QASA_SINGLE_LAUNCH")
    os.environ["QASA_SINGLE_LAUNCH"] = "1" if single else "0"
    try:
        maxp = case.bt.shape[1]
        sc = torch.full((case.cfg.batch, case.cfg.num_kv_heads, maxp), float("nan"), device="cuda") \
            if scores else None
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out, sel = qasa.sparse_decode_attention(case.cache, case.q_dev, case.bt, case.lens_dev,
                                                case.budget_dev, max_budget=case.max_budget, scores=sc,
                                                status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, qasa.decode_device_errors(int(status.item()))
        return out, sel, sc
    finally:
        if old is None:
            del os.environ["QASA_SINGLE_LAUNCH"]
        else:
            os.environ["QASA_SINGLE_LAUNCH"] = old


@pytest.mark.parametrize("name,batch,seed", [
    ("tiny", None, 51),              # 64 kept pages over 152 CTAs: most ranges hold one page or none
    ("tinyllama", 5, 52),
    ("gpt2_345m", 40, 53),           # G = 1: FFMA scoring and consumers
    ("llama_1b3_32k", 2, 54),        # units split across many CTAs
    ("serving_mix", 24, 55),         # ragged lengths and budgets
    ("headline_8k", 16, 56),
])
def test_one_launch_equals_two_launches(name, batch, seed):
    case = H.make_case(W.CONFIGS[name], seed=seed, batch=batch)
    o1, s1, c1 = _run(case, True)
    o2, s2, c2 = _run(case, False)
    assert torch.equal(s1, s2), "kept ids differ between one and two launches"
    N = W.num_pages(case.lens, case.cfg.page_size)
    for b in range(case.cfg.batch):
        assert torch.equal(c1[b, :, :N[b]], c2[b, :, :N[b]])
    H.assert_close(H.gpu_out64(o1, case.cfg.dtype), H.gpu_out64(o2, case.cfg.dtype), "one vs two launches")
    # the one-launch result against the oracle at every unit: kept sets (tie
    # rule), scores (fp32 bound) and outputs
    H.check_units(case, o1, s1, c1, H.all_units(case))


def test_one_launch_with_empty_sequences_and_full_budgets():
    cfg = W.CONFIGS["serving_mix"]
    lens = [0, 700, 16384, 0, 513, 9000]
    budgets = [5, 1000, 100, 3, 2, 1]
    case = H.make_case(cfg, seed=57, batch=len(lens), lens=lens, budgets=budgets)
    o1, s1, _ = _run(case, True, scores=False)
    o2, s2, _ = _run(case, False, scores=False)
    assert torch.equal(s1, s2)
    assert bool((s1[0] == -1).all()) and bool((s1[3] == -1).all())
    g = H.gpu_out64(o1, cfg.dtype)
    assert np.all(g[0] == 0) and np.all(g[3] == 0)
    H.assert_close(g, H.gpu_out64(o2, cfg.dtype), "one vs two launches")
    H.check_units(case, o1, s1, None, H.all_units(case))


def test_one_launch_repeated_calls_reuse_the_workspace():
    # the ready flags and tickets are cleared on the stream before every launch
    from query_aware_sparse_append_gb300 import binding as qasa
    case = H.make_case(W.CONFIGS["headline_8k"], seed=58, batch=12)
    ws = qasa.alloc_workspace(case.cache, 12, case.cfg.num_q_heads, case.bt.shape[1])
    ws.fill_(0x5A)   # garbage from an unrelated user of the buffer
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(3):
        out, sel = qasa.sparse_decode_attention(case.cache, case.q_dev, case.bt, case.lens_dev, case.budget_dev,
                                                max_budget=case.max_budget, workspace=ws, status=status)
        outs.append((out.clone(), sel.clone()))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for out, sel in outs[1:]:
        assert torch.equal(sel, outs[0][1])
        assert torch.equal(out.view(torch.int16), outs[0][0].view(torch.int16))
    H.check_units(case, outs[-1][0], outs[-1][1], None, H.all_units(case), check_bounds=False)
