"""The allocation-free decode entry point (library-owned scratch buffer).

qasa_sparse_decode_attention_noalloc serves callers that cannot allocate device
memory (a host framework owns all of it, or a device-synchronising cudaMalloc
is not allowed where they run): it runs the decode step with the library's
fixed device buffer instead of a caller workspace.  These tests call it through
the C ABI and compare it with qasa_sparse_decode_attention on the same inputs,
twice in a row (the buffer is shared and keeps the previous call's contents),
and each call's result with the CPU oracle.
This file is collected last on purpose: it must pass on its own in a fresh
process and after every other test.
"""
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


@pytest.mark.parametrize("name,batch,seed", [("headline_8k", 6, 21), ("serving_mix", 5, 22),
                                             ("gpt2_345m", 9, 23)])
def test_noalloc_matches_the_workspace_entry_point_twice(name, batch, seed):
    from query_aware_sparse_append_gb300 import binding as qasa
    case = H.make_case(W.CONFIGS[name], seed=seed, batch=batch)
    mb = case.max_budget
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_out, ref_sel = qasa.sparse_decode_attention(case.cache, case.q_dev, case.bt, case.lens_dev,
                                                    case.budget_dev, max_budget=mb, status=status)
    torch.cuda.synchronize()
    ref = H.gpu_out64(ref_out, case.cfg.dtype)
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        sel = torch.full_like(ref_sel, 7)
        code = qasa.sparse_decode_attention_noalloc(case.cache, case.q_dev, case.bt, case.lens_dev,
                                                    case.budget_dev, mb, out, sel, status=status)
        torch.cuda.synchronize()
        assert code == 0, qasa.status_string(code)
        assert int(status.item()) == 0
        assert torch.equal(sel, ref_sel), "call %d: kept pages differ" % call
        H.assert_close(H.gpu_out64(out, case.cfg.dtype), ref, "no-alloc call %d" % call)
        # and against the oracle at every unit (kept sets under the tie rule, outputs)
        H.check_units(case, out, sel, None, H.all_units(case), check_bounds=False)


def test_noalloc_rejects_shapes_beyond_its_buffer():
    from query_aware_sparse_append_gb300 import binding as qasa
    case = H.make_case(W.CONFIGS["tinyllama"], seed=24, batch=2)
    # a batch whose split-K partials need more than the fixed buffer; the call
    # must refuse before launching anything (the tensors are never read)
    big = 8192
    need = qasa.workspace_size(case.cache, big, case.cfg.num_q_heads, case.bt.shape[1])
    assert need > qasa_noalloc_bytes()
    q = torch.empty((big, case.cfg.num_q_heads, case.cfg.head_dim), dtype=torch.float16, device="cuda")
    bt = torch.zeros((big, case.bt.shape[1]), dtype=torch.int32, device="cuda")
    lens = torch.zeros(big, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    sel = torch.empty((big, case.cfg.num_kv_heads, 8), dtype=torch.int32, device="cuda")
    code = qasa.sparse_decode_attention_noalloc(case.cache, q, bt, lens, lens, 8, out, sel)
    assert code == 6, qasa.status_string(code)      # QASA_ERR_WORKSPACE


def qasa_noalloc_bytes():
    import re
    import os
    text = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                             "include", "qasa.h")).read()
    m = re.search(r"#define QASA_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    return int(m.group(1)) << int(m.group(2))
