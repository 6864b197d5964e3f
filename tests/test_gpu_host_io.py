"""The decode step with host inputs and outputs (qasa_sparse_decode_attention_host).

Inputs are staged from page-locked host tensors into the device workspace and
the outputs copied back on the same stream; the kernels are the ones of
qasa_sparse_decode_attention, so out and the kept ids must equal that call's
bit for bit.
"""
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


@pytest.mark.parametrize("name,batch,seed", [("headline_8k", 6, 71), ("serving_mix", 5, 72),
                                             ("gpt2_345m", 9, 73), ("tiny", None, 74)])
def test_host_buffers_match_the_device_call(name, batch, seed):
    from query_aware_sparse_append_gb300 import binding as qasa
    case = H.make_case(W.CONFIGS[name], seed=seed, batch=batch)
    mb = case.max_budget
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_out, ref_sel = qasa.sparse_decode_attention(case.cache, case.q_dev, case.bt, case.lens_dev, case.budget_dev,
                                                    max_budget=mb, status=status)
    q_h = case.q_dev.cpu().pin_memory()
    bt_h = case.bt.cpu().pin_memory()
    lens_h = case.lens_dev.cpu().pin_memory()
    bud_h = case.budget_dev.cpu().pin_memory()
    for call in range(2):
        out_h = torch.full(tuple(ref_out.shape), float("nan"), dtype=ref_out.dtype).pin_memory()
        sel_h = torch.full(tuple(ref_sel.shape), 7, dtype=torch.int32).pin_memory()
        qasa.sparse_decode_attention_host(case.cache, q_h, bt_h, lens_h, bud_h, mb, out_h, sel_h, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(sel_h, ref_sel.cpu()), "call %d" % call
        assert torch.equal(out_h.view(torch.int16 if out_h.element_size() == 2 else torch.int32),
                           ref_out.cpu().view(torch.int16 if out_h.element_size() == 2 else torch.int32))


def test_host_call_checks_its_workspace():
    from query_aware_sparse_append_gb300 import binding as qasa
    case = H.make_case(W.CONFIGS["tinyllama"], seed=75, batch=2)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    q_h = case.q_dev.cpu().pin_memory()
    out_h = torch.empty_like(q_h).pin_memory()
    sel_h = torch.empty((2, case.cfg.num_kv_heads, case.max_budget), dtype=torch.int32).pin_memory()
    with pytest.raises(qasa.QasaError):
        qasa.sparse_decode_attention_host(case.cache, q_h, case.bt.cpu().pin_memory(), case.lens_dev.cpu().pin_memory(),
                                          case.budget_dev.cpu().pin_memory(), case.max_budget, out_h, sel_h,
                                          workspace=small)
