"""The decode step with host inputs and outputs (qasa_sparse_decode_attention_host).

Direct form: the kernels read the page-locked host tensors and write the
outputs in host memory themselves.  Staged form (QASA_HOST_DIRECT=0, or
pageable buffers): inputs are copied into the device workspace and the outputs
copied back on the same stream.  Either way the kernels are the ones of
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


def _bits(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32)


def _host_inputs(case, pinned=True):
    def h(t):
        t = t.cpu()
        return t.pin_memory() if pinned else t.clone()
    return h(case.q_dev), h(case.bt), h(case.lens_dev), h(case.budget_dev)


def _host_outputs(ref_out, ref_sel, pinned=True):
    out_h = torch.full(tuple(ref_out.shape), float("nan"), dtype=ref_out.dtype)
    sel_h = torch.full(tuple(ref_sel.shape), 7, dtype=torch.int32)
    return (out_h.pin_memory(), sel_h.pin_memory()) if pinned else (out_h, sel_h)


@pytest.mark.parametrize("form", ["direct", "staged"])
@pytest.mark.parametrize("name,batch,seed", [("headline_8k", 6, 71), ("serving_mix", 5, 72),
                                             ("gpt2_345m", 9, 73), ("tiny", None, 74)])
def test_host_buffers_match_the_device_call(name, batch, seed, form, monkeypatch):
    from query_aware_sparse_append_gb300 import binding as qasa
    monkeypatch.setenv("QASA_HOST_DIRECT", "1" if form == "direct" else "0")
    case = H.make_case(W.CONFIGS[name], seed=seed, batch=batch)
    mb = case.max_budget
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_out, ref_sel = qasa.sparse_decode_attention(case.cache, case.q_dev, case.bt, case.lens_dev, case.budget_dev,
                                                    max_budget=mb, status=status)
    q_h, bt_h, lens_h, bud_h = _host_inputs(case)
    ws = qasa.alloc_host_workspace(case.cache, case.cfg.batch, case.cfg.num_q_heads, case.bt.shape[1], mb)
    for call in range(2):
        out_h, sel_h = _host_outputs(ref_out, ref_sel)
        # pinned host memory is device-addressable on a Grace-Blackwell node
        assert qasa.host_call_is_direct(q_h, bt_h, lens_h, bud_h, out_h, sel_h) == (form == "direct")
        qasa.sparse_decode_attention_host(case.cache, q_h, bt_h, lens_h, bud_h, mb, out_h, sel_h, workspace=ws,
                                          status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(sel_h, ref_sel.cpu()), "call %d" % call
        assert torch.equal(_bits(out_h), _bits(ref_out.cpu()))


def test_pageable_host_buffers_take_the_staged_form():
    from query_aware_sparse_append_gb300 import binding as qasa
    case = H.make_case(W.CONFIGS["headline_8k"], seed=76, batch=3)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_out, ref_sel = qasa.sparse_decode_attention(case.cache, case.q_dev, case.bt, case.lens_dev, case.budget_dev,
                                                    max_budget=case.max_budget, status=status)
    q_h, bt_h, lens_h, bud_h = _host_inputs(case, pinned=False)
    out_h, sel_h = _host_outputs(ref_out, ref_sel, pinned=False)
    assert not qasa.host_call_is_direct(q_h, bt_h, lens_h, bud_h, out_h, sel_h)
    # one pinned output among pageable buffers still stages everything
    assert not qasa.host_call_is_direct(q_h, bt_h, lens_h, bud_h, out_h.pin_memory(), sel_h)
    qasa.sparse_decode_attention_host(case.cache, q_h, bt_h, lens_h, bud_h, case.max_budget, out_h, sel_h,
                                      status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(sel_h, ref_sel.cpu()) and torch.equal(_bits(out_h), _bits(ref_out.cpu()))


def test_direct_form_with_the_single_launch_step(monkeypatch):
    # the one-launch step hands kept ids from scoring CTAs to attention CTAs
    # through the selected buffer, here in host memory
    from query_aware_sparse_append_gb300 import binding as qasa
    case = H.make_case(W.CONFIGS["serving_mix"], seed=77, batch=10)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_out, ref_sel = qasa.sparse_decode_attention(case.cache, case.q_dev, case.bt, case.lens_dev, case.budget_dev,
                                                    max_budget=case.max_budget, status=status)
    monkeypatch.setenv("QASA_HOST_DIRECT", "1")
    q_h, bt_h, lens_h, bud_h = _host_inputs(case)
    for single in ("1", "0"):
        monkeypatch.setenv("QASA_SINGLE_LAUNCH", single)
        out_h, sel_h = _host_outputs(ref_out, ref_sel)
        qasa.sparse_decode_attention_host(case.cache, q_h, bt_h, lens_h, bud_h, case.max_budget, out_h, sel_h,
                                          status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(sel_h, ref_sel.cpu())
        # the one-launch form may sum attention in another order
        H.assert_close(H.gpu_out64(out_h, case.cfg.dtype), H.gpu_out64(ref_out.cpu(), case.cfg.dtype),
                       "host single=%s" % single)


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
