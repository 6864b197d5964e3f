"""GPU parity of qasa_rebuild_page_bounds (page boxes rebuilt from the pool).

The boxes that the append kernel maintains are wiped (every element NaN), then
rebuilt from the keys in the pool.  Boxes of the pages in use must come back
bit-identical to the append-maintained ones and equal the oracle's boxes
computed from scratch; pages no sequence uses must stay untouched; a decode
step on the rebuilt boxes must give the same ids and outputs bit for bit.
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


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


def _used_pages(case):
    P = case.cfg.page_size
    used = []
    for b, L in enumerate(case.lens):
        used.extend(case.plan.block_table[b, :-(-int(L) // P)].tolist())
    return np.array(sorted(set(used)), dtype=np.int64)


def _decode(case, status):
    return _qasa().sparse_decode_attention(case.cache, case.q_dev, case.bt, case.lens_dev, case.budget_dev,
                                           max_budget=case.max_budget, status=status)


@pytest.mark.parametrize("name,dtype,batch,seed,lens", [
    ("tiny", None, 1, 41, [2041]),                        # f32, d64, partial last page
    ("tinyllama", None, 3, 42, [4096, 1000, 17]),         # f16, d64
    ("gpt2_345m", "bf16", 6, 43, None),                   # bf16, d64, ragged
    ("llama_1b3_32k", None, 2, 44, [3000, 70]),           # bf16, d128, P32, outlier channels
    ("serving_mix", None, 4, 45, None),                   # f16, d128
    ("headline_8k", "f32", 2, 46, [8192, 1001]),          # f32, d128
])
def test_rebuilt_boxes_equal_append_boxes_and_the_oracle(name, dtype, batch, seed, lens):
    qasa = _qasa()
    cfg = W.CONFIGS[name]
    if dtype:
        cfg = dataclasses.replace(cfg, dtype=dtype)
    case = H.make_case(cfg, seed=seed, batch=batch, lens=lens)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_a, sel_a = _decode(case, status)
    ref = case.cache.page_bounds.clone()

    case.cache.page_bounds.fill_(float("nan"))
    qasa.rebuild_page_bounds(case.cache, case.bt, case.lens_dev, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    used = torch.from_numpy(_used_pages(case)).cuda()
    got = case.cache.page_bounds
    assert torch.equal(_bits(got[used]), _bits(ref[used])), "rebuilt boxes differ from the append boxes"
    unused = torch.ones(got.shape[0], dtype=torch.bool, device="cuda")
    unused[used] = False
    assert bool(torch.isnan(got[unused].float()).all()), "a page no sequence uses was written"

    bounds = H.from_torch(got, cfg.dtype)
    P = cfg.page_size
    for b in range(batch):
        N = -(-int(case.lens[b]) // P)
        phys = case.plan.block_table[b, :N]
        for h in range(cfg.num_kv_heads):
            lo, hi = oracle.page_bounds(case.k64(b, h), P)
            assert np.array_equal(W.widen(bounds[phys, h, 0], cfg.dtype), lo), (b, h)
            assert np.array_equal(W.widen(bounds[phys, h, 1], cfg.dtype), hi), (b, h)

    out_r, sel_r = _decode(case, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(sel_a, sel_r)
    assert torch.equal(_bits(out_a), _bits(out_r))


def test_rebuild_of_keys_written_directly_into_the_pool():
    # a "prefill" that stores keys straight into the pool (no append kernel, no
    # boxes), then a bulk rebuild: the decode step matches the oracle
    qasa = _qasa()
    cfg = W.CONFIGS["tinyllama"]
    case = H.make_case(cfg, seed=47, batch=2, lens=[4096, 777])
    P, Hkv = cfg.page_size, cfg.num_kv_heads
    kp = case.cache.k_pool
    kp.fill_(float("nan"))
    for b in range(2):
        L = int(case.lens[b])
        k = H.to_torch(case.seqs[b].k, cfg.dtype).cuda()            # [L, Hkv, d]
        for pg in range(-(-L // P)):
            rows = min(P, L - pg * P)
            phys = int(case.plan.block_table[b, pg])
            kp[phys, :, :rows] = k[pg * P:pg * P + rows].transpose(0, 1)
    case.cache.page_bounds.fill_(float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qasa.rebuild_page_bounds(case.cache, case.bt, case.lens_dev, status=status)
    out, sel = _decode(case, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    out64, sel = H.gpu_out64(out, cfg.dtype), sel.cpu().numpy()
    for b in range(2):
        L = int(case.lens[b])
        for h in range(Hkv):
            K = case.k64(b, h)
            lo, hi = oracle.page_bounds(K, P)
            o_s, o_sel, o_out = oracle.decode_unit(case.q64(b, h), K, case.v64(b, h), lo, hi, L, P,
                                                   int(case.budgets[b]))
            kept = sel[b, h][sel[b, h] >= 0]
            ref = o_out if np.array_equal(kept, o_sel) else oracle.attention(
                case.q64(b, h), K, case.v64(b, h), L, P, kept)
            H.assert_close(out64[b, h * case.G:(h + 1) * case.G], ref, "b=%d h=%d" % (b, h))


def test_rebuild_edge_cases_and_device_errors():
    qasa = _qasa()
    cfg = W.CONFIGS["gpt2_345m"]
    case = H.make_case(cfg, seed=48, batch=3, lens=[0, 1, 300])
    ref = case.cache.page_bounds.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    case.cache.page_bounds.fill_(float("nan"))
    qasa.rebuild_page_bounds(case.cache, case.bt, case.lens_dev, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    used = torch.from_numpy(_used_pages(case)).cuda()
    assert torch.equal(_bits(case.cache.page_bounds[used]), _bits(ref[used]))

    # an out-of-range block-table entry: that page is skipped and reported
    bt = case.bt.clone()
    bt[2, 3] = case.cache.num_phys_pages + 5
    case.cache.page_bounds.fill_(float("nan"))
    qasa.rebuild_page_bounds(case.cache, bt, case.lens_dev, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x1
    good = [int(x) for x in case.plan.block_table[2, :19] if x != case.plan.block_table[2, 3]]
    g = torch.tensor(good, device="cuda")
    assert torch.equal(_bits(case.cache.page_bounds[g]), _bits(ref[g]))

    # a length beyond the block table is clamped and reported
    status.zero_()
    lens = case.lens_dev.clone()
    lens[1] = case.bt.shape[1] * cfg.page_size + 9
    qasa.rebuild_page_bounds(case.cache, case.bt, lens, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x2

    # empty batch: a no-op that needs no pointers
    assert qasa._lib.qasa_rebuild_page_bounds(case.cache.c_ref, None, 1, None, 0, None, None) == 0
