"""The bounded-wait time-out path, made to run out on purpose.

Every wait of the decode kernels on another warp, another CTA or a flag is
bounded; one that gives up sets QASA_DEVERR_TIMEOUT in the status word, the
CTA stops issuing copies, waits (with the long limit) for the copies it has
in flight, and returns.  QASA_WAIT_LIMIT_NS shortens only those waits.  At
1 us the single-launch kernel's TMA producers give up waiting for selections
that take several microseconds, so the time-out path runs every time.  The
call must return, report the time-out, and leave the device usable: the next
calls, with the normal limit, must match the oracle.
"""
import pytest
import torch

from query_aware_sparse_append_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu

TIMEOUT_BIT = 0x8   # QASA_DEVERR_TIMEOUT


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from query_aware_sparse_append_gb300 import build
    build.build()


def _step(case, status):
    from query_aware_sparse_append_gb300 import binding as qasa
    out, sel = qasa.sparse_decode_attention(case.cache, case.q_dev, case.bt, case.lens_dev, case.budget_dev,
                                            max_budget=case.max_budget, status=status)
    torch.cuda.synchronize()
    return out, sel


@pytest.mark.parametrize("name,batch,seed", [("headline_8k", 16, 61), ("serving_mix", 12, 62)])
def test_short_wait_limit_times_out_and_the_device_stays_usable(name, batch, seed, monkeypatch):
    case = H.make_case(W.CONFIGS[name], seed=seed, batch=batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    monkeypatch.setenv("QASA_SINGLE_LAUNCH", "1")
    monkeypatch.setenv("QASA_WAIT_LIMIT_NS", "1000")
    _step(case, status)
    st = int(status.item())
    assert st & TIMEOUT_BIT, "no wait ran out (status %#x)" % st
    assert st & ~TIMEOUT_BIT == 0, "unexpected device error bits %#x" % st

    monkeypatch.delenv("QASA_WAIT_LIMIT_NS")
    for single in ("1", "0"):
        monkeypatch.setenv("QASA_SINGLE_LAUNCH", single)
        status.zero_()
        out, sel = _step(case, status)
        assert int(status.item()) == 0, "single=%s: status %#x" % (single, int(status.item()))
        H.check_units(case, out, sel, None, H.all_units(case), check_bounds=False)
