"""The bounded waits of the bulk (TMA) dispatch kernels give up instead of hanging: a wait
on an mbarrier that nothing completes ends after its wall-clock limit with MOE_ERR_TIMEOUT
in the status word, and the context stays usable. No fault is involved: the barrier is a
plain shared-memory mbarrier that simply never receives its arrival."""
import time

import numpy as np
import pytest
import torch

import oracle
from workloads import make_case

from _harness import moe, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_returns_when_the_phase_completes():
    m = moe()
    st = m.new_status()
    m.moe_wait_timeout_check(st, 10 ** 9, complete=True)
    torch.cuda.synchronize()
    assert int(st.item()) == m.MOE_OK


@pytest.mark.parametrize("limit_ms", [2, 50])
def test_bounded_wait_gives_up_after_its_limit(limit_ms):
    m = moe()
    st = m.new_status()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record()
    m.moe_wait_timeout_check(st, limit_ms * 10 ** 6, complete=False)
    e1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    assert int(st.item()) == m.MOE_ERR_TIMEOUT
    waited_ms = e0.elapsed_time(e1)
    assert limit_ms * 0.9 <= waited_ms < limit_ms + 200, waited_ms
    assert wall < 5.0, wall

    # the context is still usable: a bulk-path dispatch right after matches the oracle
    w = make_case(1100, 512, 16, 4, seed=81, quant="fp8g128")
    x, ids, _ = to_dev(w)
    d = m.MoEDispatcher(w.T, w.H, w.K, w.E, quant="fp8g128")
    d.route_dispatch(x, ids)
    om = oracle.route_meta(w.topk_ids, w.E)
    oq, osc = oracle.dispatch("normal", "fp8g128", w.x, w.topk_ids, om, w.E)
    torch.cuda.synchronize()
    d.check()
    n = om.num_valid
    assert np.array_equal(d.out_q[:n].cpu().numpy(), oq[:n])
    assert np.array_equal(d.out_scales[:n].cpu().numpy().view(np.uint32), osc[:n].view(np.uint32))
