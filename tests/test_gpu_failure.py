"""GPU failure handling without a fault: the bounded device wait that every tensor-core kernel
uses gives up on a phase that nothing completes, reports GDN_ERR_TIMEOUT through a status word the
host reads, and leaves the context usable (a decode step afterwards still matches the oracle)."""
import numpy as np
import pytest
import torch

import gated_deltanet_recurrence_gb300 as gdn
import oracle
from gated_deltanet_recurrence_gb300 import synthetic
from tests._util import TOL_F32, oracle_gates, rel_l2_states

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ns", [20_000, 2_000_000])
def test_bounded_wait_gives_up_and_the_context_survives(limit_ns):
    status = torch.full((1,), 1, dtype=torch.int32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    gdn.gdn_selftest_bounded_wait(limit_ns, status)
    e1.record()
    torch.cuda.synchronize()
    assert status.item() == -6                     # GDN_ERR_TIMEOUT: the wait gave up
    ms = e0.elapsed_time(e1)
    # the bound is kept in SM cycles at 2.1 GHz, so it lasts at least limit_ns at any clock up to
    # that, and a suspended poll adds at most 0.1 ms
    assert 0.95 * limit_ns * 1e-6 <= ms < 1000.0, ms
    assert gdn.gdn_get_device_error() == 0         # the library's own error word is untouched

    cfg = synthetic.workload("decode", N=5, H=4, d=128, dtype=torch.float32, seed=13)
    inp = synthetic.decode_inputs(cfg)
    g32, b32 = oracle_gates(inp)
    state = inp["state"].cuda()
    y = gdn.gdn_recurrent_step(inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda(), g32.cuda(),
                               b32.cuda(), state, out_dtype=torch.float32)
    assert gdn.gdn_get_device_error() == 0
    y_ref, S_ref = oracle.recurrent_step(inp["q"], inp["k"], inp["v"], g32, b32, inp["state"])
    yd = y.cpu().double().numpy().reshape(-1, 128)
    yr = np.asarray(y_ref).reshape(yd.shape)
    assert np.max(np.linalg.norm(yd - yr, axis=1) / np.linalg.norm(yr, axis=1)) <= TOL_F32
    assert rel_l2_states(state.cpu(), S_ref) <= TOL_F32
