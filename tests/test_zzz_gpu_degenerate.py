"""GPU parity on the method's degenerate values, against the fp64 oracle on the same inputs:
  - zero query and key rows (normalised to zero: such a token writes nothing and reads nothing);
  - beta = 0 (pure decay of the carried state, "6.6 Gated DeltaNet" 6.6.3);
  - alpha = 1 and beta = 1 (no forgetting, full overwrite along each key);
  - near-total decay, log alpha = -30 per token (the carried state vanishes within a token; the
    chunk form's factors e^(G_i - G_j) underflow to zero rather than overflow).
Prefill on the tensor-core path (bf16, d = 128) and the CUDA-core path (fp32, d = 64), with ragged
sequences and an initial state, and the one-token decode.  The file name makes pytest run it last."""
import numpy as np
import pytest
import torch

import gated_deltanet_recurrence_gb300 as gdn
import oracle
from gated_deltanet_recurrence_gb300 import synthetic
from tests._util import (TOL_BF16, TOL_F32, cu_list, oracle_gates, oracle_prefill, rel_l2_states,
                         rel_l2_tokens)

pytestmark = pytest.mark.gpu

MODES = ["zero_qk", "beta_zero", "no_decay_full_write", "total_decay"]


def _degenerate(inp, g32, b32, mode):
    if mode == "zero_qk":            # every 5th query and every 7th key is the zero vector
        inp["q"][::5] = 0
        inp["k"][::7] = 0
    elif mode == "beta_zero":
        b32 = torch.zeros_like(b32)
    elif mode == "no_decay_full_write":
        g32, b32 = torch.zeros_like(g32), torch.ones_like(b32)
    elif mode == "total_decay":
        g32 = torch.full_like(g32, -30.0)
    return inp, g32, b32


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.float32)])
def test_prefill_degenerate_values(mode, d, dtype):
    cfg = synthetic.workload("varlen", lengths=[200, 67, 1], num_seqs=3, H=4, d=d, dtype=dtype,
                             seed=90 + d, gate=False, init_state=True, state_std=0.3)
    inp = synthetic.prefill_inputs(cfg)
    g32, b32 = oracle_gates(inp)
    inp, g32, b32 = _degenerate(inp, g32, b32, mode)
    dev = "cuda"
    out, Sf = gdn.gdn_chunk_fwd(inp["q"].to(dev), inp["k"].to(dev), inp["v"].to(dev), g32.to(dev),
                                b32.to(dev), cu_seqlens=inp["cu_seqlens"].to(dev),
                                initial_state=inp["initial_state"].to(dev), out_dtype=torch.float32)
    assert gdn.gdn_get_device_error() == 0
    out, Sf = out.cpu(), Sf.cpu()
    assert torch.isfinite(out).all() and torch.isfinite(Sf).all()
    y_ref, S_ref = oracle_prefill(inp, g32, b32, gate=False)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert rel_l2_tokens(out, y_ref, cu_list(inp)) <= tol
    assert rel_l2_states(Sf, S_ref) <= tol
    if mode == "zero_qk":            # a zero query reads nothing
        assert torch.count_nonzero(out[::5]) == 0


@pytest.mark.parametrize("mode", MODES)
def test_decode_degenerate_values(mode):
    cfg = synthetic.workload("decode", N=9, H=4, d=128, dtype=torch.bfloat16, seed=95)
    inp = synthetic.decode_inputs(cfg)
    g32, b32 = oracle_gates(inp)
    inp, g32, b32 = _degenerate(inp, g32, b32, mode)
    state = inp["state"].cuda()
    y = gdn.gdn_recurrent_step(inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda(), g32.cuda(),
                               b32.cuda(), state, out_dtype=torch.float32)
    assert gdn.gdn_get_device_error() == 0
    y, S = y.cpu(), state.cpu()
    assert torch.isfinite(y).all() and torch.isfinite(S).all()
    y_ref, S_ref = oracle.recurrent_step(inp["q"], inp["k"], inp["v"], g32, b32, inp["state"])
    yd = y.double().numpy().reshape(-1, 128)
    yr = np.asarray(y_ref).reshape(yd.shape)
    nz = np.linalg.norm(yr, axis=1) > 0
    assert np.max(np.linalg.norm(yd[nz] - yr[nz], axis=1) / np.linalg.norm(yr[nz], axis=1)) <= TOL_BF16
    assert np.abs(yd[~nz]).max(initial=0.0) == 0.0
    assert rel_l2_states(S, S_ref) <= TOL_BF16
