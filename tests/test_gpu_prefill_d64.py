"""GPU parity of the tensor-core prefill at head size 64 (bf16 q/k/v) against the fp64 oracle.

With d_k = d_v = 64 the tensor-core kernels run their 128-wide tiles with the columns past 64 filled
with zeros (the TMA loads past the tensor's last column read zeros); the head size enters only the
global-memory indexing, the q/k norms and the gate's mean over d_v.  These cases cover that path
the way the d = 128 tests cover theirs: the bench's head-size-64 workload in full, ragged and
empty sequences with initial states and norm weights, bf16 outputs leaving through the tensor
stores, grouped heads, a decay per key channel, the fused short convolution with history, and the
fused and two-kernel forms agreeing bit for bit."""
import numpy as np
import pytest
import torch

import gated_deltanet_recurrence_gb300 as gdn
from gated_deltanet_recurrence_gb300 import synthetic
from tests._util import (TOL_BF16, cu_list, oracle_conv_qkv, oracle_gates, oracle_prefill,
                         rel_l2_states, rel_l2_tokens)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _cfg(lengths, H, seed, **kw):
    return synthetic.workload("varlen", lengths=lengths, num_seqs=len(lengths), H=H, d=64,
                              dtype=torch.bfloat16, seed=seed, **kw)


def _run(inp, g32, b32, out_dtype=torch.float32, weight=None, conv_out=None):
    cs = inp["conv_state"].to(DEV) if inp.get("conv_state") is not None else None
    out, Sf = gdn.gdn_chunk_fwd(
        inp["q"].to(DEV), inp["k"].to(DEV), inp["v"].to(DEV), g32.to(DEV), b32.to(DEV),
        cu_seqlens=inp["cu_seqlens"].to(DEV) if inp["cu_seqlens"] is not None else None,
        num_seqs=inp["num_seqs"],
        initial_state=inp["initial_state"].to(DEV) if inp["initial_state"] is not None else None,
        conv_weight=inp["conv_weight"].to(DEV) if inp.get("conv_weight") is not None else None,
        conv_state=cs, conv_state_out=conv_out,
        gate_z=inp["z"].to(DEV) if inp["z"] is not None else None,
        norm_weight=weight.to(DEV) if weight is not None else None, out_dtype=out_dtype)
    assert gdn.gdn_get_device_error() == 0
    return out.float().cpu(), Sf.cpu()


def _check(inp, out_dtype=torch.float32, weight=None):
    g32, b32 = oracle_gates(inp)
    out, Sf = _run(inp, g32, b32, out_dtype=out_dtype, weight=weight)
    y_ref, S_ref = oracle_prefill(inp, g32, b32, weight=weight)
    cu = cu_list(inp)
    e_o, e_s = rel_l2_tokens(out, y_ref, cu), rel_l2_states(Sf, S_ref)
    assert e_o <= TOL_BF16 and e_s <= TOL_BF16, (e_o, e_s)


def test_workspace_and_path():
    """bf16 at d = 64 takes the tensor-core path: it asks for the same workspace as d = 128."""
    L = gdn.lib()
    assert L.gdn_chunk_fwd_workspace_size(2, 8192, 16, 64, 64, gdn.GDN_BF16) == \
        L.gdn_chunk_fwd_workspace_size(2, 8192, 16, 128, 128, gdn.GDN_BF16) > 0


def test_prefill_d64_full_size():
    """The bench's head-size-64 workload (B=2, T=4096, H=16, bf16, fused gate, bf16 output), every
    token and head."""
    _check(synthetic.prefill_inputs("prefill_d64"), out_dtype=torch.bfloat16)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_ragged_sequences_states_weights(out_dtype):
    inp = synthetic.prefill_inputs(_cfg([0, 1, 63, 64, 65, 200, 128, 3], 3, seed=81, gate=True,
                                        init_state=True))
    _check(inp, out_dtype=out_dtype, weight=torch.linspace(0.25, 2.0, 64))


def test_grouped_heads():
    _check(synthetic.prefill_inputs(_cfg([200, 64, 1, 0, 130], 8, seed=82, Hk=2, gate=True,
                                         init_state=True)), out_dtype=torch.bfloat16)


def test_per_channel_decay():
    _check(synthetic.prefill_inputs(_cfg([150, 64, 1, 0, 65], 3, seed=83, per_channel=True, gate=True,
                                         init_state=True)))


@pytest.mark.parametrize("with_state", [False, True])
def test_conv_with_history(with_state):
    lengths = [0, 1, 2, 3, 64, 65, 200]
    H, Hk = 4, 2
    inp = synthetic.prefill_inputs(_cfg(lengths, H, seed=84, Hk=Hk, conv=True, conv_state=with_state,
                                        gate=True, init_state=True))
    C = synthetic.conv_dim(H, Hk, 64)
    conv_out = torch.full((len(lengths), C, 3), 7.0, device=DEV)
    g32, b32 = oracle_gates(inp)
    out, Sf = _run(inp, g32, b32, conv_out=conv_out)
    y_ref, S_ref = oracle_prefill(inp, g32, b32)
    cu = cu_list(inp)
    assert rel_l2_tokens(out, y_ref, cu) <= TOL_BF16
    assert rel_l2_states(Sf, S_ref) <= TOL_BF16
    _, _, _, st_ref = oracle_conv_qkv(inp["q"], inp["k"], inp["v"], inp["conv_weight"], inp["conv_state"], cu)
    np.testing.assert_array_equal(conv_out.cpu().double().numpy(), st_ref)


def test_fused_and_two_kernel_forms_agree_bitwise(kernel_forms):
    inp = synthetic.prefill_inputs(_cfg([300, 64, 0, 1000, 65], 4, seed=85, gate=True, init_state=True))
    g32, b32 = oracle_gates(inp)
    outs = []
    for form in (gdn.GDN_FORM_AUTO, gdn.GDN_FORM_ON, gdn.GDN_FORM_OFF):  # fused (export form), fused, two kernels
        kernel_forms.gdn_set_kernel_forms(prefill_fused=form)
        outs.append(_run(inp, g32, b32, out_dtype=torch.bfloat16))
    for o in outs[:2]:
        assert torch.equal(o[0], outs[2][0])
        assert torch.equal(o[1], outs[2][1])
