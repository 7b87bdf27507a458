"""gdn_chunk_fwd_noalloc: the prefill for callers that cannot allocate device memory.

Such callers (code inside a framework that owns the device memory pool, a process that must not
grow after start-up, a host program holding only raw pointers) cannot hand gdn_chunk_fwd a
workspace; this entry point uses the library's fixed scratch array instead.  The test calls it
through the C ABI twice on the same inputs, with a call on a different, larger workload in between
(so the shared array holds other data when the second call starts), and checks every result
against gdn_chunk_fwd with a workspace and against the fp64 oracle.  It runs both kernel forms that
use the array: the fused cooperative launch and the two-kernel form.  Sizes beyond the array are
refused.  The file name makes pytest collect it last.
"""
import pytest
import torch

import gated_deltanet_recurrence_gb300 as gdn
from gated_deltanet_recurrence_gb300 import synthetic
from tests._util import (TOL_BF16, cu_list, oracle_gates, oracle_prefill, rel_l2_states,
                         rel_l2_tokens)

pytestmark = pytest.mark.gpu


def _case(lengths, H, seed):
    cfg = synthetic.workload("varlen", lengths=lengths, num_seqs=len(lengths), H=H, d=128,
                             dtype=torch.bfloat16, seed=seed, gate=True)
    inp = synthetic.prefill_inputs(cfg)
    g32, b32 = oracle_gates(inp)
    dev = "cuda"
    t = dict(q=inp["q"].to(dev), k=inp["k"].to(dev), v=inp["v"].to(dev), g=g32.to(dev), b=b32.to(dev),
             cu=inp["cu_seqlens"].to(dev), S0=inp["initial_state"].to(dev), z=inp["z"].to(dev))
    return inp, g32, b32, t


def _noalloc(t, H, d=128):
    T = t["q"].shape[0]
    n = t["cu"].numel() - 1
    out = torch.full((T, H, d), float("nan"), device="cuda")
    Sf = torch.full((n, H, d, d), float("nan"), device="cuda")
    gdn.gdn_chunk_fwd_noalloc(t["q"], t["k"], t["v"], t["g"], t["b"], cu_seqlens=t["cu"],
                              initial_state=t["S0"], final_state=Sf, gate_z=t["z"], out=out)
    assert gdn.gdn_get_device_error() == 0
    return out.cpu(), Sf.cpu()


@pytest.mark.parametrize("form", ["fused", "two-kernel"])
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(form, kernel_forms):
    kernel_forms.gdn_set_kernel_forms(prefill_fused=gdn.GDN_FORM_AUTO if form == "fused" else gdn.GDN_FORM_OFF)
    H = 8
    inp, g32, b32, t = _case([700, 64, 1, 257], H, seed=41)
    ws_need = gdn.lib().gdn_chunk_fwd_workspace_size(4, inp["total_T"], H, 128, 128, gdn.GDN_BF16)
    assert 0 < ws_need <= 64 * 1024 * 1024
    ref_out, ref_S = gdn.gdn_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["b"], cu_seqlens=t["cu"],
                                       initial_state=t["S0"], gate_z=t["z"], out_dtype=torch.float32)
    ref_out, ref_S = ref_out.cpu(), ref_S.cpu()
    y64, S64 = oracle_prefill(inp, g32, b32)
    # another workload (other lengths, heads and seed, more tokens) fills the array in between
    other = _case([900, 333, 64, 1000, 5], 6, seed=42)[3]
    cu_l = cu_list(inp)
    for rep in range(2):
        out, Sf = _noalloc(t, H)
        assert rel_l2_tokens(out, ref_out, cu_l) <= TOL_BF16 / 100
        assert rel_l2_states(Sf, ref_S) <= TOL_BF16 / 100
        assert rel_l2_tokens(out, y64, cu_l) <= TOL_BF16
        assert rel_l2_states(Sf, S64) <= TOL_BF16
        if rep == 0:
            _noalloc(other, 6)


def test_noalloc_refuses_sizes_beyond_the_array():
    T, H = 64 * 2048, 16
    assert gdn.lib().gdn_chunk_fwd_workspace_size(1, T, H, 128, 128, gdn.GDN_BF16) > 64 * 1024 * 1024
    x = torch.zeros(1, H, 128, dtype=torch.bfloat16, device="cuda")
    gf = torch.zeros(1, H, device="cuda")
    out = torch.zeros(1, H, 128, dtype=torch.bfloat16, device="cuda")
    L = gdn.lib()
    rc = L.gdn_chunk_fwd_noalloc(x.data_ptr(), x.data_ptr(), x.data_ptr(), gf.data_ptr(), gf.data_ptr(),
                                 None, 1, T, H, H, 128, 128, gdn.GDN_BF16, 0, 0.0, 1, None, None, None,
                                 None, None, None, None, 1e-6, out.data_ptr(), gdn.GDN_BF16, None)
    assert rc == -4  # GDN_ERR_WORKSPACE, rejected before any launch
