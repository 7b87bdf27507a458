"""gdn_chunk_fwd_noalloc: the prefill for callers that cannot allocate device memory.

Such callers (code inside a framework that owns the device memory pool, a process that must not
grow after start-up, a host program holding only raw pointers) cannot hand gdn_chunk_fwd a
workspace; this entry point uses the library's fixed scratch array instead.  The test calls it
through the C ABI twice in a row and checks both results against gdn_chunk_fwd with a workspace,
and that sizes beyond the array are refused.  The file name makes pytest collect it last.
"""
import pytest
import torch

import gated_deltanet_recurrence_gb300 as gdn
from gated_deltanet_recurrence_gb300 import synthetic
from tests._util import TOL_BF16, cu_list, oracle_gates, rel_l2_states, rel_l2_tokens

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_twice():
    cfg = synthetic.workload("varlen", lengths=[700, 64, 1, 257], num_seqs=4, H=8, d=128,
                             dtype=torch.bfloat16, seed=41, gate=True)
    inp = synthetic.prefill_inputs(cfg)
    g32, b32 = oracle_gates(inp)
    dev = "cuda"
    q, k, v, z = (inp[n].to(dev) for n in ("q", "k", "v", "z"))
    g, b, cu, S0 = g32.to(dev), b32.to(dev), inp["cu_seqlens"].to(dev), inp["initial_state"].to(dev)
    ws_need = gdn.lib().gdn_chunk_fwd_workspace_size(4, inp["total_T"], 8, 128, 128, gdn.GDN_BF16)
    assert 0 < ws_need <= 64 * 1024 * 1024
    ref_out, ref_S = gdn.gdn_chunk_fwd(q, k, v, g, b, cu_seqlens=cu, initial_state=S0, gate_z=z,
                                       out_dtype=torch.float32)
    for _ in range(2):
        out = torch.full(ref_out.shape, float("nan"), device=dev)
        Sf = torch.full(ref_S.shape, float("nan"), device=dev)
        gdn.gdn_chunk_fwd_noalloc(q, k, v, g, b, cu_seqlens=cu, initial_state=S0, final_state=Sf,
                                  gate_z=z, out=out)
        assert gdn.gdn_get_device_error() == 0
        cu_l = cu_list(inp)
        assert rel_l2_tokens(out.cpu(), ref_out.cpu(), cu_l) <= TOL_BF16 / 100
        assert rel_l2_states(Sf.cpu(), ref_S.cpu()) <= TOL_BF16 / 100


def test_noalloc_refuses_sizes_beyond_the_array():
    T, H = 64 * 2048, 16          # needs about 1.3 GB of scratch
    x = torch.zeros(1, H, 128, dtype=torch.bfloat16, device="cuda")
    gf = torch.zeros(1, H, device="cuda")
    out = torch.zeros(1, H, 128, dtype=torch.bfloat16, device="cuda")
    L = gdn.lib()
    rc = L.gdn_chunk_fwd_noalloc(x.data_ptr(), x.data_ptr(), x.data_ptr(), gf.data_ptr(), gf.data_ptr(),
                                 None, 1, T, H, H, 128, 128, gdn.GDN_BF16, 0, 0.0, 1, None, None, None,
                                 None, None, None, None, 1e-6, out.data_ptr(), gdn.GDN_BF16, None)
    assert rc == -4  # GDN_ERR_WORKSPACE, rejected before any launch
