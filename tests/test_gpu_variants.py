"""GPU parity of the grouped-head, per-key-channel-decay and short-convolution options against the
fp64 oracle, through the C ABI, on both prefill paths (tensor-core: bf16, d = 128, one decay per
head; CUDA-core: fp32 or d = 64 or a decay per key channel) and on decode.

The oracle side composes its own pieces: oracle.short_conv over the mixed q|k|v channels, then
oracle.recurrence with Hk query/key heads and g per head or per key channel."""
import numpy as np
import pytest
import torch

import gated_deltanet_recurrence_gb300 as gdn
import oracle
from gated_deltanet_recurrence_gb300 import synthetic
from tests._util import (TOL_BF16, TOL_F32, cu_list, oracle_conv_qkv, oracle_gates, oracle_prefill,
                         rel_l2_states, rel_l2_tokens)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _cfg(lengths, H, d, dtype, seed, **kw):
    return synthetic.workload("varlen", lengths=lengths, num_seqs=len(lengths), H=H, d=d, dtype=dtype,
                              seed=seed, **kw)


def _run_prefill(inp, g32, b32, conv_out=None, out_dtype=torch.float32, gate=True, in_place=False):
    cs = inp["conv_state"].to(DEV) if inp.get("conv_state") is not None else None
    if in_place:
        conv_out = cs
    out, Sf = gdn.gdn_chunk_fwd(
        inp["q"].to(DEV), inp["k"].to(DEV), inp["v"].to(DEV), g32.to(DEV), b32.to(DEV),
        cu_seqlens=inp["cu_seqlens"].to(DEV) if inp["cu_seqlens"] is not None else None,
        num_seqs=inp["num_seqs"],
        initial_state=inp["initial_state"].to(DEV) if inp["initial_state"] is not None else None,
        conv_weight=inp["conv_weight"].to(DEV) if inp.get("conv_weight") is not None else None,
        conv_state=cs, conv_state_out=conv_out,
        gate_z=inp["z"].to(DEV) if (gate and inp["z"] is not None) else None, out_dtype=out_dtype)
    assert gdn.gdn_get_device_error() == 0
    return out.float().cpu(), Sf.cpu(), (conv_out.cpu() if conv_out is not None else None)


def _check_prefill(inp, tol, gate=True, **kw):
    g32, b32 = oracle_gates(inp)
    out, Sf, _ = _run_prefill(inp, g32, b32, gate=gate, **kw)
    y_ref, S_ref = oracle_prefill(inp, g32, b32, gate=gate)
    cu = cu_list(inp)
    e_o, e_s = rel_l2_tokens(out, y_ref, cu), rel_l2_states(Sf, S_ref)
    assert e_o <= tol and e_s <= tol, (e_o, e_s)
    return e_o, e_s


# --------------------------------------------------------------------------------------------
# grouped query/key heads
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("d,dtype,H,Hk", [(128, torch.bfloat16, 8, 2), (128, torch.bfloat16, 6, 1),
                                          (64, torch.float32, 4, 2), (128, torch.float32, 4, 4)])
def test_grouped_heads_prefill(d, dtype, H, Hk):
    inp = synthetic.prefill_inputs(_cfg([200, 64, 1, 0, 130], H, d, dtype, seed=40 + H, Hk=Hk,
                                        gate=True, init_state=True))
    _check_prefill(inp, TOL_F32 if dtype == torch.float32 else TOL_BF16)


def test_grouped_heads_prefill_full_size():
    """The bench's grouped-head workload (B=2, T=4096, H=16, Hk=4, bf16, gate), every head."""
    inp = synthetic.prefill_inputs("prefill_gva")
    _check_prefill(inp, TOL_BF16)


# --------------------------------------------------------------------------------------------
# decay per key channel (CUDA-core prefill; decode)
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("d,dtype", [(64, torch.float32), (128, torch.bfloat16), (128, torch.float32)])
def test_per_channel_decay_prefill(d, dtype):
    inp = synthetic.prefill_inputs(_cfg([150, 64, 1, 0, 65], 3, d, dtype, seed=50 + d, per_channel=True,
                                        gate=True, init_state=True))
    _check_prefill(inp, TOL_F32 if dtype == torch.float32 else TOL_BF16)


def test_per_channel_decay_prefill_sampled_full_size():
    """The bench's per-channel workload (B=2, T=4096, H=16, bf16, gate): the GPU runs all heads,
    the oracle checks 3 heads of both sequences."""
    inp = synthetic.prefill_inputs("prefill_kda")
    g32, b32 = oracle_gates(inp)
    out, Sf, _ = _run_prefill(inp, g32, b32)
    heads = [0, 7, 15]
    y_ref, S_ref = oracle_prefill(inp, g32, b32, heads=heads)
    assert rel_l2_tokens(out[:, heads], y_ref, cu_list(inp)) <= TOL_BF16
    assert rel_l2_states(Sf[:, heads], S_ref) <= TOL_BF16


def test_per_channel_equal_channels_matches_scalar_path():
    """A per-channel decay with all channels equal runs the CUDA-core per-channel kernel; the
    per-head decay of the same values runs the tensor-core path; both must agree to bf16 level."""
    inp = synthetic.prefill_inputs(_cfg([300, 77], 4, 128, torch.bfloat16, seed=59, gate=False))
    g32, b32 = oracle_gates(inp)
    gpc = g32[:, :, None].expand(-1, -1, 128).contiguous()
    out_pc, S_pc, _ = _run_prefill(inp, gpc, b32, gate=False)
    out_h, S_h, _ = _run_prefill(inp, g32, b32, gate=False)
    assert rel_l2_tokens(out_pc, out_h, cu_list(inp)) <= TOL_BF16
    assert rel_l2_states(S_pc, S_h) <= TOL_BF16


# --------------------------------------------------------------------------------------------
# short convolution (prefill)
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("d,dtype,H,Hk", [(128, torch.bfloat16, 4, 2), (128, torch.bfloat16, 2, 2),
                                          (64, torch.float32, 4, 1), (128, torch.float32, 2, 2)])
@pytest.mark.parametrize("with_state", [False, True])
def test_conv_prefill(d, dtype, H, Hk, with_state):
    lengths = [0, 1, 2, 3, 64, 65, 200]
    inp = synthetic.prefill_inputs(_cfg(lengths, H, d, dtype, seed=60 + d + H, Hk=Hk, conv=True,
                                        conv_state=with_state, gate=True, init_state=True))
    C = synthetic.conv_dim(H, Hk, d)
    conv_out = torch.full((len(lengths), C, 3), 7.0, device=DEV)
    g32, b32 = oracle_gates(inp)
    out, Sf, cst = _run_prefill(inp, g32, b32, conv_out=conv_out)
    y_ref, S_ref = oracle_prefill(inp, g32, b32)
    cu = cu_list(inp)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert rel_l2_tokens(out, y_ref, cu) <= tol
    assert rel_l2_states(Sf, S_ref) <= tol
    # the carried history is raw inputs: exact
    _, _, _, st_ref = oracle_conv_qkv(inp["q"], inp["k"], inp["v"], inp["conv_weight"], inp["conv_state"], cu)
    np.testing.assert_array_equal(cst.double().numpy(), st_ref)


def test_conv_prefill_state_in_place_and_resume():
    """Two calls over the halves of each sequence, the convolution history and the state carried
    in place, equal one call over the whole sequences."""
    H, Hk, d = 4, 2, 128
    lengths = [130, 70, 5]
    inp = synthetic.prefill_inputs(_cfg(lengths, H, d, torch.bfloat16, seed=67, Hk=Hk, conv=True,
                                        gate=False, init_state=False))
    g32, b32 = oracle_gates(inp)
    cu = cu_list(inp)
    first = [min(L, [64, 33, 2][n]) for n, L in enumerate(lengths)]
    idx1 = torch.cat([torch.arange(cu[n], cu[n] + first[n]) for n in range(3)])
    idx2 = torch.cat([torch.arange(cu[n] + first[n], cu[n + 1]) for n in range(3)])
    cu1 = torch.tensor(np.concatenate([[0], np.cumsum(first)]), dtype=torch.int32, device=DEV)
    cu2 = torch.tensor(np.concatenate([[0], np.cumsum(np.array(lengths) - first)]), dtype=torch.int32, device=DEV)
    C = synthetic.conv_dim(H, Hk, d)
    cst = torch.zeros(3, C, 3, device=DEV)
    S = torch.zeros(3, H, d, d, device=DEV)
    w = inp["conv_weight"].to(DEV)
    outs = []
    for idx, cuk in ((idx1, cu1), (idx2, cu2)):
        o, _ = gdn.gdn_chunk_fwd(inp["q"][idx].to(DEV), inp["k"][idx].to(DEV), inp["v"][idx].to(DEV),
                                 g32[idx].to(DEV), b32[idx].to(DEV), cu_seqlens=cuk, initial_state=S,
                                 final_state=S, conv_weight=w, conv_state=cst, conv_state_out=cst,
                                 out_dtype=torch.float32)
        outs.append(o.cpu())
    assert gdn.gdn_get_device_error() == 0
    out = torch.empty(inp["total_T"], H, d)
    out[idx1], out[idx2] = outs[0], outs[1]
    y_ref, S_ref = oracle_prefill(inp, g32, b32, gate=False)
    assert rel_l2_tokens(out, y_ref, cu) <= TOL_BF16
    assert rel_l2_states(S.cpu(), S_ref) <= TOL_BF16


def test_conv_prefill_full_size():
    """The bench's convolution workload (B=2, T=4096, H=16, bf16, gate, zero history), every head."""
    inp = synthetic.prefill_inputs("prefill_conv")
    _check_prefill(inp, TOL_BF16)


# --------------------------------------------------------------------------------------------
# decode: grouped heads, per-channel decay, convolution with history
# --------------------------------------------------------------------------------------------

def _decode_case(N, T, H, Hk, d, dtype, per_channel, conv, seed):
    gen = torch.Generator().manual_seed(seed)
    q, k = (torch.randn(N, T, Hk, d, generator=gen).to(dtype) for _ in range(2))
    v = torch.randn(N, T, H, d, generator=gen).to(dtype)
    A_log = torch.rand(H, generator=gen) * np.log(8)
    if per_channel:
        a = torch.randn(N * T, H, d, generator=gen) - 1
        g = oracle.gates_from_logits(a.reshape(-1, H * d), A_log.repeat_interleave(d))
        g = torch.from_numpy(g).float().reshape(N, T, H, d)
    else:
        a = torch.randn(N * T, H, generator=gen) - 1
        g = torch.from_numpy(oracle.gates_from_logits(a, A_log)).float().reshape(N, T, H)
    beta = torch.sigmoid(torch.randn(N, T, H, generator=gen).double()).float()
    S0 = torch.randn(N, H, d, d, generator=gen) * 0.02
    C = synthetic.conv_dim(H, Hk, d)
    w = (torch.rand(C, 4, generator=gen) - 0.5) if conv else None
    cs = torch.randn(N, C, 3, generator=gen) if conv else None
    z = torch.randn(N, T, H, d, generator=gen)
    return q, k, v, g, beta, S0, w, cs, z


def _decode_oracle(q, k, v, g, beta, S0, w, cs, z):
    N, T, Hk, d = q.shape
    H = v.shape[2]
    flat = lambda x: x.reshape(N * T, *x.shape[2:])  # noqa: E731
    cu = np.arange(0, N * T + 1, T, dtype=np.int32)
    qf, kf, vf = flat(q), flat(k), flat(v)
    st = None
    if w is not None:
        qf, kf, vf, st = oracle_conv_qkv(qf, kf, vf, w, cs, cu)
    y, S = oracle.recurrence(qf, kf, vf, flat(g), flat(beta), cu_seqlens=cu, initial_state=S0)
    o = oracle.gate_rmsnorm_silu(y, flat(z)) if z is not None else y
    return o.reshape(N, T, H, d), S, st


@pytest.mark.parametrize("H,Hk,d,dtype,pc,conv", [
    (8, 2, 128, torch.bfloat16, False, False), (4, 4, 128, torch.bfloat16, True, False),
    (4, 4, 64, torch.float32, True, True), (6, 3, 128, torch.bfloat16, True, True),
    (4, 1, 64, torch.float32, False, True)])
def test_decode_step_options(H, Hk, d, dtype, pc, conv):
    N = 9
    q, k, v, g, beta, S0, w, cs, z = _decode_case(N, 1, H, Hk, d, dtype, pc, conv, seed=70 + H + d)
    o_ref, S_ref, st_ref = _decode_oracle(q, k, v, g, beta, S0, w, cs, z)
    S = S0.to(DEV)
    cs_gpu = cs.to(DEV) if conv else None
    cs_out = (cs_gpu if Hk == H else torch.zeros_like(cs_gpu)) if conv else None   # in place when allowed
    out = gdn.gdn_recurrent_step(q[:, 0].to(DEV), k[:, 0].to(DEV), v[:, 0].to(DEV), g[:, 0].to(DEV),
                                 beta[:, 0].to(DEV), S, conv_weight=w.to(DEV) if conv else None,
                                 conv_state=cs_gpu, conv_state_out=cs_out, gate_z=z[:, 0].to(DEV),
                                 out_dtype=torch.float32)
    assert gdn.gdn_get_device_error() == 0
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    y = out.cpu().double().numpy()
    err = np.linalg.norm((y - o_ref[:, 0]).reshape(N * H, d), axis=1) / np.linalg.norm(o_ref[:, 0].reshape(N * H, d), axis=1)
    assert err.max() <= tol
    assert rel_l2_states(S.cpu(), S_ref) <= tol
    if conv:
        np.testing.assert_array_equal(cs_out.cpu().double().numpy(), st_ref)


@pytest.mark.parametrize("H,Hk,d,dtype,pc,conv,T", [
    (8, 2, 128, torch.bfloat16, True, True, 4), (4, 4, 64, torch.float32, True, False, 3),
    (4, 2, 128, torch.bfloat16, False, True, 5)])
def test_multi_step_options(H, Hk, d, dtype, pc, conv, T):
    N, slots = 11, 20
    q, k, v, g, beta, S0, w, cs, z = _decode_case(N, T, H, Hk, d, dtype, pc, conv, seed=80 + T)
    idx = torch.randperm(slots, generator=torch.Generator().manual_seed(3))[:N].to(torch.int32)
    pool = torch.zeros(slots, H, d, d)
    pool[idx.long()] = S0
    C = synthetic.conv_dim(H, Hk, d)
    cpool_in = torch.zeros(slots, C, 3)
    if conv:
        cpool_in[idx.long()] = cs
    pool_gpu = pool.to(DEV)
    cin = cpool_in.to(DEV)
    cout = torch.full_like(cin, 5.0)
    out = gdn.gdn_recurrent_multi_step(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), beta.to(DEV), pool_gpu,
                                       state_indices=idx.to(DEV), conv_weight=w.to(DEV) if conv else None,
                                       conv_state=cin if conv else None, conv_state_out=cout if conv else None,
                                       gate_z=z.to(DEV), out_dtype=torch.float32)
    assert gdn.gdn_get_device_error() == 0
    o_ref, S_ref, st_ref = _decode_oracle(q, k, v, g, beta, S0, w, cs, z)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    y = out.cpu().double().numpy()
    err = (np.linalg.norm((y - o_ref).transpose(0, 2, 1, 3).reshape(N * H, -1), axis=1)
           / np.linalg.norm(o_ref.transpose(0, 2, 1, 3).reshape(N * H, -1), axis=1))
    assert err.max() <= tol
    assert rel_l2_states(pool_gpu.cpu()[idx.long()], S_ref) <= tol
    if conv:
        np.testing.assert_array_equal(cout.cpu()[idx.long()].double().numpy(), st_ref)


@pytest.mark.parametrize("H,Hk,d,dtype,pc,conv,T", [
    (4, 4, 128, torch.bfloat16, False, True, 1), (8, 4, 128, torch.bfloat16, True, True, 1),
    (4, 4, 128, torch.bfloat16, True, False, 4), (4, 2, 128, torch.bfloat16, False, True, 5),
    (4, 4, 128, torch.float32, True, True, 2), (4, 4, 64, torch.float32, True, True, 6)])
def test_multi_step_without_gate(H, Hk, d, dtype, pc, conv, T):
    """The raw output y (no gate): at d = 128 the streamed form's 16-warp layout of the state rows,
    with a decay per key channel, the convolution and grouped heads, one-token blocks (T = 1) and
    four-token blocks; at d = 64 the 4-warp layout.  Outputs, states and the convolution history
    against the oracle."""
    N, slots = 13, 20
    q, k, v, g, beta, S0, w, cs, _ = _decode_case(N, T, H, Hk, d, dtype, pc, conv, seed=140 + T + H)
    idx = torch.randperm(slots, generator=torch.Generator().manual_seed(9))[:N].to(torch.int32)
    pool = torch.zeros(slots, H, d, d)
    pool[idx.long()] = S0
    C = synthetic.conv_dim(H, Hk, d)
    cpool = torch.zeros(slots, C, 3)
    if conv:
        cpool[idx.long()] = cs
    pool_gpu = pool.to(DEV)
    cin = cpool.to(DEV)
    cout = torch.full_like(cin, 5.0)
    out = gdn.gdn_recurrent_multi_step(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), beta.to(DEV), pool_gpu,
                                       state_indices=idx.to(DEV), conv_weight=w.to(DEV) if conv else None,
                                       conv_state=cin if conv else None, conv_state_out=cout if conv else None,
                                       out_dtype=torch.float32)
    assert gdn.gdn_get_device_error() == 0
    o_ref, S_ref, st_ref = _decode_oracle(q, k, v, g, beta, S0, w, cs, None)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    y = out.cpu().double().numpy()
    err = (np.linalg.norm((y - o_ref).transpose(0, 2, 1, 3).reshape(N * H, -1), axis=1)
           / np.linalg.norm(o_ref.transpose(0, 2, 1, 3).reshape(N * H, -1), axis=1))
    assert err.max() <= tol
    assert rel_l2_states(pool_gpu.cpu()[idx.long()], S_ref) <= tol
    if conv:
        np.testing.assert_array_equal(cout.cpu()[idx.long()].double().numpy(), st_ref)


def test_conv_prefill_then_decode_continues_the_sequence():
    """prefill(T) with the convolution, then one decode token on the returned state and history,
    equals the oracle over T + 1 tokens."""
    H, Hk, d, T = 4, 2, 128, 77
    inp = synthetic.prefill_inputs(_cfg([T + 1], H, d, torch.bfloat16, seed=90, Hk=Hk, conv=True,
                                        gate=False, init_state=False))
    g32, b32 = oracle_gates(inp)
    q, k, v = inp["q"].to(DEV), inp["k"].to(DEV), inp["v"].to(DEV)
    w = inp["conv_weight"].to(DEV)
    C = synthetic.conv_dim(H, Hk, d)
    cst = torch.empty(1, C, 3, device=DEV)
    _, S = gdn.gdn_chunk_fwd(q[:T], k[:T], v[:T], g32[:T].to(DEV), b32[:T].to(DEV), conv_weight=w,
                             conv_state_out=cst, out_dtype=torch.float32)
    cst2 = torch.empty_like(cst)
    yd = gdn.gdn_recurrent_step(q[T:], k[T:], v[T:], g32[T:].to(DEV), b32[T:].to(DEV), S, conv_weight=w,
                                conv_state=cst, conv_state_out=cst2, out_dtype=torch.float32)
    assert gdn.gdn_get_device_error() == 0
    y_ref, S_ref = oracle_prefill(inp, g32, b32, gate=False)
    err = np.linalg.norm(yd.cpu().double().numpy()[0] - y_ref[T], axis=1) / np.linalg.norm(y_ref[T], axis=1)
    assert err.max() <= TOL_BF16
    assert rel_l2_states(S.cpu(), S_ref) <= TOL_BF16


@pytest.mark.parametrize("T", [1, 2, 4, 7])
def test_multi_step_conv_history_in_place(T):
    """With H_k == H the convolution history may be updated in place: every read of the input history
    happens before the writes (in the streamed form only the first block reads it, and the lane
    that reads a channel's history writes it).  In place and out of place give the same outputs,
    states and histories, bit for bit."""
    N, H, d, slots = 9, 4, 128, 12
    q, k, v, g, beta, S0, w, cs, z = _decode_case(N, T, H, H, d, torch.bfloat16, False, True, seed=120 + T)
    idx = torch.randperm(slots, generator=torch.Generator().manual_seed(7))[:N].to(torch.int32)
    pool = torch.zeros(slots, H, d, d)
    pool[idx.long()] = S0
    C = synthetic.conv_dim(H, H, d)
    hist = torch.randn(slots, C, 3, generator=torch.Generator().manual_seed(8))
    res = []
    for in_place in (False, True):
        P = pool.to(DEV)
        cin = hist.to(DEV)
        cout = cin if in_place else torch.zeros_like(cin)
        y = gdn.gdn_recurrent_multi_step(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), beta.to(DEV), P,
                                         state_indices=idx.to(DEV), conv_weight=w.to(DEV), conv_state=cin,
                                         conv_state_out=cout, gate_z=z.to(DEV), out_dtype=torch.float32)
        assert gdn.gdn_get_device_error() == 0
        res.append((y.cpu(), P.cpu(), cout.cpu()[idx.long()]))
    for a_, b_ in zip(res[0], res[1]):
        assert torch.equal(a_, b_)
