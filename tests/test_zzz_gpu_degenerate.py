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
    else:
        assert mode == "none", mode
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


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("T", [4, 7])
def test_multi_token_decode_degenerate_values(mode, T):
    """Pooled multi-token decode; T = 4 and T = 7 take the streamed form (blocks of four tokens, the
    last one padded with one token at T = 7)."""
    N, H, d, slots = 6, 4, 128, 9
    gen = torch.Generator().manual_seed(97 + T)
    q, k, v = (torch.randn(N, T, H, d, generator=gen).to(torch.bfloat16) for _ in range(3))
    a, b = torch.randn(N, T, H, generator=gen) - 1, torch.randn(N, T, H, generator=gen)
    A_log = torch.rand(H, generator=gen) * np.log(8)
    g64, b64 = oracle.gates_from_logits(a.reshape(-1, H), A_log, b=b.reshape(-1, H))
    g = torch.from_numpy(g64).float().reshape(N, T, H)
    beta = torch.from_numpy(b64).float().reshape(N, T, H)
    pool = torch.randn(slots, H, d, d, generator=gen) * 0.3
    idx = torch.tensor([3, 0, 8, 5, 1, 6], dtype=torch.int32)
    if mode == "zero_qk":            # whole tokens: t = 1 has a zero query, t = 2 a zero key
        q[:, 1] = 0
        k[:, 2] = 0
    inp = {"q": q, "k": k}
    _, g, beta = _degenerate(inp, g, beta, mode if mode != "zero_qk" else "none")
    pool_gpu = pool.cuda()
    out = gdn.gdn_recurrent_multi_step(q.cuda(), k.cuda(), v.cuda(), g.cuda(), beta.cuda(), pool_gpu,
                                       state_indices=idx.cuda(), out_dtype=torch.float32)
    assert gdn.gdn_get_device_error() == 0
    out, pool_new = out.cpu(), pool_gpu.cpu()
    assert torch.isfinite(out).all() and torch.isfinite(pool_new).all()
    flat = lambda x: x.reshape(N * T, H, *x.shape[3:])  # noqa: E731
    cu = np.arange(0, N * T + 1, T, dtype=np.int32)
    y_ref, S_ref = oracle.recurrence(flat(q), flat(k), flat(v), flat(g), flat(beta), cu_seqlens=cu,
                                     initial_state=pool[idx.long()])
    y = out.reshape(N * T, H, d).double().numpy()
    slab = lambda x: x.reshape(N, T, H, d).transpose(0, 2, 1, 3).reshape(N * H, -1)  # noqa: E731
    err = np.linalg.norm(slab(y - y_ref), axis=1) / np.linalg.norm(slab(y_ref), axis=1)
    assert float(np.max(err)) <= TOL_BF16
    assert rel_l2_states(pool_new[idx.long()], S_ref) <= TOL_BF16
    if mode == "zero_qk":
        assert torch.count_nonzero(out[:, 1]) == 0
