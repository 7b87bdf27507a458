"""GPU parity of gdn_recurrent_multi_step (pooled, indexed, multi-token decode) against the oracle:
N sequences pick state slots from a pool through an index array (some entries negative = padding),
run T tokens each, and the pool is updated in place.  Slots nobody selects must be untouched."""
import numpy as np
import pytest
import torch

import gated_deltanet_recurrence_gb300 as gdn
import oracle
from tests._util import TOL_BF16, TOL_F32, rel_l2_states

pytestmark = pytest.mark.gpu


def _case(N, T, H, d, dtype, slots, gate, seed):
    gen = torch.Generator().manual_seed(seed)
    q, k, v = (torch.randn(N, T, H, d, generator=gen).to(dtype) for _ in range(3))
    a = torch.randn(N, T, H, generator=gen) - 1
    b = torch.randn(N, T, H, generator=gen)
    A_log = torch.rand(H, generator=gen) * np.log(8)
    g64, b64 = oracle.gates_from_logits(a.reshape(-1, H), A_log, b=b.reshape(-1, H))
    g = torch.from_numpy(g64).float().reshape(N, T, H)
    beta = torch.from_numpy(b64).float().reshape(N, T, H)
    pool = torch.randn(slots, H, d, d, generator=gen) * 0.02
    perm = torch.randperm(slots, generator=gen)[:N].to(torch.int32)
    idx = perm.clone()
    idx[1::5] = -1                                     # padding entries
    z = torch.randn(N, T, H, d, generator=gen) if gate else None
    return q, k, v, g, beta, pool, idx, z


@pytest.mark.parametrize("d,dtype,T,gate", [(128, torch.bfloat16, 4, False), (128, torch.bfloat16, 1, True),
                                            (64, torch.float32, 3, True), (128, torch.float32, 7, False)])
def test_multi_step_matches_oracle(d, dtype, T, gate):
    N, H, slots = 37, 3, 100
    q, k, v, g, beta, pool, idx, z = _case(N, T, H, d, dtype, slots, gate, seed=d + T)
    dev = "cuda"
    pool_gpu = pool.to(dev)
    out = gdn.gdn_recurrent_multi_step(q.to(dev), k.to(dev), v.to(dev), g.to(dev), beta.to(dev), pool_gpu,
                                       state_indices=idx.to(dev), gate_z=z.to(dev) if gate else None,
                                       out_dtype=torch.float32)
    assert gdn.gdn_get_device_error() == 0
    out, pool_new = out.cpu(), pool_gpu.cpu()
    live = [n for n in range(N) if idx[n] >= 0]
    sel = torch.tensor(live)
    flat = lambda x: x[sel].reshape(len(live) * T, H, *x.shape[3:])  # noqa: E731
    cu = np.arange(0, len(live) * T + 1, T, dtype=np.int32)
    y_ref, S_ref = oracle.recurrence(flat(q), flat(k), flat(v), flat(g), flat(beta), cu_seqlens=cu,
                                     initial_state=pool[idx[sel].long()])
    if gate:
        y_ref = oracle.gate_rmsnorm_silu(y_ref, flat(z))
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    y = out[sel].reshape(len(live) * T, H, d).double().numpy()
    rel = np.linalg.norm((y - y_ref).reshape(len(live), T, H, d).transpose(0, 2, 1, 3).reshape(len(live) * H, -1), axis=1)
    den = np.linalg.norm(y_ref.reshape(len(live), T, H, d).transpose(0, 2, 1, 3).reshape(len(live) * H, -1), axis=1)
    assert float(np.max(rel / den)) <= tol
    assert rel_l2_states(pool_new[idx[sel].long()], S_ref) <= tol
    untouched = sorted(set(range(slots)) - set(int(i) for i in idx[sel]))
    assert torch.equal(pool_new[untouched], pool[untouched])


def test_multi_step_equals_single_steps():
    """T tokens in one call equal T calls of gdn_recurrent_step with the identity mapping."""
    N, T, H, d = 16, 5, 4, 128
    q, k, v, g, beta, pool, _, _ = _case(N, T, H, d, torch.bfloat16, N, False, seed=77)
    dev = "cuda"
    p1 = pool.to(dev)
    y1 = gdn.gdn_recurrent_multi_step(q.to(dev), k.to(dev), v.to(dev), g.to(dev), beta.to(dev), p1,
                                      out_dtype=torch.float32)
    p2 = pool.to(dev)
    ys = [gdn.gdn_recurrent_step(q[:, t].contiguous().to(dev), k[:, t].contiguous().to(dev),
                                 v[:, t].contiguous().to(dev), g[:, t].contiguous().to(dev),
                                 beta[:, t].contiguous().to(dev), p2, out_dtype=torch.float32) for t in range(T)]
    torch.testing.assert_close(y1, torch.stack(ys, 1), rtol=1e-5, atol=1e-6)
    torch.testing.assert_close(p1, p2, rtol=1e-5, atol=1e-7)


def test_multi_step_bad_index_is_reported():
    N, T, H, d = 4, 2, 2, 64
    q, k, v, g, beta, pool, _, _ = _case(N, T, H, d, torch.float32, 6, False, seed=5)
    dev = "cuda"
    idx = torch.tensor([0, 9, 2, -1], dtype=torch.int32, device=dev)   # 9 is out of the pool
    p = pool.to(dev)
    gdn.gdn_recurrent_multi_step(q.to(dev), k.to(dev), v.to(dev), g.to(dev), beta.to(dev), p, state_indices=idx)
    assert gdn.gdn_get_device_error() == -1
    assert torch.equal(p[[1, 3, 4, 5]].cpu(), pool[[1, 3, 4, 5]])


@pytest.mark.parametrize("T,conv", [(1, False), (2, False), (3, False), (4, False), (6, False), (9, False),
                                    (1, True), (5, True)])
def test_block_and_token_forms_agree(T, conv, kernel_forms):
    """The streamed form (the chunked update over blocks of four tokens, padded at the end, or the
    single-token step at T = 1, with the states staged through shared memory) and the token-by-token
    form compute the same recurrence: outputs, states and convolution histories agree to fp32
    rounding, gate included, with skipped sequences."""
    N, H, d, slots = 21, 4, 128, 30
    q, k, v, g, beta, pool, idx, z = _case(N, T, H, d, torch.bfloat16, slots, True, seed=300 + T)
    dev = "cuda"
    cw = cs = None
    if conv:
        gen = torch.Generator().manual_seed(400 + T)
        C = 3 * H * d
        cw = (torch.rand(C, 4, generator=gen) - 0.5).to(dev)
        cs = torch.randn(slots, C, 3, generator=gen).to(dev)
    res = {}
    for mode in ("1", "0"):
        gdn.gdn_set_kernel_forms(decode_blocks=gdn.GDN_FORM_ON if mode == "1" else gdn.GDN_FORM_OFF)
        p = pool.to(dev)
        cout = torch.zeros_like(cs) if conv else None
        y = gdn.gdn_recurrent_multi_step(q.to(dev), k.to(dev), v.to(dev), g.to(dev), beta.to(dev), p,
                                         state_indices=idx.to(dev), conv_weight=cw, conv_state=cs,
                                         conv_state_out=cout, gate_z=z.to(dev), out_dtype=torch.float32)
        assert gdn.gdn_get_device_error() == 0
        res[mode] = (y.cpu(), p.cpu(), cout.cpu() if conv else None)
    live = idx >= 0
    torch.testing.assert_close(res["1"][0][live], res["0"][0][live], rtol=1e-5, atol=1e-5)
    torch.testing.assert_close(res["1"][1], res["0"][1], rtol=1e-5, atol=1e-7)
    if conv:   # the histories are raw inputs: identical
        assert torch.equal(res["1"][2], res["0"][2])
