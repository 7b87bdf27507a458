"""Guard bands around every output: no kernel writes outside the tensors it was given.

compute-sanitizer is not available here, so out-of-bounds writes are looked for directly: each
output (and each in/out state) is a view into a larger buffer whose 64 elements before and after
hold a sentinel.  After the call the sentinels must be intact, bit for bit.  The cases cover the
ragged ends where a kernel is most likely to overrun: partial last chunks, one-token and empty
sequences, the fused gate, the convolution history and the pooled decode.  The guard keeps every
view 128-byte aligned (64 elements of 2 or 4 bytes).  The file name makes pytest run it last."""
import pytest
import torch

import gated_deltanet_recurrence_gb300 as gdn
from gated_deltanet_recurrence_gb300 import synthetic
from tests._util import oracle_gates

pytestmark = pytest.mark.gpu

G = 64                 # guard elements on each side
SENTINEL = 3.5         # exactly representable in bf16 and fp32


def guarded(shape, dtype, fill=None):
    """A contiguous tensor of `shape` inside a buffer with G sentinel elements on each side;
    returns (view, buffer).  `fill` (a tensor) initialises the view."""
    n = 1
    for s in shape:
        n *= s
    buf = torch.full((G + n + G,), SENTINEL, dtype=dtype, device="cuda")
    view = buf[G:G + n].view(shape)
    if fill is not None:
        view.copy_(fill)
    return view, buf


def intact(buf):
    head, tail = buf[:G], buf[-G:]
    return bool((head == SENTINEL).all()) and bool((tail == SENTINEL).all())


@pytest.mark.parametrize("d,dtype,gate,conv", [(128, torch.bfloat16, True, False),
                                               (128, torch.bfloat16, False, True),
                                               (64, torch.float32, True, True)])
def test_prefill_writes_stay_inside_outputs(d, dtype, gate, conv):
    lengths = [1, 0, 130, 64, 63]
    H = 4
    cfg = synthetic.workload("varlen", lengths=lengths, num_seqs=len(lengths), H=H, d=d,
                             dtype=dtype, seed=120 + d, gate=gate, init_state=True, conv=conv,
                             conv_state=conv)
    inp = synthetic.prefill_inputs(cfg)
    g32, b32 = oracle_gates(inp)
    T, n = inp["total_T"], len(lengths)
    dev = "cuda"
    out, out_buf = guarded((T, H, d), dtype)
    Sf, Sf_buf = guarded((n, H, d, d), torch.float32)
    kw = {}
    if conv:
        C = synthetic.conv_dim(H, H, d)
        cs_out, cs_buf = guarded((n, C, 3), torch.float32)
        kw = dict(conv_weight=inp["conv_weight"].to(dev), conv_state=inp["conv_state"].to(dev),
                  conv_state_out=cs_out)
    gdn.gdn_chunk_fwd(inp["q"].to(dev), inp["k"].to(dev), inp["v"].to(dev), g32.to(dev), b32.to(dev),
                      cu_seqlens=inp["cu_seqlens"].to(dev), initial_state=inp["initial_state"].to(dev),
                      final_state=Sf, gate_z=inp["z"].to(dev) if gate else None, out=out, **kw)
    assert gdn.gdn_get_device_error() == 0
    torch.cuda.synchronize()
    assert intact(out_buf), "output guard overwritten"
    assert intact(Sf_buf), "final-state guard overwritten"
    if conv:
        assert intact(cs_buf), "convolution-state guard overwritten"


@pytest.mark.parametrize("conv", [False, True])
def test_decode_writes_stay_inside_outputs(conv):
    cfg = synthetic.workload("decode", N=7, H=4, d=128, dtype=torch.bfloat16, seed=125, gate=True)
    inp = synthetic.decode_inputs(cfg)
    g32, b32 = oracle_gates(inp)
    dev = "cuda"
    N, H, d = 7, 4, 128
    state, st_buf = guarded((N, H, d, d), torch.float32, inp["state"].to(dev))
    out, out_buf = guarded((N, H, d), torch.bfloat16)
    kw = {}
    if conv:
        C = synthetic.conv_dim(H, H, d)
        w = torch.rand(C, 4, generator=torch.Generator().manual_seed(3)) - 0.5
        cs, cs_buf = guarded((N, C, 3), torch.float32, torch.randn(N, C, 3))
        kw = dict(conv_weight=w.to(dev), conv_state=cs, conv_state_out=cs)
    gdn.gdn_recurrent_step(inp["q"].to(dev), inp["k"].to(dev), inp["v"].to(dev), g32.to(dev),
                           b32.to(dev), state, gate_z=inp["z"].to(dev), out=out, **kw)
    assert gdn.gdn_get_device_error() == 0
    torch.cuda.synchronize()
    assert intact(st_buf) and intact(out_buf)
    if conv:
        assert intact(cs_buf)


@pytest.mark.parametrize("T", [1, 4, 7])
def test_pooled_decode_writes_stay_inside_outputs(T):
    N, H, d, slots = 5, 4, 128, 8
    gen = torch.Generator().manual_seed(130 + T)
    dev = "cuda"
    q, k, v = (torch.randn(N, T, H, d, generator=gen).to(torch.bfloat16).to(dev) for _ in range(3))
    g = (-torch.rand(N, T, H, generator=gen)).to(dev)
    b = torch.rand(N, T, H, generator=gen).to(dev)
    pool, pool_buf = guarded((slots, H, d, d), torch.float32, torch.randn(slots, H, d, d, generator=gen) * 0.1)
    idx = torch.tensor([7, -1, 0, 3, 6], dtype=torch.int32, device=dev)   # first and last slots used
    out, out_buf = guarded((N, T, H, d), torch.float32)
    gdn.gdn_recurrent_multi_step(q, k, v, g, b, pool, state_indices=idx, out=out)
    assert gdn.gdn_get_device_error() == 0
    torch.cuda.synchronize()
    assert intact(pool_buf) and intact(out_buf)
