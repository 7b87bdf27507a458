"""The Python binding's own checks, on the CPU (no GPU, no launch).

The C ABI receives bare pointers, so a tensor smaller than the call reads or writes, or one on
another device, can only be caught in the binding.  Every call with consistent shapes must pass
these checks and stop only at the CUDA-tensor check (CPU tensors here); each undersized or
misplaced tensor must be refused by name before the library is called."""
import pytest
import torch

import gated_deltanet_recurrence_gb300 as gdn
from gated_deltanet_recurrence_gb300 import synthetic

CUDA_ONLY = "must be CUDA tensors"


def _prefill_args(**opts):
    cfg = synthetic.workload("varlen", lengths=[70, 1, 130], num_seqs=3, H=4, d=64,
                             dtype=torch.bfloat16, seed=3, gate=True, init_state=True, **opts)
    inp = synthetic.prefill_inputs(cfg)
    T, H, d, n = inp["total_T"], 4, 64, 3
    g = torch.zeros(T, H, d) if opts.get("per_channel") else torch.zeros(T, H)
    kw = dict(cu_seqlens=inp["cu_seqlens"], initial_state=inp["initial_state"],
              final_state=torch.empty(n, H, d, d), gate_z=inp["z"], norm_weight=torch.ones(d),
              out=torch.empty(T, H, d, dtype=torch.bfloat16))
    if opts.get("conv"):
        C = synthetic.conv_dim(H, opts.get("Hk", H), d)
        kw.update(conv_weight=inp["conv_weight"], conv_state=torch.zeros(n, C, 3),
                  conv_state_out=torch.zeros(n, C, 3))
    return (inp["q"], inp["k"], inp["v"], g, torch.zeros(T, H)), kw


@pytest.mark.parametrize("opts", [{}, {"Hk": 2}, {"per_channel": True}, {"conv": True},
                                  {"conv": True, "Hk": 1}])
@pytest.mark.parametrize("fn", ["gdn_chunk_fwd", "gdn_chunk_fwd_noalloc"])
def test_consistent_prefill_call_passes_the_size_checks(fn, opts):
    pos, kw = _prefill_args(**opts)
    with pytest.raises(ValueError, match=CUDA_ONLY):
        getattr(gdn, fn)(*pos, **kw)


@pytest.mark.parametrize("name,shape", [("out", (200, 4, 64)), ("final_state", (2, 4, 64, 64)),
                                        ("initial_state", (3, 4, 64, 63)), ("gate_z", (201, 4, 32)),
                                        ("norm_weight", (32,)), ("conv_state", (3, 10, 3)),
                                        ("conv_state_out", (2, 640, 3)), ("conv_weight", (640, 3))])
def test_undersized_prefill_tensor_is_refused(name, shape):
    pos, kw = _prefill_args(conv=True)
    kw[name] = torch.zeros(shape, dtype=kw[name].dtype)
    with pytest.raises(ValueError, match=f"{name} holds"):
        gdn.gdn_chunk_fwd(*pos, **kw)


def test_undersized_prefill_inputs_are_refused():
    (q, k, v, g, b), kw = _prefill_args()
    for i, name in enumerate(("k", "v", "g", "beta")):
        args = [q, k, v, g, b]
        args[i + 1] = args[i + 1][:-1]
        with pytest.raises(ValueError, match=f"{name} holds"):
            gdn.gdn_chunk_fwd(*args, **kw)


def test_tensor_on_another_device_is_refused():
    pos, kw = _prefill_args()
    kw["gate_z"] = torch.empty(kw["gate_z"].shape, device="meta")
    with pytest.raises(ValueError, match="gate_z is on meta"):
        gdn.gdn_chunk_fwd(*pos, **kw)


def _decode_args(N=5, T=None, H=4, Hk=4, d=64, per_channel=False, conv=False, slots=None):
    lead = (N,) if T is None else (N, T)
    q, k = torch.zeros(*lead, Hk, d, dtype=torch.bfloat16), torch.zeros(*lead, Hk, d, dtype=torch.bfloat16)
    v = torch.zeros(*lead, H, d, dtype=torch.bfloat16)
    g = torch.zeros(*lead, H, d) if per_channel else torch.zeros(*lead, H)
    S = torch.zeros(slots or N, H, d, d)
    kw = dict(gate_z=torch.zeros(*lead, H, d), norm_weight=torch.ones(d),
              out=torch.empty(*lead, H, d, dtype=torch.bfloat16))
    if conv:
        C = synthetic.conv_dim(H, Hk, d)
        kw.update(conv_weight=torch.zeros(C, 4), conv_state=torch.zeros(slots or N, C, 3),
                  conv_state_out=torch.zeros(slots or N, C, 3))
    if T is not None:
        kw["state_indices"] = torch.arange(N, dtype=torch.int32)
    return (q, k, v, g, torch.zeros(*lead, H), S), kw


@pytest.mark.parametrize("opts", [{}, {"Hk": 2}, {"per_channel": True}, {"conv": True}])
def test_consistent_decode_calls_pass_the_size_checks(opts):
    pos, kw = _decode_args(**opts)
    with pytest.raises(ValueError, match=CUDA_ONLY):
        gdn.gdn_recurrent_step(*pos, **kw)
    pos, kw = _decode_args(T=3, slots=9, **opts)
    with pytest.raises(ValueError, match=CUDA_ONLY):
        gdn.gdn_recurrent_multi_step(*pos, **kw)


def test_undersized_decode_tensors_are_refused():
    pos, kw = _decode_args(conv=True)
    pos = list(pos)
    pos[5] = torch.zeros(4, 4, 64, 64)                       # a state for 4 of 5 sequences
    with pytest.raises(ValueError, match="state holds"):
        gdn.gdn_recurrent_step(*pos, **kw)
    pos, kw = _decode_args(T=3, slots=9, conv=True)
    kw["state_indices"] = torch.arange(4, dtype=torch.int32)
    with pytest.raises(ValueError, match="state_indices holds"):
        gdn.gdn_recurrent_multi_step(*pos, **kw)
    pos, kw = _decode_args(T=3, slots=9, conv=True)
    kw["conv_state"] = torch.zeros(5, kw["conv_state"].shape[1], 3)   # per sequence, not per slot
    with pytest.raises(ValueError, match="conv_state holds"):
        gdn.gdn_recurrent_multi_step(*pos, **kw)


def test_gate_and_decay_sizes():
    y, z = torch.zeros(6, 4, 64), torch.zeros(6, 4, 64)
    with pytest.raises(ValueError, match=CUDA_ONLY):
        gdn.gdn_gate_rmsnorm_silu(y, z, torch.ones(64), out=torch.empty(6, 4, 64))
    with pytest.raises(ValueError, match="z holds"):
        gdn.gdn_gate_rmsnorm_silu(y, z[:5])
    with pytest.raises(ValueError, match="out holds"):
        gdn.gdn_gate_rmsnorm_silu(y, z, out=torch.empty(6, 4, 63))
    a, b = torch.zeros(10, 4), torch.zeros(10, 4)
    with pytest.raises(ValueError, match=CUDA_ONLY):
        gdn.gdn_decay_from_logits(a, torch.zeros(4), torch.zeros(4), b)
    with pytest.raises(ValueError, match="A_log holds"):
        gdn.gdn_decay_from_logits(a, torch.zeros(3))
    with pytest.raises(ValueError, match="beta_out holds"):
        gdn.gdn_decay_from_logits(a, torch.zeros(4), b=b, beta_out=torch.empty(9, 4))


def test_missing_or_broken_library_fails_loudly(monkeypatch, tmp_path):
    """There is no fallback: without a loadable libgdn.so every call raises."""
    from gated_deltanet_recurrence_gb300 import _binding, build
    monkeypatch.setattr(build, "is_stale", lambda: False)      # do not rebuild it here
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "LIB_PATH", str(tmp_path / "absent" / "libgdn.so"))
    with pytest.raises(RuntimeError, match="not found"):
        gdn.lib()
    pos, kw = _decode_args()
    with pytest.raises(RuntimeError, match="not found"):
        gdn.gdn_recurrent_step(*pos, **kw)
    broken = tmp_path / "libgdn.so"
    broken.write_bytes(b"not a shared library")
    monkeypatch.setattr(_binding, "LIB_PATH", str(broken))
    with pytest.raises(OSError):
        gdn.lib()
