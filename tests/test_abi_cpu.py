"""CPU-only checks of the C ABI: the library builds, loads without a GPU, exports every symbol the
header declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

import gated_deltanet_recurrence_gb300 as gdn
from gated_deltanet_recurrence_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")

# a non-null, 16-byte aligned stand-in pointer; every call below must fail validation before
# it could be dereferenced or passed to CUDA
P = ctypes.c_void_p(0x10000)
NUL = None


def declared():
    src = open(HEADER).read()
    return re.findall(r"^\s*(?:int|size_t|const char\*)\s+(gdn_\w+)\s*\(", src, re.M)


def test_header_declares_the_abi():
    names = set(declared())
    assert {"gdn_chunk_fwd", "gdn_chunk_fwd_workspace_size", "gdn_recurrent_step",
            "gdn_gate_rmsnorm_silu", "gdn_decay_from_logits", "gdn_get_device_error",
            "gdn_status_string"} <= names


def test_library_exports_every_declared_symbol():
    L = gdn.lib()
    for name in declared():
        assert hasattr(L, name), name
        assert name in _binding.SIGNATURES, f"{name} has no binding"


def test_status_strings():
    L = gdn.lib()
    for code, name in _binding.STATUS.items():
        assert L.gdn_status_string(code).decode().startswith(name)


def _chunk(**kw):
    args = dict(q=P, k=P, v=P, g=P, beta=P, cu=NUL, num_seqs=1, total_T=64, H=2, Hk=2, dk=128, dv=128,
                dt=0, decay=0, scale=0.0, l2=1, cw=NUL, cin=NUL, cout=NUL, S0=NUL, Sf=NUL, z=NUL,
                w=NUL, eps=1e-6, out=P, odt=0, ws=NUL, wsb=0, stream=NUL)
    args.update(kw)
    return gdn.lib().gdn_chunk_fwd(*args.values())


def test_chunk_fwd_rejects_bad_arguments():
    assert _chunk(dt=7) == -2
    assert _chunk(odt=-1) == -2
    assert _chunk(num_seqs=0) == -1
    assert _chunk(H=0) == -1
    assert _chunk(total_T=-5) == -1
    assert _chunk(dk=96, dv=96) == -7
    assert _chunk(dk=128, dv=64) == -7
    assert _chunk(total_T=65, num_seqs=2) == -1          # equal lengths need a multiple
    assert _chunk(q=NUL) == -1
    assert _chunk(out=NUL) == -1
    assert _chunk(k=ctypes.c_void_p(0x10004)) == -1      # misaligned
    assert _chunk(w=P) == -1                              # weight without a gate
    assert _chunk(eps=-1.0) == -1
    assert _chunk(num_seqs=1 << 20, H=1 << 12, Hk=1 << 12, total_T=0) == -1  # grid too large
    assert _chunk(Hk=0) == -1
    assert _chunk(H=6, Hk=4) == -1                        # H must be a multiple of H_k
    assert _chunk(H=2, Hk=4) == -1
    assert _chunk(decay=2) == -1
    assert _chunk(cin=P) == -1                            # convolution state without weights
    assert _chunk(cout=P) == -1
    assert _chunk(cw=ctypes.c_void_p(0x10004)) == -1     # misaligned weights


def test_workspace_size_is_consistent():
    L = gdn.lib()
    for (n, T, H) in [(1, 256, 2), (2, 8192, 16), (64, 262144, 16)]:
        ws = L.gdn_chunk_fwd_workspace_size(n, T, H, 128, 128, 1)
        assert ws > 0                               # bf16, d = 128: tensor-core path
        assert _chunk(num_seqs=n, total_T=T, H=H, dt=1, odt=1, ws=NUL, wsb=0) == -4
        assert _chunk(num_seqs=n, total_T=T, H=H, dt=1, odt=1, ws=P, wsb=ws - 1) == -4
        # fp32 inputs run the CUDA-core path, which needs none; bf16 with d = 64 runs the
        # tensor-core path on 128-wide tiles and needs the same workspace as d = 128
        assert L.gdn_chunk_fwd_workspace_size(n, T, H, 128, 128, 0) == 0
        assert L.gdn_chunk_fwd_workspace_size(n, T, H, 64, 64, 1) == ws
        assert L.gdn_chunk_fwd_workspace_size(n, T, H, 64, 64, 0) == 0


def test_recurrent_step_rejects_bad_arguments():
    L = gdn.lib()

    def step(**kw):
        a = dict(q=P, k=P, v=P, g=P, beta=P, S=P, N=4, H=2, Hk=2, dk=128, dv=128, dt=1, decay=0,
                 scale=0.0, l2=1, cw=NUL, cin=NUL, cout=NUL, z=NUL, w=NUL, eps=1e-6, out=P, odt=1,
                 stream=NUL)
        a.update(kw)
        return L.gdn_recurrent_step(*a.values())

    assert step(dt=3) == -2
    assert step(N=-1) == -1
    assert step(N=0) == 0                   # nothing to do, nothing launched
    assert step(H=0) == -1
    assert step(dk=32, dv=32) == -7
    assert step(S=NUL) == -1
    assert step(S=ctypes.c_void_p(0x10008)) == -1
    assert step(w=P) == -1
    assert step(H=4, Hk=3) == -1
    assert step(decay=5) == -1
    assert step(cin=P, cout=NUL) == -1                    # state without weights
    # an in-place convolution-state update races when query/key heads are shared
    assert step(H=4, Hk=2, cw=P, cin=P, cout=P) == -1


def test_gate_and_decay_reject_bad_arguments():
    L = gdn.lib()
    assert L.gdn_gate_rmsnorm_silu(P, 0, P, NUL, 1e-6, P, 0, 10, 100, NUL) == -1   # d_v % 32
    assert L.gdn_gate_rmsnorm_silu(P, 0, P, NUL, 1e-6, P, 0, 10, 2048, NUL) == -1
    assert L.gdn_gate_rmsnorm_silu(P, 5, P, NUL, 1e-6, P, 0, 10, 128, NUL) == -2
    assert L.gdn_gate_rmsnorm_silu(NUL, 0, P, NUL, 1e-6, P, 0, 10, 128, NUL) == -1
    assert L.gdn_gate_rmsnorm_silu(P, 0, P, NUL, 1e-6, P, 0, 0, 128, NUL) == 0
    assert L.gdn_decay_from_logits(NUL, P, NUL, NUL, P, NUL, 10, 4, NUL) == -1
    assert L.gdn_decay_from_logits(P, P, NUL, P, P, NUL, 10, 4, NUL) == -1         # beta_out
    assert L.gdn_decay_from_logits(P, P, NUL, NUL, P, NUL, 10, 0, NUL) == -1
    assert L.gdn_decay_from_logits(P, P, NUL, NUL, P, NUL, 0, 4, NUL) == 0


def test_get_device_error_needs_an_output():
    assert gdn.lib().gdn_get_device_error(NUL, None) == -1


def test_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    x = torch.zeros(4, 2, 128)
    g = torch.zeros(4, 2)
    with pytest.raises(ValueError):
        gdn.gdn_chunk_fwd(x, x, x, g, g)


def test_recurrent_multi_step_rejects_bad_arguments():
    L = gdn.lib()

    def ms(**kw):
        a = dict(q=P, k=P, v=P, g=P, beta=P, S=P, slots=8, idx=NUL, N=4, T=2, H=2, Hk=2, dk=128, dv=128,
                 dt=1, decay=0, scale=0.0, l2=1, cw=NUL, cin=NUL, cout=NUL, z=NUL, w=NUL, eps=1e-6,
                 out=P, odt=1, stream=NUL)
        a.update(kw)
        return L.gdn_recurrent_multi_step(*a.values())

    assert ms(dt=9) == -2
    assert ms(T=0) == -1
    assert ms(slots=0) == -1
    assert ms(slots=3) == -1          # identity mapping needs a slot per sequence
    assert ms(N=0) == 0
    assert ms(dk=64, dv=128) == -7
    assert ms(S=NUL) == -1
    assert ms(w=P) == -1
    assert ms(H=2, Hk=4) == -1
    assert ms(H=8, Hk=2, cw=P, cin=P, cout=P) == -1


def test_chunk_fwd_noalloc_checks_arguments_before_cuda():
    """The no-allocation entry point reports argument errors exactly as gdn_chunk_fwd does, on the
    host, without first touching the CUDA runtime for its scratch array (no GPU here: a call that
    reached the runtime would answer GDN_ERR_CUDA instead)."""
    L = gdn.lib()

    def na(**kw):
        a = dict(q=P, k=P, v=P, g=P, beta=P, cu=NUL, num_seqs=1, total_T=64, H=2, Hk=2, dk=128,
                 dv=128, dt=1, decay=0, scale=0.0, l2=1, cw=NUL, cin=NUL, cout=NUL, S0=NUL, Sf=NUL,
                 z=NUL, w=NUL, eps=1e-6, out=P, odt=1, stream=NUL)
        a.update(kw)
        return L.gdn_chunk_fwd_noalloc(*a.values())

    assert na(q=NUL) == -1
    assert na(out=NUL) == -1
    assert na(dt=7) == -2
    assert na(odt=4) == -2
    assert na(dk=96, dv=96) == -7
    assert na(H=6, Hk=4) == -1
    assert na(w=P) == -1
    assert na(k=ctypes.c_void_p(0x10004)) == -1
    assert na(cin=P) == -1
    assert na(num_seqs=1, total_T=64 * 2048, H=16, Hk=16) == -4   # beyond the fixed array
    assert na(num_seqs=0) == -1


def test_selftest_bounded_wait_checks_arguments():
    L = gdn.lib()
    assert L.gdn_selftest_bounded_wait(1_000_000, NUL, NUL) == -1
    assert L.gdn_selftest_bounded_wait(1_000_000, ctypes.c_void_p(0x10002), NUL) == -1   # misaligned
    assert L.gdn_selftest_bounded_wait(999, P, NUL) == -1                                 # below 1 us
    assert L.gdn_selftest_bounded_wait(1_000_000_001, P, NUL) == -1                       # above 1 s
