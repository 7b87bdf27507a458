"""ctypes binding of libgdn.so: same names as the C ABI (include/gdn.h), torch tensors in.

Argument marshalling only: shapes are read from the tensors, every tensor is checked to sit on
the call's device and to hold at least what the call touches (the library sees bare pointers),
outputs that the caller does not pass are allocated with torch, and the call goes to the library
with the tensors' device current, on that device's current torch stream (or the stream given).  Every computation happens in the library's CUDA kernels; there is no
fallback: if libgdn.so is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libgdn.so")

GDN_F32, GDN_BF16 = 0, 1
GDN_DECAY_PER_HEAD, GDN_DECAY_PER_KEY_CHANNEL = 0, 1
GDN_CONV_KERNEL = 4
GDN_FORM_AUTO, GDN_FORM_OFF, GDN_FORM_ON = 0, 1, 2
STATUS = {0: "GDN_OK", -1: "GDN_ERR_ARG", -2: "GDN_ERR_DTYPE", -3: "GDN_ERR_CU_SEQLENS",
          -4: "GDN_ERR_WORKSPACE", -5: "GDN_ERR_LAUNCH", -6: "GDN_ERR_TIMEOUT",
          -7: "GDN_ERR_UNSUPPORTED", -8: "GDN_ERR_CUDA"}

_lib = None
_lock = threading.Lock()

_vp, _fp, _ip = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
_i, _f, _sz, _l = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_long

SIGNATURES = {
    "gdn_chunk_fwd": (_i, [_vp, _vp, _vp, _fp, _fp, _ip, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i,
                           _fp, _fp, _fp, _fp, _fp, _fp, _fp, _f, _vp, _i, _vp, _sz, _vp]),
    "gdn_chunk_fwd_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "gdn_recurrent_step": (_i, [_vp, _vp, _vp, _fp, _fp, _fp, _i, _i, _i, _i, _i, _i, _i, _f, _i,
                                _fp, _fp, _fp, _fp, _fp, _f, _vp, _i, _vp]),
    "gdn_recurrent_multi_step": (_i, [_vp, _vp, _vp, _fp, _fp, _fp, _i, _ip, _i, _i, _i, _i, _i, _i, _i,
                                      _i, _f, _i, _fp, _fp, _fp, _fp, _fp, _f, _vp, _i, _vp]),
    "gdn_gate_rmsnorm_silu": (_i, [_vp, _i, _fp, _fp, _f, _vp, _i, _l, _i, _vp]),
    "gdn_decay_from_logits": (_i, [_fp, _fp, _fp, _fp, _fp, _fp, _l, _i, _vp]),
    "gdn_chunk_fwd_noalloc": (_i, [_vp, _vp, _vp, _fp, _fp, _ip, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i,
                                   _fp, _fp, _fp, _fp, _fp, _fp, _fp, _f, _vp, _i, _vp]),
    "gdn_get_device_error": (_i, [_vp, ctypes.POINTER(ctypes.c_int)]),
    "gdn_status_string": (ctypes.c_char_p, [_i]),
    "gdn_selftest_bounded_wait": (_i, [ctypes.c_ulonglong, _vp, _vp]),
    "gdn_set_kernel_forms": (_i, [_i, _i]),
}


class GdnError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} returned {status} ({STATUS.get(status, 'unknown')})")


def lib():
    """Load libgdn.so (building it first if it is missing or older than its sources)."""
    global _lib
    with _lock:
        if _lib is None:
            from . import build as _build
            if _build.is_stale():
                _build.build()
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libgdn.so not found at {LIB_PATH}")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    if t.dtype == torch.float32:
        return GDN_F32
    raise TypeError(f"unsupported dtype {t.dtype}; use float32 or bfloat16")


def _torch_dt(code: int):
    return torch.bfloat16 if code == GDN_BF16 else torch.float32


def _p(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("all tensors must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("all tensors must be contiguous")
    return t.data_ptr()


def _f32(t, name):
    if t is not None and t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32")
    return t


def _sizes(ref, **tensors):
    """The library sees only pointers, so the binding refuses, before the call, a tensor on another
    device than `ref` or holding fewer elements than the call reads or writes through it.
    Each keyword is name=(tensor or None, elements the call touches)."""
    for name, (t, numel) in tensors.items():
        if t is None:
            continue
        if t.device != ref.device:
            raise ValueError(f"{name} is on {t.device}, the call runs on {ref.device}")
        if t.numel() < numel:
            raise ValueError(f"{name} holds {t.numel()} elements; the call touches {numel}")


def _stream(stream, ref=None):
    if stream is None:
        return torch.cuda.current_stream(ref.device if ref is not None else None).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _run(ref, fn, *args):
    """Call library function `fn` with the device of `ref` current: the library launches its
    kernels on the calling thread's current device."""
    dev = ref.get_device()
    if dev == torch.cuda.current_device():
        return fn(*args)
    with torch.cuda.device(dev):
        return fn(*args)


def _check(fn, rc):
    if rc != 0:
        raise GdnError(fn, rc)


def _decay_mode(g, per_head_dims):
    """GDN_DECAY_PER_HEAD when g has the per-head shape, else one decay per key channel."""
    return GDN_DECAY_PER_HEAD if g.dim() == per_head_dims else GDN_DECAY_PER_KEY_CHANNEL


def _conv_f32(conv_weight, conv_state, conv_state_out):
    for name, t in (("conv_weight", conv_weight), ("conv_state", conv_state),
                    ("conv_state_out", conv_state_out)):
        _f32(t, name)


def gdn_chunk_fwd(q, k, v, g, beta, cu_seqlens=None, num_seqs=None, scale=0.0, use_qk_l2norm=True,
                  initial_state=None, final_state=None, output_final_state=True, conv_weight=None,
                  conv_state=None, conv_state_out=None, gate_z=None, norm_weight=None, norm_eps=1e-6,
                  out=None, out_dtype=None, workspace=None, stream=None):
    """Chunked prefill.  q, k [total_T, H_k, d_k]; v [total_T, H, d_v] (H a multiple of H_k);
    beta [total_T, H] fp32; g [total_T, H] fp32, or [total_T, H, d_k] for a decay per key channel;
    cu_seqlens int32 [num_seqs+1] (device) or None with num_seqs equal sequences (default 1).
    conv_weight [2 H_k d_k + H d_v, 4] fuses the short convolution (conv_state: carried input
    history [num_seqs, conv_dim, 3] or None; conv_state_out: filled with the final history if
    given, may be conv_state itself).
    Returns (out, final_state); final_state is allocated unless given or not requested."""
    total_T, H_k, d_k = q.shape
    H, d_v = v.shape[1], v.shape[-1]
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32:
            raise TypeError("cu_seqlens must be int32")
        num_seqs = cu_seqlens.numel() - 1
    elif num_seqs is None:
        num_seqs = 1
    dt = _dt(q)
    if _dt(k) != dt or _dt(v) != dt:
        raise TypeError("q, k, v must share one dtype")
    odt = dt if out_dtype is None else _dt(torch.empty(0, dtype=out_dtype))
    if out is None:
        out = torch.empty((total_T, H, d_v), dtype=_torch_dt(odt), device=q.device)
    else:
        odt = _dt(out)
    if final_state is None and output_final_state:
        final_state = torch.empty((num_seqs, H, d_v, d_k), dtype=torch.float32, device=q.device)
    for name, t in (("g", g), ("beta", beta), ("initial_state", initial_state),
                    ("final_state", final_state), ("gate_z", gate_z), ("norm_weight", norm_weight)):
        _f32(t, name)
    _conv_f32(conv_weight, conv_state, conv_state_out)
    conv_dim = 2 * H_k * d_k + H * d_v
    _sizes(q, k=(k, total_T * H_k * d_k), v=(v, total_T * H * d_v),
           g=(g, total_T * H * (1 if g.dim() == 2 else d_k)), beta=(beta, total_T * H),
           cu_seqlens=(cu_seqlens, num_seqs + 1), initial_state=(initial_state, num_seqs * H * d_v * d_k),
           final_state=(final_state, num_seqs * H * d_v * d_k), gate_z=(gate_z, total_T * H * d_v),
           norm_weight=(norm_weight, d_v), out=(out, total_T * H * d_v),
           conv_weight=(conv_weight, conv_dim * GDN_CONV_KERNEL),
           conv_state=(conv_state, num_seqs * conv_dim * (GDN_CONV_KERNEL - 1)),
           conv_state_out=(conv_state_out, num_seqs * conv_dim * (GDN_CONV_KERNEL - 1)),
           workspace=(workspace, 0))
    L = lib()
    ws_need = L.gdn_chunk_fwd_workspace_size(num_seqs, total_T, H, d_k, d_v, dt)
    if ws_need and workspace is None:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    rc = _run(q, L.gdn_chunk_fwd,
              _p(q), _p(k), _p(v), _p(g), _p(beta), _p(cu_seqlens), num_seqs, total_T, H, H_k, d_k,
              d_v, dt, _decay_mode(g, 2), float(scale), int(bool(use_qk_l2norm)), _p(conv_weight),
              _p(conv_state), _p(conv_state_out), _p(initial_state), _p(final_state), _p(gate_z),
              _p(norm_weight), float(norm_eps), _p(out), odt, _p(workspace),
              workspace.numel() * workspace.element_size() if workspace is not None else 0,
              _stream(stream, q))
    _check("gdn_chunk_fwd", rc)
    return out, final_state


def gdn_chunk_fwd_noalloc(q, k, v, g, beta, cu_seqlens=None, num_seqs=None, scale=0.0,
                          use_qk_l2norm=True, initial_state=None, final_state=None, conv_weight=None,
                          conv_state=None, conv_state_out=None, gate_z=None, norm_weight=None,
                          norm_eps=1e-6, out=None, stream=None):
    """gdn_chunk_fwd with the library's fixed scratch array instead of a workspace; `out` and
    `final_state` must be passed in (this call allocates nothing, here or in the library)."""
    total_T, H_k, d_k = q.shape
    H, d_v = v.shape[1], v.shape[-1]
    if out is None:
        raise ValueError("gdn_chunk_fwd_noalloc needs a preallocated `out`")
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32:
            raise TypeError("cu_seqlens must be int32")
        num_seqs = cu_seqlens.numel() - 1
    elif num_seqs is None:
        num_seqs = 1
    dt = _dt(q)
    for name, t in (("g", g), ("beta", beta), ("initial_state", initial_state),
                    ("final_state", final_state), ("gate_z", gate_z), ("norm_weight", norm_weight)):
        _f32(t, name)
    _conv_f32(conv_weight, conv_state, conv_state_out)
    conv_dim = 2 * H_k * d_k + H * d_v
    _sizes(q, k=(k, total_T * H_k * d_k), v=(v, total_T * H * d_v),
           g=(g, total_T * H * (1 if g.dim() == 2 else d_k)), beta=(beta, total_T * H),
           cu_seqlens=(cu_seqlens, num_seqs + 1), initial_state=(initial_state, num_seqs * H * d_v * d_k),
           final_state=(final_state, num_seqs * H * d_v * d_k), gate_z=(gate_z, total_T * H * d_v),
           norm_weight=(norm_weight, d_v), out=(out, total_T * H * d_v),
           conv_weight=(conv_weight, conv_dim * GDN_CONV_KERNEL),
           conv_state=(conv_state, num_seqs * conv_dim * (GDN_CONV_KERNEL - 1)),
           conv_state_out=(conv_state_out, num_seqs * conv_dim * (GDN_CONV_KERNEL - 1)))
    rc = _run(q, lib().gdn_chunk_fwd_noalloc,
              _p(q), _p(k), _p(v), _p(g), _p(beta), _p(cu_seqlens), num_seqs, total_T, H, H_k, d_k,
              d_v, dt, _decay_mode(g, 2), float(scale), int(bool(use_qk_l2norm)), _p(conv_weight),
              _p(conv_state), _p(conv_state_out), _p(initial_state), _p(final_state), _p(gate_z),
              _p(norm_weight), float(norm_eps), _p(out), _dt(out), _stream(stream, q))
    _check("gdn_chunk_fwd_noalloc", rc)
    return out, final_state


def gdn_recurrent_step(q, k, v, g, beta, state, scale=0.0, use_qk_l2norm=True, conv_weight=None,
                       conv_state=None, conv_state_out=None, gate_z=None, norm_weight=None,
                       norm_eps=1e-6, out=None, out_dtype=None, stream=None):
    """One decode token: q, k [N, H_k, d_k]; v [N, H, d_v]; beta [N, H]; g [N, H] or [N, H, d_k];
    state [N, H, d_v, d_k] fp32 updated in place.  conv_weight [conv_dim, 4] fuses the short
    convolution with history conv_state [N, conv_dim, 3] (None: zeros) and the new history written
    to conv_state_out (may be conv_state when H_k == H).  Returns out [N, H, d_v]."""
    N, H_k, d_k = q.shape
    H, d_v = v.shape[1], v.shape[-1]
    dt = _dt(q)
    odt = dt if out_dtype is None else _dt(torch.empty(0, dtype=out_dtype))
    if out is None:
        out = torch.empty((N, H, d_v), dtype=_torch_dt(odt), device=q.device)
    else:
        odt = _dt(out)
    for name, t in (("g", g), ("beta", beta), ("state", state), ("gate_z", gate_z),
                    ("norm_weight", norm_weight)):
        _f32(t, name)
    _conv_f32(conv_weight, conv_state, conv_state_out)
    conv_dim = 2 * H_k * d_k + H * d_v
    _sizes(q, k=(k, N * H_k * d_k), v=(v, N * H * d_v), g=(g, N * H * (1 if g.dim() == 2 else d_k)),
           beta=(beta, N * H), state=(state, N * H * d_v * d_k), gate_z=(gate_z, N * H * d_v),
           norm_weight=(norm_weight, d_v), out=(out, N * H * d_v),
           conv_weight=(conv_weight, conv_dim * GDN_CONV_KERNEL),
           conv_state=(conv_state, N * conv_dim * (GDN_CONV_KERNEL - 1)),
           conv_state_out=(conv_state_out, N * conv_dim * (GDN_CONV_KERNEL - 1)))
    rc = _run(q, lib().gdn_recurrent_step,
              _p(q), _p(k), _p(v), _p(g), _p(beta), _p(state), N, H, H_k, d_k, d_v, dt,
              _decay_mode(g, 2), float(scale), int(bool(use_qk_l2norm)), _p(conv_weight),
              _p(conv_state), _p(conv_state_out), _p(gate_z), _p(norm_weight), float(norm_eps),
              _p(out), odt, _stream(stream, q))
    _check("gdn_recurrent_step", rc)
    return out


def gdn_recurrent_multi_step(q, k, v, g, beta, state_pool, state_indices=None, scale=0.0,
                             use_qk_l2norm=True, conv_weight=None, conv_state=None,
                             conv_state_out=None, gate_z=None, norm_weight=None, norm_eps=1e-6,
                             out=None, out_dtype=None, stream=None):
    """T decode tokens per sequence on pooled states: q, k [N, T, H_k, d_k]; v [N, T, H, d_v];
    beta [N, T, H]; g [N, T, H] or [N, T, H, d_k]; state_pool [slots, H, d_v, d_k] fp32 updated in
    place; state_indices int32 [N] (negative = skip) or None; conv_state / conv_state_out
    [slots, conv_dim, 3] indexed like the pool.  Returns out [N, T, H, d_v]."""
    N, T, H_k, d_k = q.shape
    H, d_v = v.shape[2], v.shape[-1]
    dt = _dt(q)
    odt = dt if out_dtype is None else _dt(torch.empty(0, dtype=out_dtype))
    if out is None:
        out = torch.empty((N, T, H, d_v), dtype=_torch_dt(odt), device=q.device)
    else:
        odt = _dt(out)
    if state_indices is not None and state_indices.dtype != torch.int32:
        raise TypeError("state_indices must be int32")
    for name, t in (("g", g), ("beta", beta), ("state_pool", state_pool), ("gate_z", gate_z),
                    ("norm_weight", norm_weight)):
        _f32(t, name)
    _conv_f32(conv_weight, conv_state, conv_state_out)
    conv_dim, slots = 2 * H_k * d_k + H * d_v, state_pool.shape[0]
    _sizes(q, k=(k, N * T * H_k * d_k), v=(v, N * T * H * d_v),
           g=(g, N * T * H * (1 if g.dim() == 3 else d_k)), beta=(beta, N * T * H),
           state_pool=(state_pool, slots * H * d_v * d_k), state_indices=(state_indices, N),
           gate_z=(gate_z, N * T * H * d_v), norm_weight=(norm_weight, d_v), out=(out, N * T * H * d_v),
           conv_weight=(conv_weight, conv_dim * GDN_CONV_KERNEL),
           conv_state=(conv_state, slots * conv_dim * (GDN_CONV_KERNEL - 1)),
           conv_state_out=(conv_state_out, slots * conv_dim * (GDN_CONV_KERNEL - 1)))
    rc = _run(q, lib().gdn_recurrent_multi_step,
              _p(q), _p(k), _p(v), _p(g), _p(beta), _p(state_pool), state_pool.shape[0],
              _p(state_indices), N, T, H, H_k, d_k, d_v, dt, _decay_mode(g, 3), float(scale),
              int(bool(use_qk_l2norm)), _p(conv_weight), _p(conv_state), _p(conv_state_out),
              _p(gate_z), _p(norm_weight), float(norm_eps), _p(out), odt, _stream(stream, q))
    _check("gdn_recurrent_multi_step", rc)
    return out


def gdn_gate_rmsnorm_silu(y, z, norm_weight=None, eps=1e-6, out=None, out_dtype=None, stream=None):
    """out = w * y / rms(y) * silu(z) over the last dimension of y (fp32 or bf16)."""
    d_v = y.shape[-1]
    rows = y.numel() // d_v if d_v else 0
    odt = _dt(y) if out_dtype is None else _dt(torch.empty(0, dtype=out_dtype))
    if out is None:
        out = torch.empty(y.shape, dtype=_torch_dt(odt), device=y.device)
    else:
        odt = _dt(out)
    _f32(z, "z")
    _f32(norm_weight, "norm_weight")
    _sizes(y, z=(z, rows * d_v), norm_weight=(norm_weight, d_v), out=(out, rows * d_v))
    rc = _run(y, lib().gdn_gate_rmsnorm_silu,
              _p(y), _dt(y), _p(z), _p(norm_weight), float(eps), _p(out), odt, rows, d_v,
              _stream(stream, y))
    _check("gdn_gate_rmsnorm_silu", rc)
    return out


def gdn_decay_from_logits(a, A_log, dt_bias=None, b=None, g_out=None, beta_out=None, stream=None):
    """g = -exp(A_log) softplus(a + dt_bias) and beta = sigmoid(b); a, b [total_T, H] fp32."""
    total_T, H = a.shape
    for name, t in (("a", a), ("A_log", A_log), ("dt_bias", dt_bias), ("b", b)):
        _f32(t, name)
    if g_out is None:
        g_out = torch.empty_like(a)
    if b is not None and beta_out is None:
        beta_out = torch.empty_like(b)
    _sizes(a, A_log=(A_log, H), dt_bias=(dt_bias, H), b=(b, total_T * H), g_out=(g_out, total_T * H),
           beta_out=(beta_out, total_T * H))
    rc = _run(a, lib().gdn_decay_from_logits,
              _p(a), _p(A_log), _p(dt_bias), _p(b), _p(g_out), _p(beta_out), total_T, H,
              _stream(stream, a))
    _check("gdn_decay_from_logits", rc)
    return (g_out, beta_out) if b is not None else g_out


def gdn_selftest_bounded_wait(limit_ns, status=None, stream=None):
    """Run the library's bounded device wait on a phase that never completes (limit_ns in
    [1e3, 1e9]); returns the int32 device tensor the kernel writes its status to
    (GDN_ERR_TIMEOUT = -6 once the wait has given up)."""
    if status is None:
        status = torch.full((1,), 1, dtype=torch.int32, device="cuda")
    if status.dtype != torch.int32 or status.numel() < 1:
        raise ValueError("status must be an int32 tensor with at least one element")
    rc = _run(status, lib().gdn_selftest_bounded_wait, int(limit_ns), _p(status),
              _stream(stream, status))
    _check("gdn_selftest_bounded_wait", rc)
    return status


def gdn_get_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device-side status word."""
    st = ctypes.c_int(0)
    _check("gdn_get_device_error", lib().gdn_get_device_error(_stream(stream), ctypes.byref(st)))
    return st.value


def gdn_set_kernel_forms(prefill_fused=GDN_FORM_AUTO, decode_blocks=GDN_FORM_AUTO):
    """Process-wide choice between the library's equivalent kernel forms (GDN_FORM_AUTO / _OFF /
    _ON for the fused prefill launch and for the four-token block decode); for comparisons and
    tests.  Call it with no arguments to restore the automatic choice."""
    _check("gdn_set_kernel_forms", lib().gdn_set_kernel_forms(int(prefill_fused), int(decode_blocks)))
