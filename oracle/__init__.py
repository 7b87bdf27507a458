"""fp64 CPU oracle of the gated delta rule -- TEST INFRASTRUCTURE ONLY.

This package is the yardstick the CUDA library is checked against.  Only the
test-suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import it.  It shares no code with the CUDA path: the arithmetic lives in
``gdn_oracle.c`` (plain C, double precision, written out loop by loop), and
this module only compiles it with gcc, converts arrays to float64 and calls it.

Functions and the passages they follow (page titles):
  recurrence            "[LLM Algorithms-2] Gated DeltaNet" sections 4, 4.3, 5;
                        "6.6 Gated DeltaNet" 6.6.4 loop; "Gated DeltaNet详解"
  chunked               "5. 线性注意力", "Delta Rule 的 Chunk 实现" (stages 1-3)
  transition_product    "[LLM Algorithms-2] Gated DeltaNet" section 7
  chunk_decay           "5. 线性注意力", stage 1 decay matrix
  gate_rmsnorm_silu     "5. 线性注意力", "门控 RMSNorm"; "6.6 Gated DeltaNet" 6.6.2
  gates_from_logits     "6.6 Gated DeltaNet" 6.6.3
  recurrent_step        "6.6 Gated DeltaNet" 6.6.8 (one token on a kept state)
  short_conv            "5. 线性注意力", "因果卷积(Causal Conv1d)" (depthwise, causal, SiLU)

The forms take q, k with Hk heads and v with H = r * Hk heads (value head h reads
query/key head h // r, the page's repeat_interleave), and g either [total_T, H]
(one decay per head) or [total_T, H, dk] (one per key channel, "6.6 Gated
DeltaNet" 6.6.7; S <- S diag(alpha_t)); the chunked form is scalar only.

Every function has at least one independent pin in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgdn_oracle.so")
_lib = None
_lock = threading.Lock()

FORM_RECURRENCE, FORM_CHUNKED, FORM_TRANSITION = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c with gcc into oracle/_build/libgdn_oracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            lib.gdn_oracle_forward.restype = ctypes.c_int
            lib.gdn_oracle_forward.argtypes = [
                ctypes.c_int, dp, dp, dp, dp, dp, ip, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int, dp, dp, dp,
                ctypes.c_int, ctypes.c_int]
            lib.gdn_oracle_short_conv.restype = ctypes.c_int
            lib.gdn_oracle_short_conv.argtypes = [dp, dp, ip, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                  dp, dp, dp, ctypes.c_int]
            lib.gdn_oracle_chunk_decay.restype = None
            lib.gdn_oracle_chunk_decay.argtypes = [dp, ctypes.c_int, dp, dp]
            lib.gdn_oracle_gate_rmsnorm_silu.restype = None
            lib.gdn_oracle_gate_rmsnorm_silu.argtypes = [dp, dp, dp, ctypes.c_double, dp,
                                                         ctypes.c_long, ctypes.c_int]
            lib.gdn_oracle_gates_from_logits.restype = None
            lib.gdn_oracle_gates_from_logits.argtypes = [dp, dp, dp, dp, dp, dp, ctypes.c_long,
                                                         ctypes.c_int]
            _lib = lib
    return _lib


def _f64(x):
    """Exact upcast to a contiguous float64 numpy array (accepts torch tensors)."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: bf16/fp32 values are exactly representable in fp64
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _cu(cu_seqlens, total_T, batch):
    if cu_seqlens is None:
        if batch is None:
            batch = 1
        if total_T % batch:
            raise ValueError("total_T not divisible by batch")
        T = total_T // batch
        return np.arange(0, total_T + 1, T if T > 0 else 1, dtype=np.int32)[: batch + 1] if T > 0 \
            else np.zeros(batch + 1, dtype=np.int32)
    if hasattr(cu_seqlens, "detach"):
        cu_seqlens = cu_seqlens.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))


def _forward(form, q, k, v, g, beta, cu_seqlens=None, batch=None, scale=None, use_qk_l2norm=True,
             initial_state=None, C=64, threads=1):
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    total_T, Hk, dk = q.shape
    H, dv = v.shape[1], v.shape[2]
    per_channel = g.ndim == 3
    if k.shape != q.shape or v.shape[0] != total_T or H % Hk \
            or g.shape != ((total_T, H, dk) if per_channel else (total_T, H)) \
            or beta.shape != (total_T, H):
        raise ValueError("shape mismatch")
    cu = _cu(cu_seqlens, total_T, batch)
    num_seqs = cu.shape[0] - 1
    if cu[0] != 0 or cu[-1] != total_T:
        raise ValueError("cu_seqlens must start at 0 and end at total_T")
    S0 = _f64(initial_state)
    if S0 is not None and S0.shape != (num_seqs, H, dv, dk):
        raise ValueError("initial_state shape")
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    y = np.zeros((total_T, H, dv), dtype=np.float64)
    S_final = np.zeros((num_seqs, H, dv, dk), dtype=np.float64)
    rc = _load().gdn_oracle_forward(
        form, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), num_seqs, H, Hk, dk, dv, int(per_channel),
        float(scale), int(bool(use_qk_l2norm)), _ptr(S0), _ptr(y), _ptr(S_final), int(C), int(threads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments (cu_seqlens not monotone, C <= 0, or a "
                         "per-channel decay given to the chunked form)")
    return y, S_final


def recurrence(q, k, v, g, beta, cu_seqlens=None, batch=None, scale=None, use_qk_l2norm=True,
               initial_state=None, threads=1):
    """Token-by-token gated delta rule.

    q, k: [total_T, Hk, dk]; v: [total_T, H, dv] with H a multiple of Hk; beta: [total_T, H];
    g (log-decay): [total_T, H], or [total_T, H, dk] for a decay per key channel;
    cu_seqlens: [num_seqs+1] or None (then ``batch`` equal sequences);
    initial_state: [num_seqs, H, dv, dk] or None (zeros).
    Returns (y [total_T, H, dv], final_state [num_seqs, H, dv, dk]) in float64.
    scale None means 1/sqrt(dk).
    """
    return _forward(FORM_RECURRENCE, q, k, v, g, beta, cu_seqlens, batch, scale, use_qk_l2norm,
                    initial_state, 1, threads)


def chunked(q, k, v, g, beta, C=64, cu_seqlens=None, batch=None, scale=None, use_qk_l2norm=True,
            initial_state=None, threads=1):
    """The chunked (UT/WY) algebra in fp64 with chunk size C; same arguments as recurrence."""
    return _forward(FORM_CHUNKED, q, k, v, g, beta, cu_seqlens, batch, scale, use_qk_l2norm,
                    initial_state, C, threads)


def transition_product(q, k, v, g, beta, cu_seqlens=None, batch=None, scale=None,
                       use_qk_l2norm=True, initial_state=None):
    """Unrolled product form S_t = S_0 A_1..A_t + sum B_i A_{i+1}..A_t (tiny T only)."""
    return _forward(FORM_TRANSITION, q, k, v, g, beta, cu_seqlens, batch, scale, use_qk_l2norm,
                    initial_state, 1, 1)


def chunk_decay(g):
    """(gcum, decay) of one chunk: inclusive cumsum and exp(gcum_i - gcum_j) for i >= j."""
    g = _f64(g).reshape(-1)
    L = g.shape[0]
    gcum = np.zeros(L)
    out = np.zeros((L, L))
    _load().gdn_oracle_chunk_decay(_ptr(g), L, _ptr(gcum), _ptr(out))
    return gcum, out


def gate_rmsnorm_silu(y, z, weight=None, eps=1e-6):
    """weight * y / sqrt(mean(y^2) + eps) * silu(z), rows over the last dimension."""
    y = _f64(y)
    z = _f64(z)
    if y.shape != z.shape:
        raise ValueError("y and z must have the same shape")
    dv = y.shape[-1]
    rows = y.size // dv if dv else 0
    w = _f64(weight)
    out = np.zeros_like(y)
    _load().gdn_oracle_gate_rmsnorm_silu(_ptr(y), _ptr(z), _ptr(w), float(eps), _ptr(out), rows, dv)
    return out


def gates_from_logits(a, A_log, dt_bias=None, b=None):
    """g = -exp(A_log) * softplus(a + dt_bias) and beta = sigmoid(b); a, b: [total_T, H]."""
    a = _f64(a)
    A_log = _f64(A_log).reshape(-1)
    total_T, H = a.shape
    dtb = _f64(dt_bias).reshape(-1) if dt_bias is not None else None
    bb = _f64(b) if b is not None else None
    g = np.zeros_like(a)
    beta = np.zeros_like(a) if bb is not None else None
    _load().gdn_oracle_gates_from_logits(_ptr(a), _ptr(A_log), _ptr(dtb), _ptr(bb), _ptr(g),
                                         _ptr(beta), total_T, H)
    return (g, beta) if bb is not None else g


def recurrent_step(q, k, v, g, beta, state, scale=None, use_qk_l2norm=True):
    """One decode token for N sequences: q, k [N, H, dk]; v [N, H, dv]; g, beta [N, H];
    state [N, H, dv, dk].  Returns (y [N, H, dv], new_state)."""
    q = _f64(q)
    N = q.shape[0]
    cu = np.arange(N + 1, dtype=np.int32)
    return recurrence(q, k, v, g, beta, cu_seqlens=cu, scale=scale, use_qk_l2norm=use_qk_l2norm,
                      initial_state=state)


def short_conv(x, weight, cu_seqlens=None, batch=None, state=None, activation=True):
    """Causal depthwise convolution (+ SiLU) over the token axis.

    x: [total_T, channels]; weight: [channels, K]; state: [num_seqs, channels, K-1] carried
    history (oldest first) or None (zeros).  Returns (out [total_T, channels], final state
    [num_seqs, channels, K-1]) in float64."""
    x = _f64(x)
    w = _f64(weight)
    total_T, channels = x.shape
    K = w.shape[1]
    if w.shape[0] != channels or K < 1:
        raise ValueError("weight must be [channels, K]")
    cu = _cu(cu_seqlens, total_T, batch)
    num_seqs = cu.shape[0] - 1
    st = _f64(state)
    if st is not None and st.shape != (num_seqs, channels, K - 1):
        raise ValueError("state shape")
    out = np.zeros_like(x)
    st_out = np.zeros((num_seqs, channels, K - 1))
    rc = _load().gdn_oracle_short_conv(_ptr(x), _ptr(w), cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                       num_seqs, channels, K, _ptr(st), _ptr(out), _ptr(st_out),
                                       int(bool(activation)))
    if rc != 0:
        raise ValueError("cu_seqlens not monotone")
    return out, st_out
