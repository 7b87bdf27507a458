"""Helpers shared by the tests: the parity metric and oracle runs on the seeded inputs."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle

THREADS = max(1, min(16, os.cpu_count() or 1))
TOL_F32 = 1e-4   # max relative L2 error per (sequence, head) slab, fp32 inputs
TOL_BF16 = 1e-2  # same metric, bf16 q/k/v with fp32 state and accumulation


def _np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def rel_l2_tokens(x, ref, cu):
    """Max over (sequence, head) slabs of ||x - ref|| / ||ref|| for token tensors [T, H, d]."""
    x, ref = _np(x), _np(ref)
    cu = [int(c) for c in (cu.tolist() if hasattr(cu, "tolist") else cu)]
    worst = 0.0
    for n in range(len(cu) - 1):
        a, b = cu[n], cu[n + 1]
        if b == a:
            continue
        d = x[a:b] - ref[a:b]                     # [L, H, d]
        num = np.sqrt((d * d).sum(axis=(0, 2)))
        den = np.sqrt((ref[a:b] ** 2).sum(axis=(0, 2)))
        worst = max(worst, float(np.max(num / np.maximum(den, 1e-30))))
    return worst


def rel_l2_states(x, ref):
    """Max over (sequence, head) of the relative L2 error of [N, H, dv, dk] states."""
    x, ref = _np(x), _np(ref)
    d = (x - ref).reshape(x.shape[0] * x.shape[1], -1)
    r = ref.reshape(d.shape)
    num = np.linalg.norm(d, axis=1)
    den = np.linalg.norm(r, axis=1)
    return float(np.max(num / np.maximum(den, 1e-30))) if d.shape[0] else 0.0


def cu_list(inp):
    if inp["cu_seqlens"] is not None:
        return inp["cu_seqlens"].cpu().tolist()
    n, T = inp["num_seqs"], inp["total_T"] // inp["num_seqs"]
    return [i * T for i in range(n + 1)]


def oracle_gates(inp):
    """g, beta from the drawn logits, in fp64 by the oracle, rounded once to fp32.  With logits per
    key channel (a [T, H, d]) each channel is its own column with its head's A_log."""
    a = inp["a"]
    if a.dim() == 3:
        T, H, d = a.shape
        g = oracle.gates_from_logits(a.reshape(T, H * d), inp["A_log"].repeat_interleave(d))
        _, beta = oracle.gates_from_logits(torch.zeros(T, H), inp["A_log"], b=inp["b"])
        return torch.from_numpy(g).float().reshape(T, H, d), torch.from_numpy(beta).float()
    g, beta = oracle.gates_from_logits(a, inp["A_log"], b=inp["b"])
    return torch.from_numpy(g).float(), torch.from_numpy(beta).float()


def oracle_conv_qkv(q, k, v, conv_weight, conv_state, cu):
    """The oracle's short convolution over the mixed q|k|v channels of raw inputs.
    Returns (q, k, v) after convolution + SiLU (float64 numpy, input shapes) and the final
    history [num_seqs, conv_dim, 3].  The convolution output is an activation of the q/k/v type
    (the page's module runs in the model dtype), so it is rounded once to that type here, as the
    kernels do, before the core sees it."""
    T, Hk, d = q.shape
    H = v.shape[1]
    dt = q.dtype if isinstance(q, torch.Tensor) else torch.float64
    x = torch.cat([torch.as_tensor(q).reshape(T, Hk * d).double(), torch.as_tensor(k).reshape(T, Hk * d).double(),
                   torch.as_tensor(v).reshape(T, H * d).double()], dim=1)
    y, st = oracle.short_conv(x, conv_weight, cu_seqlens=np.asarray(cu, dtype=np.int32), state=conv_state)
    y = torch.from_numpy(y).to(dt).double().numpy()
    qc = y[:, :Hk * d].reshape(T, Hk, d)
    kc = y[:, Hk * d:2 * Hk * d].reshape(T, Hk, d)
    vc = y[:, 2 * Hk * d:].reshape(T, H, d)
    return qc, kc, vc, st


def oracle_prefill(inp, g32, b32, scale=None, use_l2=True, threads=THREADS, gate=True,
                   heads=None, seqs=None, weight=None, eps=1e-6):
    """Run the oracle recurrence on the prefill inputs (optionally only some heads / sequences).
    Returns (y_or_o [T, H', d] float64, final [N', H', d, d])."""
    cu = cu_list(inp)
    q, k, v, z, S0 = inp["q"], inp["k"], inp["v"], inp["z"], inp["initial_state"]
    g, b = g32, b32
    if inp.get("conv_weight") is not None:
        q, k, v, _ = oracle_conv_qkv(q, k, v, inp["conv_weight"], inp.get("conv_state"), cu)
        q, k, v = (torch.from_numpy(t) for t in (q, k, v))
    if heads is not None:
        assert q.shape[1] == v.shape[1], "head sampling needs one query/key head per value head"
        sel = lambda t: t[:, heads] if t is not None else None  # noqa: E731
        q, k, v, z, g, b = (sel(t) for t in (q, k, v, z, g, b))
        S0 = S0[:, heads] if S0 is not None else None
    if seqs is not None:
        parts = [(cu[n], cu[n + 1]) for n in seqs]
        idx = torch.cat([torch.arange(a_, b_) for a_, b_ in parts]) if parts else torch.arange(0)
        q, k, v, g, b = (t[idx] for t in (q, k, v, g, b))
        z = z[idx] if z is not None else None
        S0 = S0[seqs] if S0 is not None else None
        cu = np.concatenate([[0], np.cumsum([b_ - a_ for a_, b_ in parts])]).astype(np.int32)
    y, S = oracle.recurrence(q, k, v, g, b, cu_seqlens=np.asarray(cu, dtype=np.int32), scale=scale,
                             use_qk_l2norm=use_l2, initial_state=S0, threads=threads)
    if gate and z is not None:
        y = oracle.gate_rmsnorm_silu(y, z, weight, eps=eps)
    return y, S
