"""Seeded synthetic inputs for the gated delta rule workloads.

Only random draws live here -- no step of the method: q and k are drawn raw (the kernels and
the oracle normalise them), and the gates are drawn as logits (a, b) and per-head log-rates
(A_log), which the gate preparation turns into g = log(alpha) and beta.  Both the CUDA path and
the oracle are fed from these draws, so this module is the one thing they share.

Workloads (named by what they are):
  tiny     B=1, H=2, T=256, d=64, fp32 q/k/v; zero initial state; outputs y and the final state.
  prefill  B=2, H=16, T=4096, d=128, bf16 q/k/v; fp32 gates and z; fused RMSNorm*SiLU output.
  decode   one token for 256 sequences, H=32, d=128; fp32 state ~ N(0, 0.02^2); bf16 q/k/v.
  varlen   64 packed sequences with lengths uniform in [128, 8192], H=16, d=128, bf16;
           initial states ~ N(0, 0.02^2) per sequence; final states written.
  long     B=1, H=32, T=131072, d=128, bf16; a ~ N(-4, 1) (alpha close to 1); fused gate.
  prefill_gva   the prefill workload with 4 query/key heads shared by the 16 value heads.
  prefill_kda   the prefill workload with one decay per key channel (a drawn per channel).
  prefill_conv  the prefill workload with the short convolution fused (raw q, k, v drawn; taps
                per channel ~ U(-1/2, 1/2), the default uniform bound 1/sqrt(fan_in) of a
                depthwise kernel of 4 taps; zero history, i.e. sequences that start here).
  prefill_d64   the prefill workload with head size d_k = d_v = 64.
Distributions common to all: q, k, v ~ N(0, 1); a ~ N(-1, 1) unless stated; A = exp(A_log) with
A_log ~ U[0, ln 8] per head; b ~ N(0, 1) (beta = sigmoid(b)); z ~ N(0, 1).
Options (any workload): Hk (query/key heads, default H), per_channel (a drawn [T, H, d] so that
g = -exp(A_log) softplus(a) is per key channel), conv (taps drawn), conv_state (history ~ N(0, 1)).
Draw order from one torch.Generator seeded with the workload's seed: lengths (varlen only),
q, k, v, a, A_log, b, z (if gated), initial state (if any), conv taps, conv history (if any).
"""
from __future__ import annotations

import math

import torch

WORKLOADS = {
    "tiny": dict(kind="prefill", seed=0, num_seqs=1, T=256, H=2, d=64, dtype=torch.float32,
                 a_mean=-1.0, gate=False, init_state=False),
    "prefill": dict(kind="prefill", seed=1, num_seqs=2, T=4096, H=16, d=128, dtype=torch.bfloat16,
                    a_mean=-1.0, gate=True, init_state=False),
    "decode": dict(kind="decode", seed=2, N=256, H=32, d=128, dtype=torch.bfloat16, a_mean=-1.0,
                   state_std=0.02),
    "varlen": dict(kind="prefill", seed=3, num_seqs=64, len_range=(128, 8192), H=16, d=128,
                   dtype=torch.bfloat16, a_mean=-1.0, gate=False, init_state=True, state_std=0.02),
    "long": dict(kind="prefill", seed=4, num_seqs=1, T=131072, H=32, d=128, dtype=torch.bfloat16,
                 a_mean=-4.0, gate=True, init_state=False),
    "prefill_gva": dict(kind="prefill", seed=5, num_seqs=2, T=4096, H=16, Hk=4, d=128,
                        dtype=torch.bfloat16, a_mean=-1.0, gate=True, init_state=False),
    "prefill_kda": dict(kind="prefill", seed=6, num_seqs=2, T=4096, H=16, d=128, dtype=torch.bfloat16,
                        a_mean=-1.0, gate=True, init_state=False, per_channel=True),
    "prefill_conv": dict(kind="prefill", seed=7, num_seqs=2, T=4096, H=16, d=128, dtype=torch.bfloat16,
                         a_mean=-1.0, gate=True, init_state=False, conv=True),
    "prefill_d64": dict(kind="prefill", seed=8, num_seqs=2, T=4096, H=16, d=64, dtype=torch.bfloat16,
                        a_mean=-1.0, gate=True, init_state=False),
}


def conv_dim(H, Hk, d):
    """Channels of the mixed q|k|v projection the short convolution runs over."""
    return 2 * Hk * d + H * d


def workload(name: str, **overrides) -> dict:
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    cfg["name"] = name
    return cfg


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def prefill_inputs(cfg, device="cpu", seed=None) -> dict:
    """Draw one prefill batch.  Returns q, k, v [total_T, H, d] (cfg dtype), a, b [total_T, H],
    A_log [H], z [total_T, H, d] or None, initial_state [num_seqs, H, d, d] or None,
    cu_seqlens int32 [num_seqs+1] (on `device`) or None for equal lengths, lengths (list)."""
    if isinstance(cfg, str):
        cfg = workload(cfg)
    seed = cfg["seed"] if seed is None else seed
    gen = _gen(device, seed)
    H, d, dt = cfg["H"], cfg["d"], cfg["dtype"]
    n = cfg["num_seqs"]
    if "lengths" in cfg:
        lengths = [int(x) for x in cfg["lengths"]]
    elif "len_range" in cfg:
        lo, hi = cfg["len_range"]
        lengths = torch.randint(lo, hi + 1, (n,), generator=gen, device=device).tolist()
    else:
        lengths = [cfg["T"]] * n
    total_T = int(sum(lengths))
    varlen = "len_range" in cfg or "lengths" in cfg

    def randn(*shape):
        return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)

    Hk = cfg.get("Hk", H)
    q = randn(total_T, Hk, d).to(dt)
    k = randn(total_T, Hk, d).to(dt)
    v = randn(total_T, H, d).to(dt)
    a = (randn(total_T, H, d) if cfg.get("per_channel") else randn(total_T, H)) + cfg["a_mean"]
    A_log = torch.rand(H, generator=gen, device=device, dtype=torch.float32) * math.log(8.0)
    b = randn(total_T, H)
    z = randn(total_T, H, d) if cfg.get("gate") else None
    S0 = randn(n, H, d, d) * cfg.get("state_std", 0.02) if cfg.get("init_state") else None
    C = conv_dim(H, Hk, d)
    conv_w = (torch.rand(C, 4, generator=gen, device=device) - 0.5) if cfg.get("conv") else None
    conv_s = randn(n, C, 3) if cfg.get("conv_state") else None
    cu = None
    if varlen:
        offs = [0]
        for L in lengths:
            offs.append(offs[-1] + L)
        cu = torch.tensor(offs, dtype=torch.int32, device=device)
    return dict(q=q, k=k, v=v, a=a, A_log=A_log, b=b, z=z, initial_state=S0, cu_seqlens=cu,
                num_seqs=n, lengths=lengths, total_T=total_T, conv_weight=conv_w, conv_state=conv_s,
                cfg=cfg)


def decode_inputs(cfg, device="cpu", seed=None) -> dict:
    """Draw one decode step: q, k, v [N, H, d], a, b [N, H], A_log [H], state [N, H, d, d]."""
    if isinstance(cfg, str):
        cfg = workload(cfg)
    seed = cfg["seed"] if seed is None else seed
    gen = _gen(device, seed)
    N, H, d, dt = cfg["N"], cfg["H"], cfg["d"], cfg["dtype"]

    def randn(*shape):
        return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)

    q = randn(N, H, d).to(dt)
    k = randn(N, H, d).to(dt)
    v = randn(N, H, d).to(dt)
    a = randn(N, H) + cfg["a_mean"]
    A_log = torch.rand(H, generator=gen, device=device, dtype=torch.float32) * math.log(8.0)
    b = randn(N, H)
    z = randn(N, H, d) if cfg.get("gate") else None
    state = randn(N, H, d, d) * cfg.get("state_std", 0.02)
    return dict(q=q, k=k, v=v, a=a, A_log=A_log, b=b, z=z, state=state, cfg=cfg)
