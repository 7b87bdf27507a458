#!/usr/bin/env python3
"""Benchmark of the gated delta rule library on one GB300 (or N replicas under torchrun).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdn|reference]

One step = the whole prefill path on the prefill workload (B=2 sequences x T=4096 tokens, H=16
heads, d_k=d_v=128, bf16 q/k/v, fp32 gates, fused RMSNorm*SiLU gate): gate preparation
(gdn_decay_from_logits) followed by the chunked prefill (gdn_chunk_fwd).  The decode workload
(256 sequences x 32 heads, fp32 state of 128x128, bf16 q/k/v) is timed in the same run and reported
in the "decode" object.  Inputs are resident in HBM before the timed region; L2 (129 MB) is flushed
by writing a 512 MB buffer before every timed prefill step; the decode state (512 MiB) is larger
than L2.  Times are CUDA events on the launching stream; value is whole-job tokens/s (max time over
ranks).  The "e2e" object is the same metric through the C ABI with host buffers: pinned-host
inputs copied in and the output and final state copied out inside every timed step.

--impl reference times the fp64 CPU oracle (the only reference this method has) on a bounded
sample of the same workload and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

C_CHUNK = 64


def prefill_flops_per_token_head(d, C=C_CHUNK):
    """Five C x C x d products (K K^T, Q K^T, W, U, (QK^T*D) V_new), three C x d x d products
    (W S^T, Q S^T, V_new^T K), and the triangular solve (C^3/3 per chunk), per token."""
    return 10 * C * d + 6 * d * d + C * C / 3.0


def prefill_bytes(total_T, H, d, num_seqs, qkv_bytes=2, out_bytes=2, gated=True, init_state=False):
    """Algorithmic HBM bytes of one gdn_chunk_fwd call: q, k, v, g, beta, z, out once, and the
    final (plus initial) state once per (sequence, head)."""
    per_tok_head = 3 * d * qkv_bytes + 8 + (d * 4 if gated else 0) + d * out_bytes
    states = num_seqs * H * d * d * 4 * (2 if init_state else 1)
    return total_T * H * per_tok_head + states


def decode_bytes(N, H, d, qkv_bytes=2, out_bytes=2):
    """Per (sequence, head): state read + write, q, k, v, g, beta, y."""
    return N * H * (2 * d * d * 4 + 3 * d * qkv_bytes + 8 + d * out_bytes)


def _source_digest(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profile_record(key):
    """The committed ncu figures of a launch unit in profiles/traffic.json (DRAM bytes per launch
    and, for the chunk kernels, the tensor-pipe utilisation); None when missing or when the
    kernel's sources changed after the capture (the record holds a digest of them)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[key]
    except Exception:
        return None
    if _source_digest(rec["sources"]) != rec["digest"]:
        return None
    return rec


def traffic_record(key):
    """DRAM bytes per launch of a kernel from the committed ncu capture, or None (see above)."""
    rec = profile_record(key)
    return rec.get("dram_bytes_per_launch") if rec else None


def tensor_pipe_record(key):
    """ncu sm__pipe_tensor_cycles_active (% of peak sustained over active SM cycles) per kernel of
    a launch unit, from the same digest-keyed record, or None."""
    rec = profile_record(key)
    return rec.get("tensor_pipe_pct") if rec else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": 2070.0}, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"gdn_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl != "reference" else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------------------------
# oracle (CPU) timing: the cpu_baseline leg and the --impl reference arm
# ---------------------------------------------------------------------------------------------

def time_oracle(inp, heads, threads):
    """Time the oracle (recurrence + gate) on the given heads of the prefill inputs."""
    import numpy as np
    import oracle
    q, k, v = (inp[n][:, heads] for n in ("q", "k", "v"))
    z = inp["z"][:, heads] if inp["z"] is not None else None
    n, T = inp["num_seqs"], inp["total_T"] // inp["num_seqs"]
    cu = np.arange(0, inp["total_T"] + 1, T, dtype=np.int32)
    t0 = time.perf_counter()
    g, beta = oracle.gates_from_logits(inp["a"][:, heads], inp["A_log"][heads], b=inp["b"][:, heads])
    y, S = oracle.recurrence(q, k, v, g, beta, cu_seqlens=cu, threads=threads)
    if z is not None:
        oracle.gate_rmsnorm_silu(y, z)
    return time.perf_counter() - t0


def oracle_rate(inp, H, seconds_budget=20.0, threads=None):
    """Tokens/s of the oracle on the full workload, estimated from a bounded sample of heads."""
    threads = threads or os.cpu_count() or 1
    # a one-head probe on one thread sizes the sample so that the measurement takes roughly the
    # budget; it also gives the single-thread rate
    t1 = time_oracle(inp, [0], 1)
    oracle_rate.single_thread = inp["total_T"] / (H * t1)
    per_head_parallel = t1 / min(threads, inp["num_seqs"])
    n_heads = max(1, min(H, int(seconds_budget / max(per_head_parallel, 1e-6) / 2)))
    heads = list(range(n_heads))
    th = max(1, min(threads, n_heads * inp["num_seqs"]))
    # when the whole workload is shorter than the budget, repeat full passes to fill it
    t = time_oracle(inp, heads, th)
    reps = 1
    while t < 0.5 * seconds_budget and reps < 1000:
        t += time_oracle(inp, heads, th)
        reps += 1
    tok_per_s = reps * inp["total_T"] * (n_heads / H) / t
    sample = (f"{n_heads} of {H} heads x {inp['num_seqs']} sequences x "
              f"{inp['total_T'] // inp['num_seqs']} tokens (recurrence + gate, fp64), {reps} pass(es), "
              f"{th} threads, {t:.2f} s; tokens/s scaled to all heads")
    return tok_per_s, th, sample, t


# ---------------------------------------------------------------------------------------------
# GPU measurements
# ---------------------------------------------------------------------------------------------

# time slices of each sequence in the streamed end-to-end prefill step, as shares of the sequence
# (host link overlapped with the kernels); the short last slices keep the tail after the last copy short
E2E_SPLIT = (3, 1)


def ev():
    return torch.cuda.Event(enable_timing=True)


def bench_prefill(args, dev):
    import gated_deltanet_recurrence_gb300 as gdn
    from gated_deltanet_recurrence_gb300 import synthetic
    inp_cpu = synthetic.prefill_inputs("prefill")
    cfg = inp_cpu["cfg"]
    stream = torch.cuda.current_stream()
    d_in = {k_: (v_.to(dev) if isinstance(v_, torch.Tensor) else v_) for k_, v_ in inp_cpu.items()}
    total_T, H, d, n = inp_cpu["total_T"], cfg["H"], cfg["d"], inp_cpu["num_seqs"]
    g = torch.empty(total_T, H, device=dev)
    beta = torch.empty(total_T, H, device=dev)
    out = torch.empty(total_T, H, d, dtype=torch.bfloat16, device=dev)
    Sf = torch.empty(n, H, d, d, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    ws_bytes = gdn.lib().gdn_chunk_fwd_workspace_size(n, total_T, H, d, d, gdn.GDN_BF16)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)

    def step():
        gdn.gdn_decay_from_logits(d_in["a"], d_in["A_log"], b=d_in["b"], g_out=g, beta_out=beta)
        e_mid = ev()
        e_mid.record(stream)
        gdn.gdn_chunk_fwd(d_in["q"], d_in["k"], d_in["v"], g, beta, num_seqs=n,
                          gate_z=d_in["z"], out=out, final_state=Sf, workspace=ws)
        return e_mid

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_error() == 0
    step_ms, chunk_ms = [], []
    barrier(args.world)
    torch.cuda.synchronize()
    clocks = ClockSampler(args.local)
    clocks.start()
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = ev(), ev()
        e0.record(stream)
        e_mid = step()
        e1.record(stream)
        step_ms.append((e0, e_mid, e1))
    torch.cuda.synchronize()
    barrier(args.world)
    clk = clocks.stop()
    tot = [a.elapsed_time(c) for a, _, c in step_ms]
    chunk_ms = [b_.elapsed_time(c) for _, b_, c in step_ms]
    ms = statistics.mean(tot)
    kms = statistics.mean(chunk_ms)
    assert gdn.gdn_get_device_error() == 0

    # ---- end to end through the ABI with host buffers ----
    # Every step copies all inputs in from pinned host memory and the outputs back.  The host link
    # (about 0.2 TB/s each way on this machine) takes 5x longer than the kernels, so the step is
    # streamed: every sequence is cut into time slices (E2E_SPLIT; each a contiguous host range, so one
    # copy per tensor), slice (s, p) is copied in on one stream, run by gdn_decay_from_logits +
    # gdn_chunk_fwd on another (one sequence; its initial state is slice p - 1's final state, in
    # place) and copied out on a third.  The copies of later slices overlap the kernels and the
    # copy-out of earlier ones.  Slices are whole chunks, so the result is bit-identical to the
    # single call (checked below).
    pinned = {k_: v_.pin_memory() for k_, v_ in inp_cpu.items()
              if isinstance(v_, torch.Tensor) and k_ in ("q", "k", "v", "a", "b", "z")}
    A_log_h = inp_cpu["A_log"].pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    Sf_h = torch.empty(Sf.shape, dtype=Sf.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in pinned.values()) + A_log_h.numel() * A_log_h.element_size()
    d2h = out_h.numel() * out_h.element_size() + Sf_h.numel() * Sf_h.element_size()
    Tn = total_T // n                      # tokens per sequence
    unit_ = Tn // sum(E2E_SPLIT)
    assert unit_ * sum(E2E_SPLIT) == Tn and unit_ % 64 == 0  # slices are whole chunks
    lens = [unit_ * w for w in E2E_SPLIT]
    starts = [sum(lens[:p_]) for p_ in range(len(lens))]
    # (sequence, slice, first token, length), slice-major: the first slices of every sequence first
    slices = [(sq, p_, sq * Tn + starts[p_], lens[p_]) for p_ in range(len(lens)) for sq in range(n)]
    bufs = [{k_: torch.empty((Ls,) + t.shape[1:], dtype=t.dtype, device=dev) for k_, t in pinned.items()}
            for (_, _, _, Ls) in slices]
    A_log_d = torch.empty_like(A_log_h, device=dev)
    g_p = [torch.empty(Ls, H, device=dev) for (_, _, _, Ls) in slices]
    b_p = [torch.empty(Ls, H, device=dev) for (_, _, _, Ls) in slices]
    o_p = [torch.empty(Ls, H, d, dtype=torch.bfloat16, device=dev) for (_, _, _, Ls) in slices]
    S_e = torch.empty(n, H, d, d, device=dev)
    ws_p = gdn.lib().gdn_chunk_fwd_workspace_size(1, max(lens), H, d, d, gdn.GDN_BF16)
    ws_e = torch.empty(max(ws_p, 1), dtype=torch.uint8, device=dev)
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_step():
        start = ev()
        start.record(stream)
        for s_ in (s_in, s_run, s_out):
            s_.wait_event(start)
        # all copies in are enqueued first, then the kernels, then the copies out: enqueued in
        # another order, a copy can queue behind a kernel when the streams share a hardware queue
        copied, ran = [], []
        with torch.cuda.stream(s_in):
            A_log_d.copy_(A_log_h, non_blocking=True)
            for i, (_, _, t0, Ls) in enumerate(slices):
                for k_, t in pinned.items():
                    bufs[i][k_].copy_(t[t0:t0 + Ls], non_blocking=True)
                e_ = ev()
                e_.record(s_in)
                copied.append(e_)
        with torch.cuda.stream(s_run):
            for i, (sq, p_, _, _) in enumerate(slices):
                s_run.wait_event(copied[i])
                x, S_seq = bufs[i], S_e[sq:sq + 1]
                gdn.gdn_decay_from_logits(x["a"], A_log_d, b=x["b"], g_out=g_p[i], beta_out=b_p[i])
                gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], g_p[i], b_p[i], num_seqs=1,
                                  initial_state=S_seq if p_ > 0 else None, gate_z=x["z"], out=o_p[i],
                                  final_state=S_seq, workspace=ws_e)
                e_ = ev()
                e_.record(s_run)
                ran.append(e_)
        with torch.cuda.stream(s_out):
            for i, (_, _, t0, Ls) in enumerate(slices):
                s_out.wait_event(ran[i])
                out_h[t0:t0 + Ls].copy_(o_p[i], non_blocking=True)
            Sf_h.copy_(S_e, non_blocking=True)
        for s_ in (s_in, s_run, s_out):
            stream.wait_stream(s_)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_error() == 0
    # the streamed step reproduces the single call exactly
    assert torch.equal(out_h, out.cpu()) and torch.equal(Sf_h, Sf.cpu()), "streamed e2e step differs"
    e2e_ms = []
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = ev(), ev()
        e0.record(stream)
        e2e_step()
        e1.record(stream)
        e2e_ms.append((e0, e1))
    torch.cuda.synchronize()
    e2e = statistics.mean(a.elapsed_time(b_) for a, b_ in e2e_ms)
    # kernels per step: gdn_decay_from_logits (1) + gdn_chunk_fwd (tensor-core path: chunk map and
    # either the fused kernel, taken when the units are at most half the SMs, or chunk prep + state
    # pass; 1 on the CUDA-core path)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fused = n * H <= sms // 2
    per_step = 1 + ((2 if fused else 3) if ws_bytes > 0 else 1)
    return dict(ms=ms, kernel_ms=kms, clocks=clk, e2e_ms=e2e, h2d=h2d, d2h=d2h, total_T=total_T,
                H=H, d=d, num_seqs=n, inp=inp_cpu, launches=per_step * args.steps)


def bench_decode(args, dev):
    import gated_deltanet_recurrence_gb300 as gdn
    from gated_deltanet_recurrence_gb300 import synthetic
    inp = synthetic.decode_inputs("decode")
    cfg = inp["cfg"]
    N, H, d = cfg["N"], cfg["H"], cfg["d"]
    stream = torch.cuda.current_stream()
    q, k, v, a, A_log, b = (inp[x].to(dev) for x in ("q", "k", "v", "a", "A_log", "b"))
    state = inp["state"].to(dev)
    g = torch.empty(N, H, device=dev)
    beta = torch.empty(N, H, device=dev)
    out = torch.empty(N, H, d, dtype=torch.bfloat16, device=dev)
    gdn.gdn_decay_from_logits(a, A_log, b=b, g_out=g, beta_out=beta)
    # L2 is flushed before every timed iteration (the state, 1.07 GB, is larger than L2, but the
    # tail written by the previous iteration would otherwise still be cached)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        gdn.gdn_recurrent_step(q, k, v, g, beta, state, out=out)
    torch.cuda.synchronize()
    times = []
    for _ in range(max(args.steps, 20)):
        flush.zero_()
        e0, e1 = ev(), ev()
        e0.record(stream)
        gdn.gdn_decay_from_logits(a, A_log, b=b, g_out=g, beta_out=beta)
        e_mid = ev()
        e_mid.record(stream)
        gdn.gdn_recurrent_step(q, k, v, g, beta, state, out=out)
        e1.record(stream)
        times.append((e0, e_mid, e1))
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_error() == 0
    step_ms = statistics.mean(x.elapsed_time(z) for x, _, z in times)
    kern_ms = statistics.mean(y.elapsed_time(z) for _, y, z in times)

    # pooled multi-token decode: the same 256 sequences pick their states from a 512-slot pool
    # through an index array and run T = 4 tokens each (state read and written once)
    Tm, slots = 4, 2 * N
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    qm, km, vm = (torch.randn(N, Tm, H, d, generator=gen, device=dev).to(torch.bfloat16) for _ in range(3))
    gm = -torch.rand(N, Tm, H, generator=gen, device=dev)
    bm = torch.rand(N, Tm, H, generator=gen, device=dev)
    pool = torch.randn(slots, H, d, d, generator=gen, device=dev) * 0.02
    idx = torch.randperm(slots, generator=gen, device=dev)[:N].to(torch.int32)
    outm = torch.empty(N, Tm, H, d, dtype=torch.bfloat16, device=dev)
    for _ in range(args.warmup):
        gdn.gdn_recurrent_multi_step(qm, km, vm, gm, bm, pool, state_indices=idx, out=outm)
    torch.cuda.synchronize()
    mt = []
    for _ in range(max(args.steps, 20)):
        flush.zero_()
        e0, e1 = ev(), ev()
        e0.record(stream)
        gdn.gdn_recurrent_multi_step(qm, km, vm, gm, bm, pool, state_indices=idx, out=outm)
        e1.record(stream)
        mt.append((e0, e1))
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_error() == 0
    multi_ms = statistics.mean(x.elapsed_time(y) for x, y in mt)
    multi_bytes = N * H * (2 * d * d * 4 + Tm * (3 * d * 2 + 8 + d * 2)) + N * 4
    return dict(ms=step_ms, kernel_ms=kern_ms, N=N, H=H, d=d, multi_ms=multi_ms, multi_T=Tm,
                multi_bytes=multi_bytes, multi_slots=slots)


def bench_variants(args, dev):
    """The prefill options on the prefill workload's sizes (B=2 x T=4096, H=16, d=128, bf16, fused
    gate): 4 query/key heads shared by 16 value heads, a decay per key channel, the fused short
    convolution, and head size 64; plus one decode step with the convolution and its history updated
    in place.  Each
    timed region is one gdn_chunk_fwd (or gdn_recurrent_step) call, L2 flushed before every call."""
    import gated_deltanet_recurrence_gb300 as gdn
    from gated_deltanet_recurrence_gb300 import synthetic
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    peaks, _ = load_peaks()
    res = {}
    steps = max(3, min(args.steps, 10))
    for name in ("prefill_gva", "prefill_kda", "prefill_conv", "prefill_d64"):
        inp = synthetic.prefill_inputs(name)
        cfg = inp["cfg"]
        total_T, H, d, n = inp["total_T"], cfg["H"], cfg["d"], inp["num_seqs"]
        Hk = cfg.get("Hk", H)
        q, k, v, z = (inp[x].to(dev) for x in ("q", "k", "v", "z"))
        A_log, b = inp["A_log"].to(dev), inp["b"].to(dev)
        a = inp["a"].to(dev)
        if a.dim() == 3:  # one log-decay per key channel: each channel is a column with its head's A_log
            g = gdn.gdn_decay_from_logits(a.reshape(total_T, H * d), A_log.repeat_interleave(d)).reshape(total_T, H, d)
            _, beta = gdn.gdn_decay_from_logits(torch.zeros_like(b), A_log, b=b)
        else:
            g, beta = gdn.gdn_decay_from_logits(a, A_log, b=b)
        cw = inp["conv_weight"].to(dev) if inp["conv_weight"] is not None else None
        out = torch.empty(total_T, H, d, dtype=torch.bfloat16, device=dev)
        Sf = torch.empty(n, H, d, d, device=dev)
        ws_bytes = gdn.lib().gdn_chunk_fwd_workspace_size(n, total_T, H, d, d, gdn.GDN_BF16)
        ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)

        def call():
            gdn.gdn_chunk_fwd(q, k, v, g, beta, num_seqs=n, conv_weight=cw, gate_z=z, out=out,
                              final_state=Sf, workspace=ws)

        for _ in range(2):
            call()
        torch.cuda.synchronize()
        assert gdn.gdn_get_device_error() == 0
        ts = []
        for _ in range(steps):
            flush.zero_()
            e0, e1 = ev(), ev()
            e0.record(stream)
            call()
            e1.record(stream)
            ts.append((e0, e1))
        torch.cuda.synchronize()
        assert gdn.gdn_get_device_error() == 0
        ms = statistics.mean(x.elapsed_time(y) for x, y in ts)
        per_tok_head = (2 * Hk / H + 1) * d * 2 + 4 * (d if a.dim() == 3 else 1) + 4 + d * 4 + d * 2
        byts = total_T * H * per_tok_head + n * H * d * d * 4
        gbs = byts / (ms / 1e3) / 1e9
        path = "tensor-core" if ws_bytes > 0 else "cuda-core"
        res[name] = {"tokens_per_s": total_T / (ms / 1e3), "ms": ms, "path": path, "H": H, "H_k": Hk,
                     "decay": "per key channel" if a.dim() == 3 else "per head",
                     "conv": cw is not None, "algorithmic_bytes": byts, "hbm_gbs": gbs,
                     "hbm_frac": gbs / peaks["hbm_gbs"]}
        del q, k, v, z, g, beta, out, Sf, ws

    # decode with the fused convolution, history updated in place
    inp = synthetic.decode_inputs("decode")
    cfg = inp["cfg"]
    N, H, d = cfg["N"], cfg["H"], cfg["d"]
    q, k, v, a, A_log, b = (inp[x].to(dev) for x in ("q", "k", "v", "a", "A_log", "b"))
    state = inp["state"].to(dev)
    g, beta = gdn.gdn_decay_from_logits(a, A_log, b=b)
    C = synthetic.conv_dim(H, H, d)
    gen = torch.Generator(device=dev)
    gen.manual_seed(11)
    cw = torch.rand(C, 4, generator=gen, device=dev) - 0.5
    cs = torch.randn(N, C, 3, generator=gen, device=dev)
    out = torch.empty(N, H, d, dtype=torch.bfloat16, device=dev)

    def dcall():
        gdn.gdn_recurrent_step(q, k, v, g, beta, state, conv_weight=cw, conv_state=cs, conv_state_out=cs, out=out)

    for _ in range(3):
        dcall()
    torch.cuda.synchronize()
    ts = []
    for _ in range(max(args.steps, 20)):
        flush.zero_()
        e0, e1 = ev(), ev()
        e0.record(stream)
        dcall()
        e1.record(stream)
        ts.append((e0, e1))
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_error() == 0
    ms = statistics.mean(x.elapsed_time(y) for x, y in ts)
    byts = decode_bytes(N, H, d) + N * C * 3 * 4 * 2 + C * 16
    res["decode_conv"] = {"tokens_per_s": N / (ms / 1e3), "ms": ms, "algorithmic_bytes": byts,
                          "hbm_gbs": byts / (ms / 1e3) / 1e9,
                          "hbm_frac": byts / (ms / 1e3) / 1e9 / peaks["hbm_gbs"]}
    return res


def two_kernel_time(call, flush, steps=3):
    """Mean CUDA-event time of one gdn_chunk_fwd call in the two-kernel form (chunk preparation,
    then the serial pass), L2 flushed before each call."""
    import gated_deltanet_recurrence_gb300 as gdn
    stream = torch.cuda.current_stream()
    gdn.gdn_set_kernel_forms(prefill_fused=gdn.GDN_FORM_OFF)
    try:
        call()
        torch.cuda.synchronize()
        ts = []
        for _ in range(steps):
            flush.zero_()
            e0, e1 = ev(), ev()
            e0.record(stream)
            call()
            e1.record(stream)
            ts.append((e0, e1))
        torch.cuda.synchronize()
    finally:
        gdn.gdn_set_kernel_forms()
    return statistics.mean(x.elapsed_time(y) for x, y in ts)


def bench_workloads(args, dev, names):
    """The other prefill workloads (tiny: 1 x 256 tokens, H = 2, d = 64, fp32; varlen: 64 sequences
    of 128-8192 tokens with initial states; long: one 131,072-token sequence, H = 32, fused gate),
    timed like the headline step: gdn_decay_from_logits + gdn_chunk_fwd, L2 flushed before every
    step, CUDA events.  The long workload also reports the serial pass's share of the call."""
    import gated_deltanet_recurrence_gb300 as gdn
    from gated_deltanet_recurrence_gb300 import synthetic
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    res = {}
    for wl in names:
        inp = synthetic.prefill_inputs(wl)
        cfg = inp["cfg"]
        H, d, n, T = cfg["H"], cfg["d"], inp["num_seqs"], inp["total_T"]
        q, k, v, a, A_log, b = (inp[x].to(dev) for x in ("q", "k", "v", "a", "A_log", "b"))
        z = inp["z"].to(dev) if inp["z"] is not None else None
        S0 = inp["initial_state"].to(dev) if inp["initial_state"] is not None else None
        cu = inp["cu_seqlens"].to(dev) if inp["cu_seqlens"] is not None else None
        g = torch.empty(T, H, device=dev)
        beta = torch.empty(T, H, device=dev)
        out = torch.empty(T, H, d, dtype=q.dtype, device=dev)
        Sf = torch.empty(n, H, d, d, device=dev)
        dt = gdn.GDN_BF16 if q.dtype == torch.bfloat16 else gdn.GDN_F32
        ws = torch.empty(max(gdn.lib().gdn_chunk_fwd_workspace_size(n, T, H, d, d, dt), 1),
                         dtype=torch.uint8, device=dev)

        def step():
            gdn.gdn_decay_from_logits(a, A_log, b=b, g_out=g, beta_out=beta)
            gdn.gdn_chunk_fwd(q, k, v, g, beta, cu_seqlens=cu, num_seqs=n, initial_state=S0, gate_z=z,
                              out=out, final_state=Sf, workspace=ws)

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        ts = []
        for _ in range(min(args.steps, 10)):
            flush.zero_()
            e0, e1 = ev(), ev()
            e0.record(stream)
            step()
            e1.record(stream)
            ts.append((e0, e1))
        torch.cuda.synchronize()
        assert gdn.gdn_get_device_error() == 0
        ms = statistics.mean(x.elapsed_time(y) for x, y in ts)
        eb = q.element_size()
        byts = prefill_bytes(T, H, d, n, qkv_bytes=eb, out_bytes=eb, gated=z is not None,
                             init_state=S0 is not None)
        fused = n * H <= sms // 2
        tc = q.dtype == torch.bfloat16 and d == 128
        path = ("CUDA-core" if not tc else "tensor-core fused" if fused else "tensor-core two-kernel")
        peaks, peak_src = load_peaks()
        gbs = byts / (ms / 1e3) / 1e9
        res[wl] = {"metric": "prefill tokens/s", "value": T / (ms / 1e3), "unit": "tokens/s",
                   "tokens": T, "num_seqs": n, "units": n * H, "H": H, "d": d,
                   "dtype": "bf16" if q.dtype == torch.bfloat16 else "f32", "ms_per_step": ms,
                   "path": path, "steps": len(ts),
                   "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes": byts,
                                "traffic": traffic_record(f"gdn_chunk_fwd[{wl}]"),
                                "peak_source": f"{peak_src} hbm_gbs", "timed": "whole step"}}
        if wl == "long" and tc:
            # the serial state pass's share: the two-kernel form (preparation, then the serial pass)
            # timed live, split by the committed ncu launch list of the same call (digest-keyed)
            def call():
                gdn.gdn_chunk_fwd(q, k, v, g, beta, cu_seqlens=cu, num_seqs=n, initial_state=S0, gate_z=z,
                                  out=out, final_state=Sf, workspace=ws)
            rec = profile_record("gdn_chunk_fwd[long]") or {}
            res[wl]["serial_pass"] = {"two_kernel_call_ms": two_kernel_time(call, flush),
                                      "share_of_two_kernel_call": rec.get("serial_pass_share"),
                                      "kernel_us_ncu": rec.get("kernel_us"),
                                      "source": "ncu launch list in profiles/traffic.json (null once the sources change)"}
        del q, k, v, a, b, z, S0, out, ws, g, beta, Sf
        torch.cuda.empty_cache()
    return res


def run_gdn(args):
    dev = torch.device("cuda", args.local)
    torch.cuda.set_device(dev)
    if args.prefill_form != "auto":
        import gated_deltanet_recurrence_gb300 as gdn
        gdn.gdn_set_kernel_forms(prefill_fused=gdn.GDN_FORM_ON if args.prefill_form == "fused" else gdn.GDN_FORM_OFF)
    peaks, peak_src = load_peaks()
    if args.workloads:
        res = bench_workloads(args, dev, [w for w in args.workloads.split(",") if w])
        if args.rank == 0:
            print(json.dumps({"workloads": res, "l2": "flushed (512 MB write) before each step",
                              "step": "gdn_decay_from_logits + gdn_chunk_fwd"}), flush=True)
        return
    if args.only == "decode":
        dc = bench_decode(args, dev)
        if args.rank == 0:
            print(json.dumps({"decode_ms": dc["ms"], "decode_kernel_ms": dc["kernel_ms"]}), flush=True)
        return
    pf = bench_prefill(args, dev)
    if args.only == "prefill":
        if args.rank == 0:
            print(json.dumps({"prefill_ms": pf["ms"], "prefill_kernel_ms": pf["kernel_ms"],
                              "e2e_ms": pf["e2e_ms"]}), flush=True)
        return
    dc = bench_decode(args, dev)
    variants = bench_variants(args, dev) if not args.no_variants else None
    workloads = bench_workloads(args, dev, ["tiny", "varlen", "long"]) if not args.no_workloads else None
    world = args.world
    ms = max_over_ranks(pf["ms"], world)
    e2e_ms = max_over_ranks(pf["e2e_ms"], world)
    dms = max_over_ranks(dc["ms"], world)
    tokens = pf["total_T"] * world
    value = tokens / (ms / 1e3)

    # roofline of the dominant launch unit: the gdn_chunk_fwd call (chunk map + the fused chunk
    # preparation / serial pass kernel for this few-unit workload; inseparable behind the C ABI),
    # timed live with CUDA events around the call
    th = pf["total_T"] * pf["H"]
    flops = th * prefill_flops_per_token_head(pf["d"])
    byts = prefill_bytes(pf["total_T"], pf["H"], pf["d"], pf["num_seqs"])
    k_s = pf["kernel_ms"] / 1e3
    tr = traffic_record("gdn_chunk_fwd[prefill]")
    roof = {"bound": "hbm", "achieved": byts / k_s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": byts / k_s / 1e9 / peaks["hbm_gbs"], "traffic": tr,
            "kernel": ("gdn_chunk_fwd (chunk_map_kernel + chunk_fused_kernel: chunk preparation and serial "
                       "pass in one cooperative launch)"),
            "algorithmic_bytes": byts, "algorithmic_flops": flops,
            "tensor_tflops": flops / k_s / 1e12,
            "tensor_pipe_pct_ncu": tensor_pipe_record("gdn_chunk_fwd[prefill]"),
            "tensor_frac": flops / k_s / 1e12 / peaks["bf16_tflops"],
            "peak_source": f"{peak_src} hbm_gbs; tensor_frac of {peak_src} bf16_tflops (burst)",
            "note": "arithmetic intensity 116 FLOP/B is below the bf16 ridge, so HBM is the bound; "
                    "the 64-step serial chunk chain per (sequence, head) is what limits it in practice"}
    dbytes = decode_bytes(dc["N"], dc["H"], dc["d"])
    d_gbs = dbytes / (dc["kernel_ms"] / 1e3) / 1e9
    decode = {"metric": "decode tokens/s", "value": dc["N"] * world / (dms / 1e3), "unit": "tokens/s",
              "ms_per_step": dms, "kernel_ms": dc["kernel_ms"],
              "config": {"workload": "decode", "N": dc["N"], "H": dc["H"], "d_k": dc["d"], "d_v": dc["d"],
                         "state": "fp32", "qkv": "bf16"},
              "roofline": {"bound": "hbm", "achieved": d_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": d_gbs / peaks["hbm_gbs"], "traffic": traffic_record("decode_kernel[decode]"),
                           "kernel": "decode_kernel", "algorithmic_bytes": dbytes,
                           "peak_source": f"{peak_src} hbm_gbs"},
              "multi_token": {"tokens_per_s": dc["N"] * dc["multi_T"] * world / (dc["multi_ms"] / 1e3),
                              "ms": dc["multi_ms"], "T": dc["multi_T"], "pool_slots": dc["multi_slots"],
                              "entry_point": "gdn_recurrent_multi_step", "kernel": "decode_stream_kernel",
                              "traffic": traffic_record("decode_stream_kernel[multi_token]"),
                              "hbm_gbs": dc["multi_bytes"] / (dc["multi_ms"] / 1e3) / 1e9,
                              "frac": dc["multi_bytes"] / (dc["multi_ms"] / 1e3) / 1e9 / peaks["hbm_gbs"]}}
    line = {
        "metric": "prefill tokens/s", "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "prefill", "num_seqs": pf["num_seqs"], "seq_len": pf["total_T"] // pf["num_seqs"],
                   "H": pf["H"], "d_k": pf["d"], "d_v": pf["d"], "chunk": C_CHUNK, "gate": "rmsnorm_silu",
                   "step": "gdn_decay_from_logits + gdn_chunk_fwd", "l2": "flushed (512 MB write) before each step",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "decode": decode,
        "variants": variants,
        "workloads": workloads,
        "e2e": {"value": tokens / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": pf["h2d"],
                "d2h_bytes_per_step": pf["d2h"], "ms_per_step": e2e_ms},
        "gpu_launches": pf["launches"],
        "clocks": pf["clocks"],
        "peaks": {"source": peak_src, "hbm_gbs": peaks.get("hbm_gbs"), "bf16_tflops": peaks.get("bf16_tflops")},
    }
    if args.rank == 0 and not args.no_cpu_baseline:
        rate, th, sample, _ = oracle_rate(pf["inp"], pf["H"], seconds_budget=args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": th, "kind": "oracle",
                                "sample": sample, "single_thread_value": oracle_rate.single_thread,
                                "host_cores": os.cpu_count()}
    if args.rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args):
    if args.rank != 0:
        return
    from gated_deltanet_recurrence_gb300 import synthetic
    inp = synthetic.prefill_inputs("prefill")
    cfg = inp["cfg"]
    rates = []
    for _ in range(args.warmup):
        oracle_rate(inp, cfg["H"], seconds_budget=3.0)
    last = None
    for _ in range(args.steps):
        last = oracle_rate(inp, cfg["H"], seconds_budget=3.0)
        rates.append(last[0])
    value = statistics.mean(rates)
    line = {"impl": "reference", "metric": "prefill tokens/s", "value": value, "unit": "tokens/s",
            "n_gpus": args.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": inp["total_T"] / value * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "prefill", "num_seqs": inp["num_seqs"],
                       "seq_len": inp["total_T"] // inp["num_seqs"], "H": cfg["H"], "d_k": cfg["d"],
                       "d_v": cfg["d"], "gate": "rmsnorm_silu"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": last[1], "kind": "oracle",
                             "sample": last[2]},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    ap.add_argument("--cpu-seconds", type=float, default=20.0, help="budget of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the grouped-head / per-channel-decay / convolution measurements")
    ap.add_argument("--only", choices=["all", "prefill", "decode"], default="all",
                    help="time only one workload (profiling runs); the driver uses the default")
    ap.add_argument("--workloads", default="",
                    help="comma list of prefill workloads to time alone instead (tiny, varlen, long)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the tiny / varlen / long workload lines of the default run")
    ap.add_argument("--prefill-form", choices=["auto", "fused", "two-kernel"], default="auto",
                    help="force one prefill kernel form (profiling runs); the driver uses the default")
    args = ap.parse_args()
    if args.warmup < 3:
        print("note: warm-up raised to 3 steps", file=sys.stderr)
        args.warmup = 3
    args.world, args.rank, args.local = dist_setup(args)
    try:
        if args.impl == "reference":
            run_reference(args)
        else:
            run_gdn(args)
    finally:
        if args.world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
