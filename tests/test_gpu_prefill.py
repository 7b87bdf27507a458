"""GPU parity of the chunked prefill (gdn_chunk_fwd through the C ABI) against the fp64 oracle.

Full-size workloads are compared element by element where the oracle finishes in seconds (tiny,
prefill) and on sampled (sequence, head) slabs otherwise (varlen, long), always in the launch
configuration the benchmark times.  The edge cases cover empty and ragged sequences, both head
sizes, no normalisation, weights, aliasing of the initial and final state, resuming from a
returned state, and a malformed cu_seqlens reported through the device error word."""
import numpy as np
import pytest
import torch

import gated_deltanet_recurrence_gb300 as gdn
import oracle
from gated_deltanet_recurrence_gb300 import synthetic
from tests._util import (TOL_BF16, TOL_F32, cu_list, oracle_gates, oracle_prefill, rel_l2_states,
                         rel_l2_tokens)

pytestmark = pytest.mark.gpu


def run_gpu(inp, g32, b32, out_dtype=None, weight=None, use_l2=True, scale=0.0, gate=True,
            initial_state="inp", final_state=None):
    dev = "cuda"
    S0 = inp["initial_state"] if isinstance(initial_state, str) else initial_state
    out, Sf = gdn.gdn_chunk_fwd(
        inp["q"].to(dev), inp["k"].to(dev), inp["v"].to(dev), g32.to(dev), b32.to(dev),
        cu_seqlens=inp["cu_seqlens"].to(dev) if inp["cu_seqlens"] is not None else None,
        num_seqs=inp["num_seqs"], scale=scale, use_qk_l2norm=use_l2,
        initial_state=S0.to(dev) if S0 is not None else None, final_state=final_state,
        gate_z=inp["z"].to(dev) if (gate and inp["z"] is not None) else None,
        norm_weight=weight.to(dev) if weight is not None else None, out_dtype=out_dtype)
    assert gdn.gdn_get_device_error() == 0
    return out.float().cpu(), Sf.cpu()


def check(inp, tol, **kw):
    g32, b32 = oracle_gates(inp)
    out, Sf = run_gpu(inp, g32, b32, **kw)
    y_ref, S_ref = oracle_prefill(inp, g32, b32, scale=None if kw.get("scale", 0) <= 0 else kw["scale"],
                                  use_l2=kw.get("use_l2", True), gate=kw.get("gate", True),
                                  weight=kw.get("weight"))
    cu = cu_list(inp)
    e_o, e_s = rel_l2_tokens(out, y_ref, cu), rel_l2_states(Sf, S_ref)
    assert e_o <= tol and e_s <= tol, (e_o, e_s)
    return e_o, e_s


def test_tiny_fp32_full():
    """tiny workload (B=1, H=2, T=256, d=64, fp32): relative L2 <= 1e-4."""
    e = check(synthetic.prefill_inputs("tiny"), TOL_F32, out_dtype=torch.float32)
    print("tiny", e)


def test_prefill_bf16_full():
    """prefill workload (B=2, H=16, T=4096, d=128, bf16, fused gate): relative L2 <= 1e-2."""
    e = check(synthetic.prefill_inputs("prefill"), TOL_BF16)
    print("prefill", e)


def test_prefill_bf16_raw_y_fp32_out():
    inp = synthetic.prefill_inputs(synthetic.workload("prefill", T=1000, seed=21))
    check(inp, TOL_BF16, out_dtype=torch.float32, gate=False)


def test_varlen_sampled_sequences():
    """varlen workload (64 packed sequences, ~262K tokens, H=16, initial states): the GPU runs the
    whole batch; the oracle checks 6 sequences (the shortest, the longest and 4 more) on all heads
    and every final state's shape; raw y output."""
    inp = synthetic.prefill_inputs("varlen")
    g32, b32 = oracle_gates(inp)
    out, Sf = run_gpu(inp, g32, b32, out_dtype=torch.float32)
    L = inp["lengths"]
    seqs = sorted({int(np.argmin(L)), int(np.argmax(L)), 0, 17, 40, 63})
    y_ref, S_ref = oracle_prefill(inp, g32, b32, seqs=seqs)
    cu = cu_list(inp)
    y = torch.cat([out[cu[n]:cu[n + 1]] for n in seqs])
    cu_s = np.concatenate([[0], np.cumsum([L[n] for n in seqs])])
    assert rel_l2_tokens(y, y_ref, cu_s) <= TOL_BF16
    assert rel_l2_states(Sf[seqs], S_ref) <= TOL_BF16


def test_long_sampled_heads():
    """long workload (B=1, H=32, T=131072, alpha close to 1, fused gate): the GPU runs all 32
    heads; the oracle checks 3 heads over the whole sequence."""
    inp = synthetic.prefill_inputs("long", device="cpu")
    g32, b32 = oracle_gates(inp)
    out, Sf = run_gpu(inp, g32, b32)
    heads = [0, 13, 31]
    y_ref, S_ref = oracle_prefill(inp, g32, b32, heads=heads, threads=3)
    cu = cu_list(inp)
    assert rel_l2_tokens(out[:, heads], y_ref, cu) <= TOL_BF16
    assert rel_l2_states(Sf[:, heads], S_ref) <= TOL_BF16


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ragged_and_empty_sequences(d, dtype):
    lengths = [0, 1, 63, 64, 65, 200, 128, 3]
    cfg = synthetic.workload("varlen", lengths=lengths, num_seqs=len(lengths), H=3, d=d, dtype=dtype,
                             seed=31, gate=True)
    inp = synthetic.prefill_inputs(cfg)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    w = torch.linspace(0.25, 2.0, d)
    check(inp, tol, out_dtype=torch.float32, weight=w)


def test_no_l2norm_and_explicit_scale():
    cfg = synthetic.workload("varlen", lengths=[130, 77], num_seqs=2, H=2, d=128, dtype=torch.float32,
                             seed=32)
    inp = synthetic.prefill_inputs(cfg)
    # unnormalised keys make the recurrence unstable unless they are small: shrink them
    inp["k"] = inp["k"] * 0.08
    inp["q"] = inp["q"] * 0.08
    check(inp, TOL_F32, out_dtype=torch.float32, use_l2=False, scale=0.7)


def test_final_state_may_alias_initial_state():
    cfg = synthetic.workload("varlen", lengths=[100, 64, 0, 7], num_seqs=4, H=2, d=128,
                             dtype=torch.bfloat16, seed=33)
    inp = synthetic.prefill_inputs(cfg)
    g32, b32 = oracle_gates(inp)
    S = inp["initial_state"].cuda()
    out, _ = gdn.gdn_chunk_fwd(inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda(), g32.cuda(),
                               b32.cuda(), cu_seqlens=inp["cu_seqlens"].cuda(), initial_state=S,
                               final_state=S, out_dtype=torch.float32)
    y_ref, S_ref = oracle_prefill(inp, g32, b32)
    assert rel_l2_tokens(out.cpu(), y_ref, cu_list(inp)) <= TOL_BF16
    assert rel_l2_states(S.cpu(), S_ref) <= TOL_BF16
    # the empty sequence keeps its initial state exactly
    assert torch.equal(S[2].cpu(), inp["initial_state"][2])


def test_resume_from_returned_state_and_continue_with_decode():
    """prefill(T1) -> state -> prefill(T2) equals prefill(T1 + T2); then one decode step on the
    returned state equals the oracle's next token."""
    cfg = synthetic.workload("prefill", num_seqs=1, T=301, H=4, seed=34, gate=False)
    inp = synthetic.prefill_inputs(cfg)
    g32, b32 = oracle_gates(inp)
    dev = "cuda"
    T1 = 130
    args = [t.to(dev) for t in (inp["q"], inp["k"], inp["v"], g32, b32)]
    y1, S1 = gdn.gdn_chunk_fwd(*[t[:T1] for t in args], out_dtype=torch.float32)
    y2, S2 = gdn.gdn_chunk_fwd(*[t[T1:300] for t in args], initial_state=S1, out_dtype=torch.float32)
    y_ref, S_ref = oracle.recurrence(inp["q"][:300], inp["k"][:300], inp["v"][:300], g32[:300],
                                     b32[:300])
    y = torch.cat([y1, y2]).cpu()
    assert rel_l2_tokens(y, y_ref, [0, 300]) <= TOL_BF16
    assert rel_l2_states(S2.cpu(), S_ref) <= TOL_BF16
    yd = gdn.gdn_recurrent_step(*[t[300:301] for t in args], S2, out_dtype=torch.float32)
    y_all, S_all = oracle.recurrence(inp["q"], inp["k"], inp["v"], g32, b32)
    np.testing.assert_allclose(yd.cpu().double().numpy()[0], y_all[300], rtol=2e-2, atol=2e-3)
    assert rel_l2_states(S2.cpu(), S_all) <= TOL_BF16


def test_malformed_cu_seqlens_reported_on_device():
    """A cu_seqlens that decreases is caught by the kernel, which then writes nothing for that
    sequence; gdn_get_device_error returns GDN_ERR_CU_SEQLENS once and clears the word."""
    T, H, d = 128, 2, 64
    x = torch.randn(T, H, d, device="cuda")
    g = torch.zeros(T, H, device="cuda")
    cu = torch.tensor([0, 100, 50, 128], dtype=torch.int32, device="cuda")
    out = torch.full((T, H, d), 7.0, device="cuda")
    gdn.gdn_chunk_fwd(x, x, x, g, g, cu_seqlens=cu, out=out)
    assert gdn.gdn_get_device_error() == -3
    assert gdn.gdn_get_device_error() == 0
    cu_bad = torch.tensor([0, 64, 4096], dtype=torch.int32, device="cuda")   # past total_T
    gdn.gdn_chunk_fwd(x, x, x, g, g, cu_seqlens=cu_bad, out=out)
    assert gdn.gdn_get_device_error() == -3


def test_gated_output_matches_standalone_gate():
    """The fused gate epilogue equals the raw output passed through gdn_gate_rmsnorm_silu.  With an
    fp32 output both evaluate the norm and SiLU in fp32 ("5. 线性注意力", 门控 RMSNorm), so they
    agree to fp32 rounding; with a bf16 output the fused epilogue's packed half-precision SiLU
    (relative error near 1e-3) stays below the output's own 2^-9 rounding."""
    inp = synthetic.prefill_inputs(synthetic.workload("prefill", T=200, H=4, seed=35))
    g32, b32 = oracle_gates(inp)
    o_fused, _ = run_gpu(inp, g32, b32, out_dtype=torch.float32)
    y_raw, _ = run_gpu(inp, g32, b32, out_dtype=torch.float32, gate=False)
    o_sep = gdn.gdn_gate_rmsnorm_silu(y_raw.cuda(), inp["z"].cuda(), out_dtype=torch.float32).cpu()
    assert rel_l2_tokens(o_fused, o_sep, cu_list(inp)) <= 1e-5
    o_bf16, _ = run_gpu(inp, g32, b32, out_dtype=torch.bfloat16)
    assert rel_l2_tokens(o_bf16.float(), o_sep, cu_list(inp)) <= 4e-3


def test_gate_prep_then_prefill_end_to_end():
    """The full path from logits: gdn_decay_from_logits on the GPU, then gdn_chunk_fwd, against the
    oracle's fp64 gate preparation and recurrence."""
    inp = synthetic.prefill_inputs(synthetic.workload("prefill", T=512, H=4, seed=36))
    dev = "cuda"
    g, beta = gdn.gdn_decay_from_logits(inp["a"].to(dev), inp["A_log"].to(dev), b=inp["b"].to(dev))
    out, Sf = gdn.gdn_chunk_fwd(inp["q"].to(dev), inp["k"].to(dev), inp["v"].to(dev), g, beta,
                                num_seqs=2, gate_z=inp["z"].to(dev))
    g64, b64 = oracle.gates_from_logits(inp["a"], inp["A_log"], b=inp["b"])
    y_ref, S_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g64, b64, batch=2)
    o_ref = oracle.gate_rmsnorm_silu(y_ref, inp["z"])
    assert rel_l2_tokens(out.float().cpu(), o_ref, [0, 512, 1024]) <= TOL_BF16
    assert rel_l2_states(Sf.cpu(), S_ref) <= TOL_BF16


@pytest.mark.parametrize("name,kw", [("prefill", {}), ("prefill_kda", {}), ("prefill_conv", {}),
                                     ("varlen", dict(lengths=[300, 64, 0, 1000, 65], num_seqs=5, H=4))])
def test_fused_and_two_kernel_paths_agree_bitwise(name, kw, kernel_forms):
    """Few (sequence, head) units run the fused cooperative kernel (preparation and serial pass at
    once; with few pairs in the export form, whose outputs other CTAs form);
    gdn_set_kernel_forms(GDN_FORM_OFF) selects the two-kernel path.  All run the same arithmetic in
    the same order, so outputs and final states must be identical bit for bit."""
    cfg = synthetic.workload(name if name != "varlen" else "varlen", **kw) if kw else synthetic.workload(name)
    inp = synthetic.prefill_inputs(cfg)
    g32, b32 = oracle_gates(inp)
    dev = "cuda"
    args = [inp[x].to(dev) for x in ("q", "k", "v")] + [g32.to(dev), b32.to(dev)]
    kwargs = dict(cu_seqlens=inp["cu_seqlens"].to(dev) if inp["cu_seqlens"] is not None else None,
                  num_seqs=inp["num_seqs"],
                  initial_state=inp["initial_state"].to(dev) if inp["initial_state"] is not None else None,
                  conv_weight=inp["conv_weight"].to(dev) if inp.get("conv_weight") is not None else None,
                  gate_z=inp["z"].to(dev) if inp["z"] is not None else None)
    outs = {}
    # AUTO: fused (in the export form where it applies: decay per head, no convolution, few pairs);
    # ON: fused whenever the pairs number fewer than the SMs; OFF: two kernels
    for mode, form in (("1", gdn.GDN_FORM_AUTO), ("2", gdn.GDN_FORM_ON), ("0", gdn.GDN_FORM_OFF)):
        gdn.gdn_set_kernel_forms(prefill_fused=form)
        out, Sf = gdn.gdn_chunk_fwd(*args, **kwargs)
        assert gdn.gdn_get_device_error() == 0
        outs[mode] = (out.cpu(), Sf.cpu())
    assert torch.equal(outs["2"][0], outs["0"][0])
    assert torch.equal(outs["2"][1], outs["0"][1])
    assert torch.equal(outs["1"][0], outs["0"][0])
    assert torch.equal(outs["1"][1], outs["0"][1])
