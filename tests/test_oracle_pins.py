"""Pins of the fp64 oracle against facts the pages and the mathematics fix.

None of these re-types the oracle's own formula: each expected value comes from a
printed worked example (tests/golden), a closed form of a special case, an
invariant stated on the pages, a library routine, or a second formulation that
reaches the same result by different algebra.  The mutation tests at the end plant
plausible mistakes in a copy of the oracle's C source and check that some pin
catches each of them.
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = np.array([float(x) for x in rest])
    return vals


def _rand_inputs(rng, T, H, dk, dv, n_seqs=1, g_scale=1.0):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    g = -g_scale * rng.random((T, H))
    beta = rng.random((T, H))
    return q, k, v, g, beta


# --------------------------------------------------------------------------------------
# printed worked examples
# --------------------------------------------------------------------------------------

def test_worked_example_g0_all_forms():
    """'5. 线性注意力', 一个简单例子: K = V = I, beta = 1, g = 0 gives o = I (unscaled)."""
    gd = _read_golden("chunk_worked_example_g0.txt")
    d, T = int(gd["d"][0]), int(gd["T"][0])
    k = gd["k"].reshape(T, 1, d)
    v = gd["v"].reshape(T, 1, d)
    q = gd["q"].reshape(T, 1, d)
    g = gd["g"].reshape(T, 1)
    beta = gd["beta"].reshape(T, 1)
    for fn in (oracle.recurrence,
               lambda *a, **kw: oracle.chunked(*a, C=int(gd["C"][0]), **kw),
               oracle.transition_product):
        y1, S = fn(q, k, v, g, beta, scale=1.0, use_qk_l2norm=False)
        np.testing.assert_allclose(y1.reshape(-1), gd["o_unscaled"], atol=1e-15)
        np.testing.assert_allclose(S.reshape(-1), gd["S_final"], atol=1e-15)
        ys, _ = fn(q, k, v, g, beta, use_qk_l2norm=False)  # default scale 1/sqrt(d)
        np.testing.assert_allclose(ys.reshape(-1), gd["o_scaled"], atol=1e-15)
        # with the in-kernel normalisation the unit rows shrink by 1/sqrt(1 + 1e-6)
        yl, _ = fn(q, k, v, g, beta, use_qk_l2norm=True)
        np.testing.assert_allclose(yl.reshape(-1), gd["o_scaled"], atol=2e-6)


def test_decay_matrix_example():
    """'5. 线性注意力', 阶段 1 numeric example, C = 4."""
    gd = _read_golden("chunk_decay_example.txt")
    gcum, decay = oracle.chunk_decay(gd["g"])
    np.testing.assert_allclose(gcum, gd["gcum"], atol=1e-15)
    np.testing.assert_allclose(decay.reshape(-1), gd["decay"], atol=1e-15)


def test_gated_unit_key_example():
    gd = _read_golden("gated_unit_key_example.txt")
    d, T = int(gd["d"][0]), int(gd["T"][0])
    k = gd["k"].reshape(T, 1, d)
    for fn in (oracle.recurrence, lambda *a, **kw: oracle.chunked(*a, C=2, **kw),
               lambda *a, **kw: oracle.chunked(*a, C=4, **kw), oracle.transition_product):
        y, _ = fn(k, k, gd["v"].reshape(T, 1, d), gd["g"].reshape(T, 1), gd["beta"].reshape(T, 1),
                  use_qk_l2norm=False)
        np.testing.assert_allclose(y.reshape(-1), gd["o_scaled"], atol=1e-15)


# --------------------------------------------------------------------------------------
# invariants and closed forms
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("form", ["recurrence", "chunked16", "chunked64"])
def test_unit_key_full_write_invariant(form):
    """'[LLM Algorithms-2] Gated DeltaNet' 2.2: ||k|| = 1, beta = 1  =>  S_t k_t = v_t,
    whatever the decay and the earlier tokens; with q = k this is y_t = scale * v_t."""
    rng = np.random.default_rng(1)
    T, H, dk, dv = 100, 2, 16, 12
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv, g_scale=0.5)
    beta[:] = 1.0
    S0 = rng.standard_normal((1, H, dv, dk))
    fn = oracle.recurrence if form == "recurrence" else \
        (lambda *a, **kw: oracle.chunked(*a, C=int(form[7:]), **kw))
    y, S = fn(k, k, v, g, beta, scale=0.37, initial_state=S0)
    kn = k / np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)
    # y_t = S_t (0.37 k_t) = 0.37 * ||k_t||^2 ... only the unit-norm direction matters:
    # S_t kn_t = v_t exactly when ||kn_t|| = 1; kn_t has norm sqrt(s/(s+eps)) so allow 1e-6
    np.testing.assert_allclose(y, 0.37 * v, rtol=0, atol=1e-5)
    np.testing.assert_allclose(np.einsum("hrc,hc->hr", S[0], kn[-1]), v[-1], atol=1e-5)


def test_beta_zero_is_pure_decay():
    """beta = 0: the write vanishes ('[LLM Algorithms-2]' 2.2, I - 0 k k^T = I), so
    S_t = alpha_t S_{t-1} and y_t = (prod_{s<=t} alpha_s) S_0 q_t."""
    rng = np.random.default_rng(2)
    T, H, dk, dv = 70, 3, 8, 6
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv)
    beta[:] = 0.0
    S0 = rng.standard_normal((1, H, dv, dk))
    for fn in (oracle.recurrence, lambda *a, **kw: oracle.chunked(*a, C=16, **kw)):
        y, S = fn(q, k, v, g, beta, scale=1.0, use_qk_l2norm=False, initial_state=S0)
        decay = np.cumprod(np.exp(g), axis=0)  # [T, H], products of alphas
        expect = decay[:, :, None] * np.einsum("hrc,thc->thr", S0[0], q)
        np.testing.assert_allclose(y, expect, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(S[0], decay[-1][:, None, None] * S0[0], rtol=1e-12)


def test_alpha_one_beta_zero_leaves_state():
    rng = np.random.default_rng(3)
    T, H, dk, dv = 40, 1, 8, 8
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv)
    g[:] = 0.0
    beta[:] = 0.0
    S0 = rng.standard_normal((1, H, dv, dk))
    _, S = oracle.recurrence(q, k, v, g, beta, initial_state=S0)
    np.testing.assert_array_equal(S, S0)


@pytest.mark.parametrize("form", ["recurrence", "chunked4", "chunked64", "transition"])
def test_orthogonal_keys_reduce_to_gated_linear_attention(form):
    """With orthonormal keys the prediction S_{t-1} k_t is zero, so the delta rule writes
    beta_t v_t k_t^T and y = ((Q K^T) * D) diag(beta) V with D_ij = alpha_{j+1}...alpha_i
    (j <= i): masked matrix products, computed here with numpy from cumulative products of
    alpha rather than sums of logs.  dk != dv catches transposed operands."""
    rng = np.random.default_rng(4)
    T, dk, dv = 12, 16, 5
    Kfull, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Kfull[:T].reshape(T, 1, dk)              # orthonormal rows
    q = rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    g = -rng.random((T, 1))
    beta = rng.random((T, 1))
    # an initial state that every key annihilates: rows in the orthogonal complement
    comp = Kfull[T:]                              # (dk - T) x dk
    S0 = (rng.standard_normal((dv, dk - T)) @ comp).reshape(1, 1, dv, dk)
    alpha = np.exp(g[:, 0])
    D = np.zeros((T, T))
    for i in range(T):
        for j in range(i + 1):
            D[i, j] = np.prod(alpha[j + 1:i + 1])
    scale = 0.5
    Q, K, V = q[:, 0], k[:, 0], v[:, 0]
    expect = scale * (((Q @ K.T) * D) @ (beta[:, 0:1] * V))
    expect += scale * np.cumprod(alpha)[:, None] * (Q @ S0[0, 0].T)
    expect_S = np.prod(alpha) * S0[0, 0] + sum(
        np.prod(alpha[j + 1:]) * beta[j, 0] * np.outer(V[j], K[j]) for j in range(T))
    if form == "recurrence":
        fn = oracle.recurrence
    elif form == "transition":
        fn = oracle.transition_product
    else:
        fn = lambda *a, **kw: oracle.chunked(*a, C=int(form[7:]), **kw)  # noqa: E731
    y, S = fn(q, k, v, g, beta, scale=scale, use_qk_l2norm=False, initial_state=S0)
    np.testing.assert_allclose(y[:, 0], expect, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S[0, 0], expect_S, rtol=1e-12, atol=1e-13)


def test_erase_write_form_and_gated_linear_reference():
    """'[LLM Algorithms-2]' 4 second box: S_t = alpha_t S_{t-1}(I - beta_t k k^T) + beta_t v k^T,
    written with explicit dk x dk matrices (a different expansion from the oracle's
    decay / predict / write steps)."""
    rng = np.random.default_rng(5)
    T, H, dk, dv = 30, 2, 7, 4
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv)
    S0 = rng.standard_normal((1, H, dv, dk))
    y, S = oracle.recurrence(q, k, v, g, beta, scale=1.0, use_qk_l2norm=False, initial_state=S0)
    for h in range(H):
        St = S0[0, h].copy()
        for t in range(T):
            kt = k[t, h]
            St = math.exp(g[t, h]) * St @ (np.eye(dk) - beta[t, h] * np.outer(kt, kt)) \
                + beta[t, h] * np.outer(v[t, h], kt)
            np.testing.assert_allclose(y[t, h], St @ q[t, h], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(S[0, h], St, rtol=1e-11, atol=1e-12)


def test_geometry_of_erase_matrix():
    """'[LLM Algorithms-2]' 2.2: for unit k, (I - beta k k^T) scales the k direction by 1 - beta
    and leaves the orthogonal directions alone.  Checked through one oracle step with alpha = 1
    and v = 0 (then S_1 = S_0 (I - beta k k^T))."""
    rng = np.random.default_rng(6)
    dk, dv = 9, 3
    kk = rng.standard_normal(dk)
    kk /= np.linalg.norm(kk)
    w = rng.standard_normal(dk)
    w -= (w @ kk) * kk
    S0 = rng.standard_normal((1, 1, dv, dk))
    beta = 0.3
    _, S1 = oracle.recurrence(np.zeros((1, 1, dk)), kk.reshape(1, 1, dk), np.zeros((1, 1, dv)),
                              np.zeros((1, 1)), np.full((1, 1), beta), use_qk_l2norm=False,
                              initial_state=S0)
    np.testing.assert_allclose(S1[0, 0] @ kk, (1 - beta) * (S0[0, 0] @ kk), atol=1e-14)
    np.testing.assert_allclose(S1[0, 0] @ w, S0[0, 0] @ w, atol=1e-14)


# --------------------------------------------------------------------------------------
# formulations agree (brute force on tiny inputs)
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 130])
@pytest.mark.parametrize("C", [2, 4, 16, 64])
def test_chunked_equals_recurrence(T, C):
    """'[LLM Algorithms-2]' 7: the chunked and the recurrent paths must agree; in fp64 they do to
    rounding, including a ragged last chunk, a non-zero initial state and dk != dv."""
    rng = np.random.default_rng(100 + T * 7 + C)
    H, dk, dv = 2, 12, 10
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv, g_scale=2.0)
    S0 = rng.standard_normal((1, H, dv, dk))
    for l2 in (True, False):
        y0, S0f = oracle.recurrence(q, k, v, g, beta, use_qk_l2norm=l2, initial_state=S0)
        y1, S1f = oracle.chunked(q, k, v, g, beta, C=C, use_qk_l2norm=l2, initial_state=S0)
        np.testing.assert_allclose(y1, y0, rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(S1f, S0f, rtol=1e-11, atol=1e-11)


def test_transition_product_equals_recurrence():
    rng = np.random.default_rng(7)
    T, H, dk, dv = 11, 2, 6, 5
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv)
    S0 = rng.standard_normal((1, H, dv, dk))
    y0, Sa = oracle.recurrence(q, k, v, g, beta, initial_state=S0)
    y1, Sb = oracle.transition_product(q, k, v, g, beta, initial_state=S0)
    np.testing.assert_allclose(y1, y0, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(Sb, Sa, rtol=1e-12, atol=1e-13)


def test_varlen_equals_separate_sequences():
    """Packed sequences are independent: running them packed (cu_seqlens, one of them empty)
    equals running each alone; an empty sequence returns its initial state."""
    rng = np.random.default_rng(8)
    lens = [5, 0, 64, 70, 1]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, H, dk, dv = int(cu[-1]), 2, 8, 8
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv)
    S0 = rng.standard_normal((len(lens), H, dv, dk))
    y, S = oracle.recurrence(q, k, v, g, beta, cu_seqlens=cu, initial_state=S0, threads=3)
    yc, Sc = oracle.chunked(q, k, v, g, beta, C=16, cu_seqlens=cu, initial_state=S0, threads=2)
    np.testing.assert_allclose(yc, y, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(Sc, S, rtol=1e-11, atol=1e-12)
    for n, L in enumerate(lens):
        a, b = cu[n], cu[n + 1]
        yn, Sn = oracle.recurrence(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b],
                                   initial_state=S0[n:n + 1])
        np.testing.assert_array_equal(y[a:b], yn)
        np.testing.assert_array_equal(S[n], Sn[0])
    np.testing.assert_array_equal(S[1], S0[1])


def test_prefill_split_equals_whole():
    """The final state resumes a sequence: prefill(T1) -> state -> prefill(T2) = prefill(T1+T2)."""
    rng = np.random.default_rng(9)
    T, H, dk, dv = 90, 2, 8, 8
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv)
    y, S = oracle.chunked(q, k, v, g, beta, C=16)
    ya, Sa = oracle.chunked(q[:37], k[:37], v[:37], g[:37], beta[:37], C=16)
    yb, Sb = oracle.chunked(q[37:], k[37:], v[37:], g[37:], beta[37:], C=16, initial_state=Sa)
    np.testing.assert_allclose(np.concatenate([ya, yb]), y, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(Sb, S, rtol=1e-11, atol=1e-12)


def test_recurrent_step_continues_prefill():
    """'6.6 Gated DeltaNet' 6.6.8: decoding token by token on the kept state gives the same
    outputs as the whole sequence."""
    rng = np.random.default_rng(10)
    T, H, dk, dv = 9, 3, 8, 6
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv)
    y, S = oracle.recurrence(q, k, v, g, beta)
    st = np.zeros((1, H, dv, dk))
    for t in range(T):
        yt, st = oracle.recurrent_step(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1],
                                       beta[t:t + 1], st)
        np.testing.assert_allclose(yt[0], y[t], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(st, S, rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------------------------------
# output gate and gate preparation
# --------------------------------------------------------------------------------------

def test_gate_rmsnorm_silu_special_cases_and_library():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    rows, dv = 7, 16
    # constant rows: y = c * 1 gives RMSNorm(y) = sign(c) / sqrt(1 + eps / c^2)
    c = np.array([2.0, -0.5, 3e-3, -7.0, 1.0, 0.25, -1.0])
    y = np.repeat(c[:, None], dv, axis=1)
    z = rng.standard_normal((rows, dv))
    out = oracle.gate_rmsnorm_silu(y, z, eps=1e-6)
    silu = z / (1 + np.exp(-z))
    expect = (np.sign(c) / np.sqrt(1 + 1e-6 / c ** 2))[:, None] * silu
    np.testing.assert_allclose(out, expect, rtol=1e-14, atol=0)
    # z = 0 closes the gate
    np.testing.assert_array_equal(oracle.gate_rmsnorm_silu(y, np.zeros_like(z)), 0.0 * y)
    # random rows with a weight against torch's rms_norm and silu in float64
    y = rng.standard_normal((rows, dv))
    w = rng.standard_normal(dv)
    ty, tz, tw = (torch.from_numpy(a) for a in (y, z, w))
    ref = torch.nn.functional.rms_norm(ty, (dv,), weight=tw, eps=1e-6) * torch.nn.functional.silu(tz)
    np.testing.assert_allclose(oracle.gate_rmsnorm_silu(y, z, w, eps=1e-6), ref.numpy(),
                               rtol=1e-13, atol=1e-15)


def test_gates_from_logits():
    """'6.6 Gated DeltaNet' 6.6.3: alpha = exp(-A softplus(a + dt_bias)), beta = sigmoid(b);
    checked against numpy's logaddexp (softplus) and the limits of the formula."""
    rng = np.random.default_rng(12)
    T, H = 50, 4
    a = rng.normal(-1, 3, (T, H))
    a[0] = [-60.0, 0.0, 40.0, 800.0]
    b = rng.normal(0, 3, (T, H))
    A_log = rng.uniform(0, math.log(8), H)
    dt = rng.normal(0, 1, H)
    g, beta = oracle.gates_from_logits(a, A_log, dt_bias=dt, b=b)
    A = np.exp(A_log)
    np.testing.assert_allclose(g, -A * np.logaddexp(0.0, a + dt), rtol=1e-14)
    np.testing.assert_allclose(beta, 1 / (1 + np.exp(-b)), rtol=1e-14)
    g0 = oracle.gates_from_logits(a[:1], A_log)
    assert abs(g0[0, 0]) < 1e-20                             # softplus(-60) ~ e^-60
    np.testing.assert_allclose(g0[0, 1], -A[1] * math.log(2.0), rtol=1e-15)
    np.testing.assert_allclose(g0[0, 3], -A[3] * 800.0, rtol=1e-15)
    assert np.all(g <= 0) and np.all(np.exp(g) <= 1)       # alpha in (0, 1]


# --------------------------------------------------------------------------------------
# grouped query/key heads: "5. 线性注意力" forward code, repeat_interleave of q and k
# --------------------------------------------------------------------------------------

def test_grouped_heads_equal_interleaved_repeat():
    """With Hk query/key heads and H = r * Hk value heads, the page repeats each query/key head r
    times in place (repeat_interleave along the head axis) before the core; the grouped call must
    equal the core on those expanded inputs, for every form."""
    rng = np.random.default_rng(50)
    T, Hk, r, dk, dv = 21, 2, 3, 5, 4
    q = rng.standard_normal((T, Hk, dk))
    k = rng.standard_normal((T, Hk, dk))
    v = rng.standard_normal((T, Hk * r, dv))
    g = -rng.random((T, Hk * r))
    beta = rng.random((T, Hk * r))
    S0 = rng.standard_normal((1, Hk * r, dv, dk)) * 0.3
    qe, ke = np.repeat(q, r, axis=1), np.repeat(k, r, axis=1)   # numpy repeat == repeat_interleave
    for fn in (oracle.recurrence, lambda *a, **kw: oracle.chunked(*a, C=4, **kw),
               oracle.transition_product):
        y, S = fn(q, k, v, g, beta, initial_state=S0)
        ye, Se = fn(qe, ke, v, g, beta, initial_state=S0)
        np.testing.assert_allclose(y, ye, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(S, Se, rtol=1e-12, atol=1e-12)
    # the interleaved order matters: tiling the heads instead gives another result
    yt, _ = oracle.recurrence(np.tile(q, (1, r, 1)), np.tile(k, (1, r, 1)), v, g, beta, initial_state=S0)
    assert np.abs(yt - ye).max() > 1e-3


# --------------------------------------------------------------------------------------
# decay per key channel: "6.6 Gated DeltaNet" 6.6.7 (alpha_t a vector over channels)
# --------------------------------------------------------------------------------------

def _pc_inputs(rng, T, H, dk, dv):
    q, k, v, _, beta = _rand_inputs(rng, T, H, dk, dv)
    g = -rng.random((T, H, dk)) * 0.8
    return q, k, v, g, beta


def test_per_channel_equal_channels_is_scalar_decay():
    """A per-channel decay with every channel equal is the scalar decay of the head."""
    rng = np.random.default_rng(51)
    q, k, v, g, beta = _rand_inputs(rng, 19, 2, 6, 5)
    S0 = rng.standard_normal((1, 2, 5, 6)) * 0.2
    gpc = np.repeat(g[:, :, None], 6, axis=2)
    for fn in (oracle.recurrence, oracle.transition_product):
        y, S = fn(q, k, v, gpc, beta, initial_state=S0)
        ys, Ss = oracle.recurrence(q, k, v, g, beta, initial_state=S0)
        np.testing.assert_allclose(y, ys, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(S, Ss, rtol=1e-12, atol=1e-13)


def test_per_channel_beta_zero_closed_form():
    """beta = 0: nothing is written, so S_t = S_0 diag(prod_s alpha_s) and y_t = S_t q_t with the
    products taken channel by channel over the key axis."""
    rng = np.random.default_rng(52)
    T, H, dk, dv = 13, 2, 6, 5
    q, k, v, g, beta = _pc_inputs(rng, T, H, dk, dv)
    beta[:] = 0.0
    S0 = rng.standard_normal((1, H, dv, dk))
    y, S = oracle.recurrence(q, k, v, g, beta, initial_state=S0, use_qk_l2norm=False, scale=1.0)
    gsum = np.cumsum(g, axis=0)                      # [T, H, dk]
    for t in range(T):
        for h in range(H):
            St = S0[0, h] * np.exp(gsum[t, h])[None, :]
            np.testing.assert_allclose(y[t, h], St @ q[t, h], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S[0], S0[0] * np.exp(gsum[-1])[:, None, :], rtol=1e-12)


def test_per_channel_unit_key_invariant():
    """||k|| = 1, beta = 1: the write makes S_t k_t = v_t whatever the decay, so with q = k the
    output is scale * v_t exactly."""
    rng = np.random.default_rng(53)
    T, H, dk, dv = 17, 2, 8, 6
    _, k, v, g, beta = _pc_inputs(rng, T, H, dk, dv)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    beta[:] = 1.0
    S0 = rng.standard_normal((1, H, dv, dk))
    y, _ = oracle.recurrence(k, k, v, g, beta, initial_state=S0, use_qk_l2norm=False, scale=0.5)
    np.testing.assert_allclose(y, 0.5 * v, rtol=1e-10, atol=1e-12)


def test_per_channel_transition_equals_recurrence():
    """The unrolled product form with A_t = diag(alpha_t)(I - beta k k^T) built as explicit dense
    matrices equals the token loop."""
    rng = np.random.default_rng(54)
    q, k, v, g, beta = _pc_inputs(rng, 9, 2, 5, 4)
    S0 = rng.standard_normal((1, 2, 4, 5)) * 0.5
    y1, S1 = oracle.recurrence(q, k, v, g, beta, initial_state=S0)
    y2, S2 = oracle.transition_product(q, k, v, g, beta, initial_state=S0)
    np.testing.assert_allclose(y1, y2, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(S1, S2, rtol=1e-11, atol=1e-12)


def test_per_channel_decay_not_taken_by_chunked_form():
    rng = np.random.default_rng(55)
    q, k, v, g, beta = _pc_inputs(rng, 8, 1, 4, 4)
    with pytest.raises(ValueError):
        oracle.chunked(q, k, v, g, beta, C=4)


# --------------------------------------------------------------------------------------
# causal depthwise short convolution: "5. 线性注意力", "因果卷积(Causal Conv1d)"
# --------------------------------------------------------------------------------------

def _silu(x):
    return x / (1.0 + np.exp(-x))


def test_conv_identity_tap_is_silu():
    """A filter that keeps only the current token (tap K-1 = 1, the rest 0) gives SiLU(x)."""
    rng = np.random.default_rng(56)
    x = rng.standard_normal((11, 7))
    w = np.zeros((7, 4))
    w[:, 3] = 1.0
    y, st = oracle.short_conv(x, w)
    np.testing.assert_allclose(y, _silu(x), rtol=1e-15, atol=1e-16)
    y0, _ = oracle.short_conv(x, w, activation=False)
    np.testing.assert_array_equal(y0, x)


def test_conv_impulse_response():
    """The page's step-by-step picture: output t sees inputs t-3..t, the current one last, so a
    unit impulse at t = 0 reads the filter back in reverse, then zeros (SiLU(0) = 0)."""
    w = np.array([[0.5, -1.0, 2.0, 0.25]])
    x = np.zeros((7, 1))
    x[0, 0] = 1.0
    y, _ = oracle.short_conv(x, w)
    expect = _silu(np.array([0.25, 2.0, -1.0, 0.5, 0.0, 0.0, 0.0]))
    np.testing.assert_allclose(y[:, 0], expect, rtol=1e-15)


def test_conv_matches_library_conv1d():
    """One sequence from zero history equals the page's nn.Conv1d(groups=C, padding=K-1) cut back
    to T, followed by SiLU (torch.nn.functional on the CPU, float64)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(57)
    T, Cn, K = 23, 9, 4
    x = rng.standard_normal((T, Cn))
    w = rng.standard_normal((Cn, K))
    ref = torch.nn.functional.conv1d(torch.tensor(x.T[None]), torch.tensor(w[:, None, :]),
                                     padding=K - 1, groups=Cn)[0, :, :T]
    ref = torch.nn.functional.silu(ref).numpy().T
    y, _ = oracle.short_conv(x, w)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-14)


def test_conv_varlen_split_and_state():
    """Packed sequences do not see each other; the final state holds the last K-1 inputs, oldest
    first (for short sequences the older part comes from the initial state); a sequence split in
    two with the state carried across equals the whole."""
    rng = np.random.default_rng(58)
    Cn, K = 5, 4
    lens = [9, 2, 0, 6]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    x = rng.standard_normal((cu[-1], Cn))
    w = rng.standard_normal((Cn, K))
    s0 = rng.standard_normal((len(lens), Cn, K - 1))
    y, st = oracle.short_conv(x, w, cu_seqlens=cu, state=s0)
    for n, L in enumerate(lens):
        yn, stn = oracle.short_conv(x[cu[n]:cu[n + 1]], w, state=s0[n:n + 1])
        np.testing.assert_array_equal(y[cu[n]:cu[n + 1]], yn)
        hist = np.concatenate([s0[n].T, x[cu[n]:cu[n + 1]]])   # [K-1+L, Cn], oldest first
        np.testing.assert_array_equal(st[n], hist[-(K - 1):].T)
    xa = x[:9]
    ya, sa = oracle.short_conv(xa, w)
    y1, s1 = oracle.short_conv(xa[:4], w)
    y2, s2 = oracle.short_conv(xa[4:], w, state=s1)
    np.testing.assert_allclose(np.concatenate([y1, y2]), ya, rtol=1e-15)
    np.testing.assert_array_equal(s2, sa)


# --------------------------------------------------------------------------------------
# q/k normalisation and the query scale: "6.6 Gated DeltaNet" 6.6.4 (x / sqrt(sum x^2 + 1e-6),
# q scaled by 1/sqrt(d_k))
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("form", ["recurrence", "chunked4"])
def test_qk_normalisation_and_scale_closed_form(form):
    """One token from a zero state with beta = 1 and q = k = delta u (u a unit vector): the state is
    v k^T / sqrt(delta^2 + eps) and y = S q_hat = v * scale * delta^2 / (delta^2 + eps).  With
    delta^2 = eps the factor is exactly one half, which fixes where eps sits; with the
    normalisation off, y = v * scale * delta^2."""
    run = {"recurrence": oracle.recurrence,
           "chunked4": lambda *a, **kw: oracle.chunked(*a, C=4, **kw)}[form]
    rng = np.random.default_rng(21)
    dk, dv = 8, 5
    u = rng.standard_normal(dk)
    u /= np.linalg.norm(u)
    v = rng.standard_normal((1, 1, dv))
    g, beta = np.zeros((1, 1)), np.ones((1, 1))
    for delta2, scale in [(1e-6, None), (1e-6, 0.3), (4.0, None)]:
        x = (math.sqrt(delta2) * u)[None, None, :]
        y, _ = run(x, x, v, g, beta, batch=1, scale=scale)
        sc = 1 / math.sqrt(dk) if scale is None else scale
        np.testing.assert_allclose(y[0, 0], v[0, 0] * sc * delta2 / (delta2 + 1e-6), rtol=1e-12)
        y, _ = run(x, x, v, g, beta, batch=1, scale=scale, use_qk_l2norm=False)
        np.testing.assert_allclose(y[0, 0], v[0, 0] * sc * delta2, rtol=1e-12)


@pytest.mark.parametrize("form", ["recurrence", "chunked16"])
def test_output_invariant_to_raw_qk_scale(form):
    """With the normalisation on, multiplying the raw q or k of any token by a positive constant
    changes nothing beyond the eps term (relative ~eps / |x|^2)."""
    run = {"recurrence": oracle.recurrence,
           "chunked16": lambda *a, **kw: oracle.chunked(*a, C=16, **kw)}[form]
    rng = np.random.default_rng(22)
    T, H, dk, dv = 37, 2, 16, 8
    # raw norms around 40, so the eps term stays below 1e-8 relative even after scaling by 0.3
    q, k = 10 * rng.standard_normal((T, H, dk)), 10 * rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    g, beta = -rng.uniform(0, 1, (T, H)), rng.uniform(0, 1, (T, H))
    S0 = rng.standard_normal((1, H, dv, dk)) * 0.1
    y0, s0 = run(q, k, v, g, beta, batch=1, initial_state=S0)
    cq = rng.uniform(0.3, 5.0, (T, H, 1))
    ck = rng.uniform(0.3, 5.0, (T, H, 1))
    y1, s1 = run(q * cq, k * ck, v, g, beta, batch=1, initial_state=S0)
    np.testing.assert_allclose(y1, y0, rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(s1, s0, rtol=1e-6, atol=1e-9)


# --------------------------------------------------------------------------------------
# planted mistakes: each mutation of the oracle must be caught by a pin above
# --------------------------------------------------------------------------------------

MUTATIONS = {
    # delta read from the undecayed state (decay applied after the prediction)
    "undecayed_prediction": ("for (int j = 0; j < dk; ++j) pred += S[(long)r * dk + j] * kn[j];",
                             "for (int j = 0; j < dk; ++j) pred += S[(long)r * dk + j] / al[j] * kn[j];"),
    # beta dropped from the write
    "dropped_beta": ("S[(long)r * dk + j] += beta * e[r] * kn[j];",
                     "S[(long)r * dk + j] += e[r] * kn[j];"),
    # output read with the key instead of the query
    "query_as_key": ("            for (int j = 0; j < dk; ++j) acc += S[(long)r * dk + j] * qn[j];",
                     "            for (int j = 0; j < dk; ++j) acc += S[(long)r * dk + j] * kn[j];"),
    # chunk decay off by one (exclusive cumsum)
    "exclusive_cumsum": ("for (int i = 0; i < L; ++i) { acc += g[i]; gcum[i] = acc; }",
                         "for (int i = 0; i < L; ++i) { gcum[i] = acc; acc += g[i]; }"),
    # transposed state in the chunked output
    "transposed_inter": ("inter += Q[(long)i * dk + x] * S[(long)r * dk + x];",
                         "inter += Q[(long)i * dk + x] * S[(long)(x % dv) * dk + (r % dk)];"),
    # wrong sign of the substitution matrix
    "attn_sign": ("a = -bt[i] * dot * decay[(long)i * L + j];",
                  "a = bt[i] * dot * decay[(long)i * L + j];"),
    # rms over the sum instead of the mean
    "rms_sum": ("ms /= dv;", "ms /= 1;"),
    # grouped heads tiled (h % Hk) instead of interleaved (h / r)
    "gva_modulo": ("const int hk = h / (j->H / j->Hk);", "const int hk = h % j->Hk;"),
    # per-channel decay applied to the value rows of S instead of its key columns
    "decay_on_rows": ("for (int j = 0; j < dk; ++j) S[(long)r * dk + j] *= al[j];",
                      "for (int j = 0; j < dk; ++j) S[(long)r * dk + j] *= al[r % dk];"),
    # transition matrix with the per-channel decay on the wrong side
    "transition_decay_side": ("alpha * ((i == j ? 1.0 : 0.0) - beta * kn[i] * kn[j]);",
                              "exp(s->g_per_channel ? gt[j] : gt[0]) * ((i == j ? 1.0 : 0.0) - beta * kn[i] * kn[j]);"),
    # convolution taps in reverse order
    "conv_taps_reversed": ("acc += w[(long)c * K + j] * xp[t + j];",
                           "acc += w[(long)c * K + (K - 1 - j)] * xp[t + j];"),
    # carried convolution state stored newest first
    "conv_state_newest_first": ("state_out[((long)n * channels + c) * (K - 1) + j] = xp[T + j];",
                                "state_out[((long)n * channels + c) * (K - 1) + j] = xp[T + K - 2 - j];"),
    # SiLU left out of the convolution
    "conv_no_silu": ("out[(bos + t) * channels + c] = silu ? acc * sigmoid(acc) : acc;",
                     "out[(bos + t) * channels + c] = acc;"),
    # the query left unnormalised in the token recurrence
    "query_unnormalised": ("l2_normalise(qt, qn, dk, s->use_l2);", "l2_normalise(qt, qn, dk, 0);"),
    # the key left unnormalised in the chunked form
    "chunk_key_unnormalised": ("l2_normalise(s->k + t * s->qk_stride, K + (long)i * dk, dk, s->use_l2);",
                               "l2_normalise(s->k + t * s->qk_stride, K + (long)i * dk, dk, 0);"),
    # eps outside the square root of the normalisation
    "l2_eps_outside_sqrt": ("1.0 / sqrt(ss + L2_EPS)", "1.0 / (sqrt(ss) + L2_EPS)"),
    # query scale dropped in the token recurrence
    "query_scale_dropped": ("for (int j = 0; j < dk; ++j) qn[j] *= s->scale;",
                            "for (int j = 0; j < dk; ++j) qn[j] *= 1.0;"),
    # the initial state ignored by the token recurrence
    "initial_state_ignored": ("    if (s->S0) memcpy(S, s->S0, sizeof(double) * dv * dk);\n\n    for (int t = 0;",
                              "\n\n    for (int t = 0;"),
    # beta left out of U = T diag(beta) V in the chunked form
    "chunk_u_without_beta": ("acc += attn[(long)i * L + j] * bt[j] * V[(long)j * dv + r];",
                             "acc += attn[(long)i * L + j] * V[(long)j * dv + r];"),
    # the decay left out of W = T diag(beta e^gc) K
    "chunk_w_without_decay": ("acc += attn[(long)i * L + j] * bt[j] * exp(gcum[j]) * K[(long)j * dk + x];",
                              "acc += attn[(long)i * L + j] * bt[j] * K[(long)j * dk + x];"),
    # the diagonal kept in the strictly lower A
    "chunk_a_with_diagonal": ("                if (j < i) {", "                if (j <= i) {"),
    # the diagonal dropped from the intra-chunk Q K^T mask
    "chunk_qk_strict": ("                if (j <= i)\n", "                if (j < i)\n"),
    # the inter-chunk term not decayed to the token
    "chunk_inter_undecayed": ("                inter *= exp(gcum[i]);", "                inter *= 1.0;"),
    # SiLU replaced by the bare sigmoid in the gate
    "gate_sigmoid_not_silu": ("out[r * dv + c] = wc * yr[c] * inv * zr[c] * sigmoid(zr[c]);",
                              "out[r * dv + c] = wc * yr[c] * inv * sigmoid(zr[c]);"),
    # the norm weight ignored
    "gate_weight_ignored": ("double wc = w ? w[c] : 1.0;", "double wc = 1.0;"),
    # dt_bias left out of the softplus
    "softplus_without_bias": ("g[i] = -exp(A_log[h]) * softplus(a[i] + bias);",
                              "g[i] = -exp(A_log[h]) * softplus(a[i]);"),
    # A_log used as A
    "a_log_not_exponentiated": ("g[i] = -exp(A_log[h]) * softplus(a[i] + bias);",
                                "g[i] = -A_log[h] * softplus(a[i] + bias);"),
}


def _mutant(tmp_path, name):
    import ctypes
    import subprocess
    src = open(oracle._SRC).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(path),
                    "-lm", "-lpthread"], check=True)
    return ctypes.CDLL(str(so))


PIN_TESTS = [
    test_worked_example_g0_all_forms,
    test_decay_matrix_example,
    test_gated_unit_key_example,
    lambda: test_unit_key_full_write_invariant("recurrence"),
    lambda: test_unit_key_full_write_invariant("chunked16"),
    lambda: [test_orthogonal_keys_reduce_to_gated_linear_attention(f)
             for f in ("recurrence", "chunked4", "chunked64", "transition")],
    test_erase_write_form_and_gated_linear_reference,
    test_beta_zero_is_pure_decay,
    lambda: test_chunked_equals_recurrence(65, 16),
    test_gate_rmsnorm_silu_special_cases_and_library,
    test_grouped_heads_equal_interleaved_repeat,
    test_per_channel_equal_channels_is_scalar_decay,
    test_per_channel_beta_zero_closed_form,
    test_per_channel_unit_key_invariant,
    test_per_channel_transition_equals_recurrence,
    test_conv_identity_tap_is_silu,
    test_conv_impulse_response,
    test_conv_matches_library_conv1d,
    test_conv_varlen_split_and_state,
    test_gates_from_logits,
    lambda: [test_qk_normalisation_and_scale_closed_form(f) for f in ("recurrence", "chunked4")],
    lambda: [test_output_invariant_to_raw_qk_scale(f) for f in ("recurrence", "chunked16")],
]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path, monkeypatch):
    lib = _mutant(tmp_path, name)
    real = oracle._load()
    for fn in ("gdn_oracle_forward", "gdn_oracle_chunk_decay", "gdn_oracle_gate_rmsnorm_silu",
               "gdn_oracle_gates_from_logits"):
        getattr(lib, fn).restype = getattr(real, fn).restype
        getattr(lib, fn).argtypes = getattr(real, fn).argtypes
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = 0
    for pin in PIN_TESTS:
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin catches the planted mistake {name!r}"
