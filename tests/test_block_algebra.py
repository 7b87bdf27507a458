"""The block form of multi-token decode (the streamed decode kernel's blocks of four tokens, and its
one-token blocks at T = 1), checked as algebra on the CPU (fp64, numpy).

The multi-token decode kernel takes a unit's tokens in blocks of four (one at T = 1) in the chunked form of
"[LLM Algorithms-2] Gated DeltaNet" section 4, with G_t the block's cumulative log decay (per key
channel, or one value per head), padding tokens (k = q = v = 0, beta = 0, no decay) after the last
one, and, per state row r:
    A[i][j] = beta_i sum_c k_i[c] k_j[c] e^(G_i - G_j)[c]  (j < i),  T = (I + A)^-1
    V_new[i][r] = sum_j T[i][j] beta_j v_j[r] - s_r . (sum_j T[i][j] beta_j e^G_j . k_j)
    y_i[r] = s_r . (e^G_i . q_i) + sum_(j <= i) M[i][j] V_new[j][r],
             M[i][j] = sum_c q_i[c] k_j[c] e^(G_i - G_j)[c]
    s_r <- e^G_last . s_r + sum_j V_new[j][r] (e^(G_last - G_j) . k_j)
This test restates those equations in numpy and holds them against the oracle's token-by-token
recurrence, so the regrouping itself is pinned independently of any kernel (the GPU tests then hold
the kernel against the oracle)."""
import numpy as np
import pytest

import oracle

BLK = 4


def _block_form(q, k, v, g, beta, S0, BLK=BLK, drop_update_decay=False):
    """One (sequence, head): q, k [T, dk] already normalised and scaled; v [T, dv]; g [T, dk] log decay;
    beta [T]; S0 [dv, dk]; blocks of BLK tokens.  Returns y [T, dv], S [dv, dk]."""
    T, dk = k.shape
    S = S0.copy()
    ys = []
    for t0 in range(0, T, BLK):
        n = min(BLK, T - t0)
        pad = BLK - n

        def padded(x):
            return np.concatenate([x[t0:t0 + n], np.zeros((pad,) + x.shape[1:])], axis=0)

        kb, qb, vb, gb = padded(k), padded(q), padded(v), padded(g)
        bb = np.concatenate([beta[t0:t0 + n], np.zeros(pad)])
        G = np.cumsum(gb, axis=0)                                   # [BLK, dk]
        A = np.zeros((BLK, BLK))
        M = np.zeros((BLK, BLK))
        for i in range(BLK):
            for j in range(BLK):
                ratio = np.exp(G[i] - G[j])
                if j < i:
                    A[i, j] = bb[i] * np.sum(kb[i] * kb[j] * ratio)
                if j <= i:
                    M[i, j] = np.sum(qb[i] * kb[j] * ratio)
        Tm = np.linalg.inv(np.eye(BLK) + A)
        Uc = Tm * bb[None, :]                                       # T diag(beta)
        W = Uc @ (np.exp(G) * kb)                                   # [BLK, dk]
        U = Uc @ vb                                                 # [BLK, dv]
        Vn = U - W @ S.T                                            # [BLK, dv]
        Y = (np.exp(G) * qb) @ S.T + M @ Vn                         # [BLK, dv]
        Kd = np.exp(G[-1][None, :] - G) * kb                        # [BLK, dk]
        S = (S if drop_update_decay else S * np.exp(G[-1])[None, :]) + Vn.T @ Kd
        ys.append(Y[:n])
    return np.concatenate(ys, axis=0), S


@pytest.mark.parametrize("T,per_channel,blk", [(1, False, 4), (3, False, 4), (4, False, 4), (9, False, 4),
                                               (4, True, 4), (7, True, 4), (1, False, 1), (1, True, 1),
                                               (5, True, 1)])
def test_block_form_equals_the_recurrence(T, per_channel, blk):
    rng = np.random.default_rng(100 + T + 10 * per_channel)
    dk, dv = 16, 12
    q = rng.standard_normal((T, 1, dk))
    k = rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    g = -rng.uniform(0.0, 2.0, (T, 1, dk) if per_channel else (T, 1))
    beta = rng.uniform(0.0, 1.0, (T, 1))
    S0 = rng.standard_normal((1, 1, dv, dk)) * 0.3
    y_ref, S_ref = oracle.recurrence(q, k, v, g, beta, batch=1, initial_state=S0)
    # the oracle normalises q, k and scales q by 1/sqrt(dk); the block form takes them prepared
    qn = q[:, 0] / np.sqrt((q[:, 0] ** 2).sum(1, keepdims=True) + 1e-6) / np.sqrt(dk)
    kn = k[:, 0] / np.sqrt((k[:, 0] ** 2).sum(1, keepdims=True) + 1e-6)
    gc = g[:, 0] if per_channel else np.repeat(g[:, :1], dk, axis=1)
    y, S = _block_form(qn, kn, v[:, 0], gc, beta[:, 0], S0[0, 0], BLK=blk)
    np.testing.assert_allclose(y, y_ref[:, 0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(S, S_ref[0, 0], rtol=1e-10, atol=1e-12)


def test_padding_tokens_change_nothing():
    """A block padded with k = q = v = 0, beta = 0 and no decay leaves the state as the real tokens
    left it (the reason any T works in blocks of four)."""
    rng = np.random.default_rng(5)
    dk, dv = 8, 8
    q, k = rng.standard_normal((2, dk)), rng.standard_normal((2, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((2, dv))
    g = -rng.uniform(0, 1, (2, dk))
    beta = rng.uniform(0, 1, 2)
    S0 = rng.standard_normal((dv, dk))
    y2, S2 = _block_form(q, k, v, g, beta, S0)             # two real tokens, two padding tokens
    y1a, S1 = _block_form(q[:1], k[:1], v[:1], g[:1], beta[:1], S0)
    y1b, S1b = _block_form(q[1:], k[1:], v[1:], g[1:], beta[1:], S1)
    np.testing.assert_allclose(S2, S1b, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y2, np.concatenate([y1a, y1b]), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("blk", [1, 4])
def test_planted_mistake_is_caught(blk):
    """The same comparison with the decay left out of the state update (s_r <- s_r + ...) fails:
    the pin distinguishes the regrouping from a plausible wrong one."""
    rng = np.random.default_rng(7)
    T, dk, dv = 6, 16, 12
    q, k, v = rng.standard_normal((T, 1, dk)), rng.standard_normal((T, 1, dk)), rng.standard_normal((T, 1, dv))
    g = -rng.uniform(0.1, 2.0, (T, 1))
    beta = rng.uniform(0.0, 1.0, (T, 1))
    S0 = rng.standard_normal((1, 1, dv, dk)) * 0.3
    y_ref, S_ref = oracle.recurrence(q, k, v, g, beta, batch=1, initial_state=S0)
    qn = q[:, 0] / np.sqrt((q[:, 0] ** 2).sum(1, keepdims=True) + 1e-6) / np.sqrt(dk)
    kn = k[:, 0] / np.sqrt((k[:, 0] ** 2).sum(1, keepdims=True) + 1e-6)
    gc = np.repeat(g[:, :1], dk, axis=1)
    y, S = _block_form(qn, kn, v[:, 0], gc, beta[:, 0], S0[0, 0], BLK=blk, drop_update_decay=True)
    assert not np.allclose(S, S_ref[0, 0], rtol=1e-6, atol=1e-8)
    assert not np.allclose(y, y_ref[:, 0], rtol=1e-6, atol=1e-8)
