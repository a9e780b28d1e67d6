"""The chunked forms of the gated-delta recurrence, in fp64, against the
oracle's token-by-token recurrence (CPU, no GPU).

Two forms are pinned here.  (1) The state update the tensor-core build uses:
with g_t = sum_{s<=t} log alpha_s, Gamma_t = e^{g_t}, D = diag(beta_j
e^{g_C - g_j}) and L''_tj = beta_t k_t.k_j (j < t), W'' = (I + L'')^{-1},
  U~ = D W''^T K,   T_C = Gamma_C I - U~^T diag(Gamma) K,
  S_C = Gamma_C S_0 + U~^T (V - diag(Gamma) K S_0).
(2) Per-token outputs from the same decay-free inverse: with E_ts =
e^{g_t - g_s} (t >= s, 0 above), (I + L)^{-1} = W'' (x) E entry by entry
(every factor <= 1), so
  U = (W'' (x) E) diag(beta) (V - diag(Gamma) K S_0),
  O = diag(Gamma) Q S_0 + (tril(E) (x) Q K^T) U.
The segment recurrence is that of the HYPIC pages' linear layers (article
“小红书联合北大、上交提出 HYPIC：混合注意力大模型首 Token 延迟降低 3.25 倍，实现位置无关缓存”,
section "线性层"): S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
o_t = S_t^T q_t.
"""
import numpy as np
import pytest

import oracle
from oracle import GATED_DELTA

TIGHT = 1e-11


def _chunk(rng, n, dk, dv, slow):
    q = rng.standard_normal((n, dk))
    k = rng.standard_normal((n, dk))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((n, dv))
    a = np.exp(-np.log1p(np.exp(rng.standard_normal(n))) / (64.0 if slow else 1.0))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal(n)))
    S0 = rng.standard_normal((dk, dv))
    return q, k, v, a, b, S0


def _decay_free_inverse(k, b):
    n = k.shape[0]
    Lpp = np.tril(b[:, None] * (k @ k.T), -1)  # L''_tj = beta_t k_t.k_j, j < t
    return np.linalg.inv(np.eye(n) + Lpp)


@pytest.mark.parametrize("slow", [False, True])
@pytest.mark.parametrize("n", [1, 7, 16])
def test_build_state_update_form(n, slow):
    rng = np.random.default_rng(900 + n + 50 * slow)
    dk, dv = 8, 6
    q, k, v, a, b, S0 = _chunk(rng, n, dk, dv, slow)
    g = np.cumsum(np.log(a))
    Gam = np.exp(g)
    Dm = np.diag(b * np.exp(g[-1] - g))
    W = _decay_free_inverse(k, b)
    Ut = Dm @ W.T @ k                                   # U~ = D W''^T K
    T = Gam[-1] * np.eye(dk) - Ut.T @ (Gam[:, None] * k)
    S = Gam[-1] * S0 + Ut.T @ (v - Gam[:, None] * (k @ S0))
    Tr, Sr = oracle.pair(GATED_DELTA, k[None], v[None], a[None], b[None])
    Sf, _, _ = oracle.recurrence(GATED_DELTA, q[None], k[None], v[None], a[None], b[None], S0=S0[None],
                                 want_o=False)
    np.testing.assert_allclose(T, Tr[0], rtol=0, atol=TIGHT)
    np.testing.assert_allclose(S, Sf[0], rtol=0, atol=TIGHT * np.abs(Sf).max())
    # the pair itself (S_0 = 0) and the composition law on this chunk
    np.testing.assert_allclose(Ut.T @ v, Sr[0], rtol=0, atol=TIGHT)
    np.testing.assert_allclose(Tr[0] @ S0 + Sr[0], Sf[0], rtol=0, atol=TIGHT * np.abs(Sf).max())


@pytest.mark.parametrize("slow", [False, True])
@pytest.mark.parametrize("n", [1, 5, 16, 64])
def test_chunk_outputs_from_the_decay_free_inverse(n, slow):
    rng = np.random.default_rng(700 + n + 50 * slow)
    dk, dv = 8, 6
    q, k, v, a, b, S0 = _chunk(rng, n, dk, dv, slow)
    g = np.cumsum(np.log(a))
    Gam = np.exp(g)
    E = np.tril(np.exp(np.minimum(g[:, None] - g[None, :], 0.0)))   # e^{g_t - g_s}, t >= s
    W = _decay_free_inverse(k, b)
    # (I + L)^{-1} with the decays, L_ts = beta_t e^{g_t - g_s} k_t.k_s, equals W'' (x) E
    L = np.tril(b[:, None] * E * (k @ k.T), -1)
    np.testing.assert_allclose(W * E, np.linalg.inv(np.eye(n) + L), rtol=0, atol=TIGHT)
    assert np.all(np.abs(E) <= 1.0)
    U = (W * E) @ (b[:, None] * (v - Gam[:, None] * (k @ S0)))
    O = Gam[:, None] * (q @ S0) + (E * (q @ k.T)) @ U
    S = Gam[-1] * S0 + k.T @ (E[-1][:, None] * U)
    Sf, o, _ = oracle.recurrence(GATED_DELTA, q[None], k[None], v[None], a[None], b[None], S0=S0[None])
    scale = max(1.0, np.abs(o).max())
    np.testing.assert_allclose(O, o[0], rtol=0, atol=TIGHT * scale)
    np.testing.assert_allclose(S, Sf[0], rtol=0, atol=TIGHT * np.abs(Sf).max())


def test_chunk_forms_catch_a_shifted_decay():
    """A plausible slip -- the decay of the current token left out of E
    (e^{g_{t-1} - g_s}) -- changes the outputs well beyond the tolerance."""
    rng = np.random.default_rng(11)
    n, dk, dv = 16, 8, 6
    q, k, v, a, b, S0 = _chunk(rng, n, dk, dv, False)
    g = np.cumsum(np.log(a))
    Gam = np.exp(g)
    gm = np.concatenate([[0.0], g[:-1]])
    E_bad = np.tril(np.exp(np.minimum(gm[:, None] - g[None, :], 0.0)))
    W = _decay_free_inverse(k, b)
    U = (W * E_bad) @ (b[:, None] * (v - Gam[:, None] * (k @ S0)))
    O = Gam[:, None] * (q @ S0) + (E_bad * (q @ k.T)) @ U
    _, o, _ = oracle.recurrence(GATED_DELTA, q[None], k[None], v[None], a[None], b[None], S0=S0[None])
    assert np.abs(O - o[0]).max() > 1e-3
