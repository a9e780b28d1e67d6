"""Pins of the fp64 oracle against what the HYPIC pages and mathematics fix.

Each test checks the oracle against something other than itself: dense
brute-force products, closed forms, exact identities the pages state, the
pages' printed numbers, or an independent library routine.  The cases are
chosen so that a plausible slip in the oracle (a dropped term, a sign, a
transposed operand, a wrong token order) fails at least one of them.
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import GATED_DELTA, SCALAR_DECAY, DIAG_GATE, KDA

HERE = os.path.dirname(os.path.abspath(__file__))
TIGHT = 1e-12


def _rand_tokens(rng, n, dk, dv, mode, slow=False, unit_k=True):
    q = rng.standard_normal((n, dk))
    k = rng.standard_normal((n, dk))
    if unit_k:
        q /= np.linalg.norm(q, axis=1, keepdims=True)
        k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((n, dv))
    sp = np.log1p(np.exp(rng.standard_normal(n if mode not in (DIAG_GATE, KDA) else (n, dk))))
    a = np.exp(-sp / (64.0 if slow else 1.0))
    if mode == SCALAR_DECAY:
        a = np.full(n, 1.0 - 2.0 ** -6)
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal(n))) if mode in (GATED_DELTA, KDA) else None
    return q, k, v, a, b


def _dense_A(mode, k, a, b):
    dk = k.shape[0]
    if mode == GATED_DELTA:
        return a * (np.eye(dk) - b * np.outer(k, k))
    if mode == SCALAR_DECAY:
        return a * np.eye(dk)
    if mode == KDA:
        return (np.eye(dk) - b * np.outer(k, k)) @ np.diag(a)
    return np.diag(a)


def _dense_W(mode, k, v, b):
    return (b if mode in (GATED_DELTA, KDA) else 1.0) * np.outer(k, v)


def _bf(x):
    return None if x is None else x[None]


@pytest.mark.parametrize("mode", [GATED_DELTA, SCALAR_DECAY, DIAG_GATE, KDA])
@pytest.mark.parametrize("n", [1, 3, 8])
def test_brute_force_dense_products(mode, n):
    """Tiny d: T is the ordered product of dense A_t, S and o follow from
    dense matrix steps (transition applied on the left, newest token last)."""
    rng = np.random.default_rng(100 + 7 * mode + n)
    dk = dv = 4
    q, k, v, a, b = _rand_tokens(rng, n, dk, dv, mode)
    S0 = rng.standard_normal((dk, dv))
    T_bf = np.eye(dk)
    S_bf = S0.copy()
    o_bf = np.zeros((n, dv))
    for t in range(n):
        At = _dense_A(mode, k[t], a[t], None if b is None else b[t])
        T_bf = At @ T_bf
        S_bf = At @ S_bf + _dense_W(mode, k[t], v[t], None if b is None else b[t])
        o_bf[t] = S_bf.T @ q[t]
    T, Sz = oracle.pair(mode, k[None], v[None], a[None], _bf(b))
    Sf, o, _ = oracle.recurrence(mode, q[None], k[None], v[None], a[None], _bf(b), S0=S0[None])
    np.testing.assert_allclose(T[0], T_bf, rtol=0, atol=TIGHT)
    np.testing.assert_allclose(Sf[0], S_bf, rtol=0, atol=TIGHT)
    np.testing.assert_allclose(o[0], o_bf, rtol=0, atol=TIGHT)
    # the pair applied to S0 gives the same state: T S0 + S(C|0)
    np.testing.assert_allclose(T[0] @ S0 + Sz[0], S_bf, rtol=0, atol=TIGHT)


@pytest.mark.parametrize("mode", [GATED_DELTA, SCALAR_DECAY, DIAG_GATE])
def test_composition_law(mode):
    """S(C1 C2) = T(C2) S(C1) + S(C2) (article “小红书联合北大、上交提出 HYPIC：混合注意力大模型首 Token 延迟降低 3.25 倍，实现位置无关缓存”, 线性层)."""
    rng = np.random.default_rng(11 + mode)
    dk = dv = 8
    n1, n2 = 37, 29
    q, k, v, a, b = _rand_tokens(rng, n1 + n2, dk, dv, mode, slow=True)
    S_cat, _, _ = oracle.recurrence(mode, q[None], k[None], v[None], a[None], _bf(b), want_o=False)
    sl1, sl2 = slice(0, n1), slice(n1, n1 + n2)
    T1, S1 = oracle.pair(mode, k[None, sl1], v[None, sl1], a[None, sl1], None if b is None else b[None, sl1])
    T2, S2 = oracle.pair(mode, k[None, sl2], v[None, sl2], a[None, sl2], None if b is None else b[None, sl2])
    composed = oracle.compose(T2, S2, S1)
    np.testing.assert_allclose(composed, S_cat, rtol=0, atol=1e-12)
    # T of the concatenation is the ordered product T2 T1 (not T1 T2)
    T12, _ = oracle.pair(mode, k[None], v[None], a[None], _bf(b))
    np.testing.assert_allclose(T12[0], T2[0] @ T1[0], rtol=0, atol=1e-12)
    if mode == GATED_DELTA:
        assert np.linalg.norm(T2[0] @ T1[0] - T1[0] @ T2[0]) > 1e-3
    # the law is not vacuous here: T2 S1 is a sizeable part of the state
    assert np.linalg.norm(T2[0] @ S1[0]) > 0.05 * np.linalg.norm(S_cat[0])


def test_associativity_of_pairs():
    rng = np.random.default_rng(5)
    dk = dv = 6
    ns = [11, 17, 9]
    q, k, v, a, b = _rand_tokens(rng, sum(ns), dk, dv, GATED_DELTA, slow=True)
    cuts = np.cumsum([0] + ns)
    P = []
    for i in range(3):
        s = slice(cuts[i], cuts[i + 1])
        P.append(oracle.pair(GATED_DELTA, k[None, s], v[None, s], a[None, s], b[None, s]))

    def comp(p2, p1):  # (T2,S2) o (T1,S1)
        return p2[0] @ p1[0], oracle.compose(p2[0], p2[1], p1[1])

    left = comp(comp(P[2], P[1]), P[0])
    right = comp(P[2], comp(P[1], P[0]))
    whole = oracle.pair(GATED_DELTA, k[None], v[None], a[None], b[None])
    for x, y in ((left, right), (left, whole)):
        np.testing.assert_allclose(x[0], y[0], atol=1e-12, rtol=0)
        np.testing.assert_allclose(x[1], y[1], atol=1e-12, rtol=0)


@pytest.mark.parametrize("gamma", [1.0 - 2.0 ** -5, 1.0 - 2.0 ** -10, 0.5])
def test_scalar_decay_closed_form(gamma):
    """Pure decay: T_C = gamma^L I and S(C|0) = sum_t gamma^(L-t) k_t v_t^T."""
    rng = np.random.default_rng(3)
    n, dk, dv = 200, 8, 5
    k = rng.standard_normal((n, dk))
    v = rng.standard_normal((n, dv))
    a = np.full(n, gamma)
    T, S = oracle.pair(SCALAR_DECAY, k[None], v[None], a[None])
    np.testing.assert_allclose(T[0], gamma ** n * np.eye(dk), rtol=1e-12, atol=0)
    wts = gamma ** (n - 1 - np.arange(n))
    S_cf = np.einsum("t,ti,tj->ij", wts, k, v)
    np.testing.assert_allclose(S[0], S_cf, rtol=1e-11, atol=1e-12)


def test_diagonal_gate_closed_form():
    """Diagonal gate: T = diag(prod_t alpha_t) and
    S = sum_t diag(prod_{s>t} alpha_s) k_t v_t^T."""
    rng = np.random.default_rng(4)
    n, dk, dv = 40, 6, 3
    k = rng.standard_normal((n, dk))
    v = rng.standard_normal((n, dv))
    a = rng.uniform(0.8, 1.0, size=(n, dk))
    T, S = oracle.pair(DIAG_GATE, k[None], v[None], a[None])
    np.testing.assert_allclose(T[0], np.diag(np.prod(a, axis=0)), rtol=1e-12, atol=0)
    later = np.vstack([np.prod(a[t + 1:], axis=0) for t in range(n)])  # [n, dk]
    S_cf = np.einsum("ti,ti,tj->ij", later, k, v)
    np.testing.assert_allclose(S[0], S_cf, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("mode", [SCALAR_DECAY, DIAG_GATE])
def test_naive_addition_exact_for_plain_linear_attention(mode):
    """With A_t = I (plain linear attention) summing zero-initial states is
    exact (article “小红书联合北大、上交提出 HYPIC：混合注意力大模型首 Token 延迟降低 3.25 倍，实现位置无关缓存”, 线性层)."""
    rng = np.random.default_rng(8)
    dk = dv = 5
    ns = [13, 21, 8]
    n = sum(ns)
    k = rng.standard_normal((n, dk))
    v = rng.standard_normal((n, dv))
    a = np.ones((n, dk)) if mode == DIAG_GATE else np.ones(n)
    S_cat, _, _ = oracle.recurrence(mode, None, k[None], v[None], a[None], want_o=False)
    cuts = np.cumsum([0] + ns)
    naive = sum(oracle.pair(mode, k[None, cuts[i]:cuts[i + 1]], v[None, cuts[i]:cuts[i + 1]],
                            a[None, cuts[i]:cuts[i + 1]])[1][0] for i in range(3))
    np.testing.assert_allclose(naive, S_cat[0], rtol=0, atol=1e-12)
    # and equals the plain sum of outer products
    np.testing.assert_allclose(S_cat[0], k.T @ v, rtol=0, atol=1e-12)


@pytest.mark.parametrize("mode", [GATED_DELTA, SCALAR_DECAY, DIAG_GATE])
def test_naive_addition_wrong_under_decay(mode):
    """Under decay, gating or delta erasure the straw man is structurally
    wrong (article “小红书联合北大、上交提出 HYPIC：混合注意力大模型首 Token 延迟降低 3.25 倍，实现位置无关缓存”, 线性层)."""
    rng = np.random.default_rng(9 + mode)
    dk = dv = 8
    n1 = n2 = 64
    q, k, v, a, b = _rand_tokens(rng, n1 + n2, dk, dv, mode, slow=True)
    S_cat, _, _ = oracle.recurrence(mode, q[None], k[None], v[None], a[None], _bf(b), want_o=False)
    bb = (lambda s: None if b is None else b[None, s])
    _, S1 = oracle.pair(mode, k[None, :n1], v[None, :n1], a[None, :n1], bb(slice(0, n1)))
    _, S2 = oracle.pair(mode, k[None, n1:], v[None, n1:], a[None, n1:], bb(slice(n1, None)))
    err = np.linalg.norm(S1[0] + S2[0] - S_cat[0]) / np.linalg.norm(S_cat[0])
    assert err > 0.01


def test_retnet_slow_decay_naive_error_matches_pages():
    """The pages' figure: 22% of the state norm at 256 tokens on a slow-decay
    RetNet head.  For scalar decay the straw man's error is exactly
    (1 - gamma^256) S(C1|0); the slowest-but-two head of the decay workload,
    gamma = 1 - 2^-10, gives 1 - gamma^256 = 0.221."""
    with open(os.path.join(HERE, "golden", "pages_numbers.json")) as f:
        pages = json.load(f)["naive_add_error_retnet_slow_decay"]
    n = pages["tokens"]
    gamma = 1.0 - 2.0 ** -10
    rng = np.random.default_rng(22)
    dk = dv = 16
    k = rng.standard_normal((2 * n, dk)) / np.sqrt(dk)
    v = rng.standard_normal((2 * n, dv))
    a = np.full(2 * n, gamma)
    S_cat, _, _ = oracle.recurrence(SCALAR_DECAY, None, k[None], v[None], a[None], want_o=False)
    _, S1 = oracle.pair(SCALAR_DECAY, k[None, :n], v[None, :n], a[None, :n])
    _, S2 = oracle.pair(SCALAR_DECAY, k[None, n:], v[None, n:], a[None, n:])
    rel = np.linalg.norm(S1[0] + S2[0] - S_cat[0]) / np.linalg.norm(S1[0])
    assert rel == pytest.approx(1.0 - gamma ** n, rel=1e-10)
    assert abs(rel - pages["value"]) < 0.005


def test_gated_delta_determinant_lemma():
    """det A_t = alpha^d (1 - beta |k|^2), so log det T_C is the sum."""
    rng = np.random.default_rng(12)
    n, dk = 12, 5
    q, k, v, a, b = _rand_tokens(rng, n, dk, dk, GATED_DELTA, slow=True, unit_k=False)
    k *= 0.6
    T, _ = oracle.pair(GATED_DELTA, k[None], v[None], a[None], b[None])
    sign, logdet = np.linalg.slogdet(T[0])
    expect = np.sum(dk * np.log(a) + np.log(np.abs(1.0 - b * np.sum(k * k, axis=1))))
    assert logdet == pytest.approx(expect, rel=1e-10)


def test_gated_delta_contraction_and_projector():
    rng = np.random.default_rng(13)
    n, dk = 30, 6
    q, k, v, a, b = _rand_tokens(rng, n, dk, dk, GATED_DELTA, slow=True)
    T, _ = oracle.pair(GATED_DELTA, k[None], v[None], a[None], b[None])
    assert np.linalg.norm(T[0], 2) <= np.prod(a) * (1 + 1e-12)
    # alpha = beta = 1, unit k: the last token's transition is a projector,
    # so k_L^T T_C = 0 (left null vector) while T_C k_L is not zero.
    a1 = np.ones(n)
    b1 = np.ones(n)
    T1, _ = oracle.pair(GATED_DELTA, k[None], v[None], a1[None], b1[None])
    assert np.linalg.norm(k[-1] @ T1[0]) < 1e-12
    assert np.linalg.norm(T1[0] @ k[-1]) > 1e-3


def test_gated_delta_special_cases():
    rng = np.random.default_rng(14)
    n, dk = 9, 4
    q, k, v, a, b = _rand_tokens(rng, n, dk, dk, GATED_DELTA)
    # beta = 0: no write, no erasure: T = prod(alpha) I, S = 0
    T, S = oracle.pair(GATED_DELTA, k[None], v[None], a[None], np.zeros((1, n)))
    np.testing.assert_allclose(T[0], np.prod(a) * np.eye(dk), rtol=1e-12, atol=0)
    assert np.all(S == 0)
    # alpha = 0 on the last token resets everything
    a0 = a.copy()
    a0[-1] = 0.0
    T, S = oracle.pair(GATED_DELTA, k[None], v[None], a0[None], b[None])
    assert np.all(T == 0)
    np.testing.assert_allclose(S[0], b[-1] * np.outer(k[-1], v[-1]), atol=1e-15)
    # empty segment: identity pair
    T, S = oracle.pair(GATED_DELTA, k[None, :0], v[None, :0], a[None, :0], b[None, :0])
    np.testing.assert_array_equal(T[0], np.eye(dk))
    assert np.all(S == 0)


def test_seam_then_body_equals_whole_segment():
    """Re-running a segment's seam token by token and then applying its body
    pair is the whole segment's map (the seam-window reading)."""
    rng = np.random.default_rng(15)
    dk = dv = 8
    n, w = 50, 8
    q, k, v, a, b = _rand_tokens(rng, n, dk, dv, GATED_DELTA, slow=True)
    S0 = rng.standard_normal((1, dk, dv))
    Sw, o_seam, _ = oracle.recurrence(GATED_DELTA, q[None, :w], k[None, :w], v[None, :w],
                                      a[None, :w], b[None, :w], S0=S0)
    Tb, Sb = oracle.pair(GATED_DELTA, k[None, w:], v[None, w:], a[None, w:], b[None, w:])
    Sf, o_all, _ = oracle.recurrence(GATED_DELTA, q[None], k[None], v[None], a[None], b[None], S0=S0)
    np.testing.assert_allclose(oracle.compose(Tb, Sb, Sw), Sf, atol=1e-12, rtol=0)
    np.testing.assert_allclose(o_seam[0], o_all[0, :w], atol=1e-12, rtol=0)


def test_recording_positions():
    rng = np.random.default_rng(16)
    dk = dv = 4
    n = 20
    q, k, v, a, b = _rand_tokens(rng, n, dk, dv, GATED_DELTA)
    _, _, rec = oracle.recurrence(GATED_DELTA, q[None], k[None], v[None], a[None], b[None],
                                  record_at=[0, 7, 20], want_o=False)
    assert np.all(rec[0, 0] == 0)
    S7, _, _ = oracle.recurrence(GATED_DELTA, q[None, :7], k[None, :7], v[None, :7], a[None, :7],
                                 b[None, :7], want_o=False)
    np.testing.assert_array_equal(rec[0, 1], S7[0])
    Sf, _, _ = oracle.recurrence(GATED_DELTA, q[None], k[None], v[None], a[None], b[None], want_o=False)
    np.testing.assert_array_equal(rec[0, 2], Sf[0])


def test_compose_against_matmul():
    rng = np.random.default_rng(17)
    T = rng.standard_normal((3, 7, 7))
    Sc = rng.standard_normal((3, 7, 5))
    S0 = rng.standard_normal((3, 7, 5))
    np.testing.assert_allclose(oracle.compose(T, Sc, S0), T @ S0 + Sc, atol=1e-12, rtol=0)


def test_causal_conv():
    rng = np.random.default_rng(18)
    n, ch, K = 30, 6, 4
    x = rng.standard_normal((n, ch))
    ident = np.zeros((ch, K))
    ident[:, 0] = 1.0
    np.testing.assert_array_equal(oracle.causal_conv(x, ident), x)
    shift = np.zeros((ch, K))
    shift[:, 1] = 1.0
    y = oracle.causal_conv(x, shift)
    assert np.all(y[0] == 0)
    np.testing.assert_array_equal(y[1:], x[:-1])
    w = rng.standard_normal((ch, K))
    y = oracle.causal_conv(x, w)
    for c in range(ch):
        np.testing.assert_allclose(y[:, c], np.convolve(x[:, c], w[c])[:n], atol=1e-12)
    # a later token only sees the last K-1 tokens: a stream started K-1 tokens
    # before position p reproduces y[p:] exactly (prefix independence)
    p = 17
    y2 = oracle.causal_conv(x[p - (K - 1):], w)
    np.testing.assert_allclose(y2[K - 1:], y[p:], atol=1e-12)


def test_silu():
    """SiLU = x sigma(x) pinned by identities that do not restate it: the odd
    part silu(x) - silu(-x) = x (sigma(x) + sigma(-x) = 1), the logistic as
    (1 + tanh(x / 2)) / 2, silu(0) = 0 with slope 1/2 there, the asymptotes
    x and 0, and finiteness far out on both sides."""
    rng = np.random.default_rng(31)
    x = rng.standard_normal(200) * 6
    np.testing.assert_allclose(oracle.silu(x) - oracle.silu(-x), x, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(oracle.silu(x), x * 0.5 * (1.0 + np.tanh(0.5 * x)), rtol=1e-13, atol=1e-15)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    hstep = 1e-6
    slope = (oracle.silu(np.array([hstep]))[0] - oracle.silu(np.array([-hstep]))[0]) / (2 * hstep)
    assert abs(slope - 0.5) < 1e-9
    big = np.array([40.0, 800.0])
    np.testing.assert_allclose(oracle.silu(big), big, rtol=1e-15)
    far = oracle.silu(np.array([-40.0, -800.0]))
    assert np.all(np.isfinite(far)) and abs(far[0]) < 1e-15 and far[1] == 0.0


def test_l2_normalize():
    """Hand-computed rows: (3, 4) has norm 5, so with eps = 0 it maps to
    (0.6, 0.8) and with eps = 11 (sqrt(25 + 11) = 6) to (1/2, 2/3); (1, 2, 2)
    has norm 3, so with eps = 7 (sqrt(9 + 7) = 4) it maps to (1/4, 1/2, 1/2).
    Rows are normalised independently; a zero row stays zero; the result is
    invariant to scaling the row when eps = 0."""
    x = np.array([[3.0, 4.0], [0.0, 0.0], [-4.0, 3.0]])
    np.testing.assert_allclose(oracle.l2_normalize(x, eps=0.0)[[0, 2]], [[0.6, 0.8], [-0.8, 0.6]], rtol=0, atol=1e-15)
    np.testing.assert_allclose(oracle.l2_normalize(x, eps=11.0), [[0.5, 2.0 / 3.0], [0.0, 0.0], [-2.0 / 3.0, 0.5]],
                               rtol=0, atol=1e-15)
    np.testing.assert_allclose(oracle.l2_normalize(np.array([[1.0, 2.0, 2.0]]), eps=7.0), [[0.25, 0.5, 0.5]],
                               rtol=0, atol=1e-15)
    rng = np.random.default_rng(19)
    y = rng.standard_normal((10, 16)) * 5
    np.testing.assert_allclose(oracle.l2_normalize(3.0 * y, eps=0.0), oracle.l2_normalize(y, eps=0.0), rtol=1e-12)
    assert np.all(oracle.l2_normalize(np.zeros((1, 4))) == 0)


def test_kda_reduces_to_gated_delta_and_diagonal_gate():
    """KDA with the same decay on every channel is gated delta (diag(alpha)
    commutes with the projector); KDA with beta = 0 is the diagonal gate
    without a write, so T = diag(prod alpha) and S(C|0) = 0."""
    rng = np.random.default_rng(77)
    n, dk, dv = 37, 6, 5
    q, k, v, a, b = _rand_tokens(rng, n, dk, dv, KDA, slow=True)
    a_uni = np.repeat(a[:, :1], dk, axis=1)
    T1, S1 = oracle.pair(KDA, k[None], v[None], a_uni[None], b[None])
    T2, S2 = oracle.pair(GATED_DELTA, k[None], v[None], a_uni[None, :, 0], b[None])
    np.testing.assert_allclose(T1, T2, rtol=0, atol=TIGHT)
    np.testing.assert_allclose(S1, S2, rtol=0, atol=TIGHT)
    T0, S0 = oracle.pair(KDA, k[None], v[None], a[None], np.zeros((1, n)))
    np.testing.assert_allclose(T0[0], np.diag(np.prod(a, axis=0)), rtol=1e-13, atol=0)
    assert np.abs(S0).max() == 0.0


def test_kda_composition_law():
    """S(C1 C2) = T(C2) S(C1) + S(C2) for KDA pairs, against the recurrence
    over the concatenated stream."""
    rng = np.random.default_rng(78)
    n1, n2, dk, dv = 23, 31, 8, 8
    q, k, v, a, b = _rand_tokens(rng, n1 + n2, dk, dv, KDA, slow=True)
    T1, S1 = oracle.pair(KDA, k[None, :n1], v[None, :n1], a[None, :n1], b[None, :n1])
    T2, S2 = oracle.pair(KDA, k[None, n1:], v[None, n1:], a[None, n1:], b[None, n1:])
    Sf, _, _ = oracle.recurrence(KDA, None, k[None], v[None], a[None], b[None], want_o=False)
    np.testing.assert_allclose(T2[0] @ S1[0] + S2[0], Sf[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(oracle.compose(T2, S2, S1)[0], Sf[0], rtol=0, atol=1e-12)


@pytest.mark.parametrize("name", ["tiny_gdn", "decay_retnet", "decay_diag", "kda_tiny"])
def test_body_outputs_end_on_the_pair(name):
    """The body outputs of a segment's first prefill end on its pair: the
    last body token's output is S(C|0)^T q of that token, with S(C|0) from
    the pair routine (an independent code path: transitions applied to a
    zero state, no outputs)."""
    from linear_attn_state_chunked_gb300 import workloads as W
    from oracle import reference as ref
    wl = W.make(name, device="cpu")
    d = wl.desc
    items = [(0, s, 0) for s in range(wl.n_seg)]
    outs = ref.body_output_reference(d, wl.tok, wl.seg_off, items)
    _, Sref = ref.pair_reference(d, wl.tok, wl.seg_off, items)
    for (l, s, h), o, S in zip(items, outs, Sref):
        if len(o) == 0:
            continue
        lo, hi = int(wl.seg_off[s]), int(wl.seg_off[s + 1])
        q, _, _, _, _ = ref.chain_stream(wl.tok, d["mode"], l, h, np.arange(lo, hi), d.get("conv_k", 0))
        np.testing.assert_allclose(o[-1], S.T @ q[-1], rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("mode", [GATED_DELTA, SCALAR_DECAY, DIAG_GATE, KDA])
def test_body_outputs_brute_force(mode):
    """Every per-token output of a segment body's first prefill, against
    dense brute force on a tiny case (d = 4): S_t = A_t S_{t-1} + W_t from
    S = 0 at the body's first token, o_t = S_t^T q_t.  An off-by-one in which
    state is dotted with q, a skipped seam offset or a transposed S fails."""
    from oracle import reference as ref
    rng = np.random.default_rng(300 + mode)
    L, H, dk, w = 1, 2, 4, 2
    lens = [5, 1, 7]
    N = sum(lens)
    seg_off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    tok = {"q": np.zeros((L, N, H, dk)), "k": np.zeros((L, N, H, dk)), "v": np.zeros((L, N, H, dk)),
           "beta": None, "conv_w": None}
    per_head = []
    for h in range(H):
        q, k, v, a, b = _rand_tokens(rng, N, dk, dk, mode, slow=True)
        tok["q"][0, :, h], tok["k"][0, :, h], tok["v"][0, :, h] = q, k, v
        per_head.append((q, k, v, a, b))
    if mode == SCALAR_DECAY:
        tok["alpha"] = np.array([[per_head[h][3][0] for h in range(H)]])
    elif mode in (DIAG_GATE, KDA):
        tok["alpha"] = np.stack([ph[3] for ph in per_head], axis=1)[None]
    else:
        tok["alpha"] = np.stack([ph[3] for ph in per_head], axis=1)[None]
    if mode in (GATED_DELTA, KDA):
        tok["beta"] = np.stack([ph[4] for ph in per_head], axis=1)[None]
    desc = dict(mode=mode, seam_w=w, conv_k=0, conv_act=0)
    items = [(0, s, h) for s in range(len(lens)) for h in range(H)]
    outs = ref.body_output_reference(desc, tok, seg_off, items)
    for (l, s, h), o in zip(items, outs):
        q, k, v, a, b = per_head[h]
        lo, hi = int(seg_off[s]), int(seg_off[s + 1])
        body = range(lo + min(w, hi - lo), hi)
        assert o.shape == (len(body), dk)
        S = np.zeros((dk, dk))
        for i, t in enumerate(body):
            S = _dense_A(mode, k[t], a[t], None if b is None else b[t]) @ S + \
                _dense_W(mode, k[t], v[t], None if b is None else b[t])
            np.testing.assert_allclose(o[i], S.T @ q[t], rtol=0, atol=1e-12)
