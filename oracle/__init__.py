"""fp64 CPU oracle for the linear-attention hot path of position-independent
caching (HYPIC).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the CUDA library and imports nothing from it.

The arithmetic primitives below are the plain definitions (see ``oracle.c``
for the recurrence, the pair and composition, cited there):

* :func:`recurrence` -- the per-token recurrence S_t = A_t S_{t-1} + W_t,
  o_t = S_t^T q_t (HYPIC pages: article “小红书联合北大、上交提出 HYPIC：混合注意力大模型首 Token 延迟降低 3.25 倍，实现位置无关缓存”, section "线性层";
  article “Xiaohongshu, Peking University, Shanghai Jiao Tong University Unveil HYPIC to Slash First Token Latency by 3.25x in Hybrid Attention Models”, linear-layer paragraph; the gated-delta convention with
  scalar-decay and diagonal-gate specialisations).
* :func:`pair` -- (T_C, S(C|0)) of a segment: ordered product of the
  transitions and the zero-initial final state (same sections).
* :func:`compose` -- S(C1 C2) = T(C2) S(C1) + S(C2) (same sections).
* :func:`causal_conv` and :func:`l2_normalize` -- the causal depthwise
  convolution that the pages' "convolution state warm-up" patch refers to
  (article “小红书联合北大、上交提出 HYPIC：混合注意力大模型首 Token 延迟降低 3.25 倍，实现位置无关缓存”, section "线性层", last paragraph), followed by the
  per-head L2 normalisation of q and k that gated-delta layers apply after
  it.  The pages give neither formula; the readings are: kernel size K, lag j
  multiplies x_{t-j}, zero history before the request start, no bias, and
  x / sqrt(sum x^2 + eps) with eps = 1e-6.
* :func:`silu` -- the optional activation between the conv and the
  normalisation (x sigma(x), as public gated-delta layers apply it; not on
  the pages, off unless a descriptor asks for it).

Parity status: every primitive is pinned by ``tests/test_oracle_pins.py``.
"""
import ctypes
import numpy as np

from . import build as _build

GATED_DELTA, SCALAR_DECAY, DIAG_GATE, KDA = 0, 1, 2, 3
L2_EPS = 1e-6

_lib = None
_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(_build.build())
        lib.orc_recurrence.restype = ctypes.c_int
        lib.orc_recurrence.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int64, ctypes.c_int,
                                       _dp, _dp, _dp, _dp, _dp, _dp, _dp,
                                       ctypes.c_int, _i64p, _dp]
        lib.orc_pair.restype = ctypes.c_int
        lib.orc_pair.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_int64, ctypes.c_int,
                                 _dp, _dp, _dp, _dp, _dp, _dp]
        lib.orc_compose.restype = ctypes.c_int
        lib.orc_compose.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    _dp, _dp, _dp, _dp]
        _lib = lib
    return _lib


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x):
    if x is None:
        return None
    return x.ctypes.data_as(_dp)


def _check_shapes(mode, k, v, a, b):
    C, n, dk = k.shape
    if v.shape[:2] != (C, n):
        raise ValueError("v must be [n_chain, n, dv]")
    if mode in (DIAG_GATE, KDA):
        if a.shape != (C, n, dk):
            raise ValueError("per-channel alpha must be [n_chain, n, dk]")
    elif a.shape != (C, n):
        raise ValueError("alpha must be [n_chain, n]")
    if mode in (GATED_DELTA, KDA) and (b is None or b.shape != (C, n)):
        raise ValueError("the delta modes need beta [n_chain, n]")
    return C, n, dk, v.shape[2]


def recurrence(mode, q, k, v, a, b=None, S0=None, record_at=(), want_o=True):
    """Sequential fp64 recurrence over n tokens for each of C chains.

    q, k: [C, n, dk]; v: [C, n, dv]; a: [C, n] (gated delta: alpha, scalar
    decay: gamma per token) or [C, n, dk] (diagonal gate, KDA); b: [C, n]
    (gated delta and KDA); S0: [C, dk, dv] or None for zero.
    Returns (S_final [C, dk, dv], o [C, n, dv] or None, S_rec [C, R, dk, dv])
    where S_rec[:, r] is the state just before token record_at[r].
    """
    k, v, a = _f64(k), _f64(v), _f64(a)
    b = None if b is None else _f64(b)
    C, n, dk, dv = _check_shapes(mode, k, v, a, b)
    q = _f64(q) if (want_o and q is not None) else None
    if want_o and (q is None or q.shape != (C, n, dk)):
        raise ValueError("q must be [n_chain, n, dk] when outputs are wanted")
    S = np.zeros((C, dk, dv)) if S0 is None else _f64(S0).copy()
    o = np.zeros((C, n, dv)) if want_o else None
    rec = np.ascontiguousarray(np.asarray(record_at, dtype=np.int64))
    S_rec = np.zeros((C, len(rec), dk, dv))
    rc = _load().orc_recurrence(mode, dk, dv, n, C, _ptr(q), _ptr(k), _ptr(v),
                                _ptr(a), _ptr(b), _ptr(S), _ptr(o), len(rec),
                                rec.ctypes.data_as(_i64p), _ptr(S_rec))
    if rc != 0:
        raise RuntimeError("orc_recurrence failed (%d)" % rc)
    return S, o, S_rec


def pair(mode, k, v, a, b=None):
    """(T_C, S(C|0)) of each chain's n tokens: T [C, dk, dk], S [C, dk, dv]."""
    k, v, a = _f64(k), _f64(v), _f64(a)
    b = None if b is None else _f64(b)
    C, n, dk, dv = _check_shapes(mode, k, v, a, b)
    T = np.zeros((C, dk, dk))
    S = np.zeros((C, dk, dv))
    rc = _load().orc_pair(mode, dk, dv, n, C, _ptr(k), _ptr(v), _ptr(a),
                          _ptr(b), _ptr(T), _ptr(S))
    if rc != 0:
        raise RuntimeError("orc_pair failed (%d)" % rc)
    return T, S


def compose(T, Sc, S_in):
    """T S_in + Sc for each chain: T [C, dk, dk], Sc and S_in [C, dk, dv]."""
    T, Sc, S_in = _f64(T), _f64(Sc), _f64(S_in)
    C, dk, dv = Sc.shape
    out = np.zeros((C, dk, dv))
    rc = _load().orc_compose(dk, dv, C, _ptr(T), _ptr(Sc), _ptr(S_in), _ptr(out))
    if rc != 0:
        raise RuntimeError("orc_compose failed (%d)" % rc)
    return out


def causal_conv(x, w):
    """Causal depthwise convolution along the token axis.

    x: [n, ch] raw tokens of one stream in request order; w: [ch, K] with
    w[c, j] multiplying x[t - j, c]; tokens before the stream start are zero.
    """
    x = _f64(x)
    w = _f64(w)
    n = x.shape[0]
    y = np.zeros_like(x)
    for j in range(w.shape[1]):
        if j < n:
            y[j:] += w[:, j] * x[:n - j]
    return y


def silu(x):
    """x * sigma(x), sigma the logistic function 1 / (1 + e^-x), evaluated
    without overflow for either sign of x."""
    x = _f64(x)
    e = np.exp(-np.abs(x))
    sig = np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))
    return x * sig


def l2_normalize(x, eps=L2_EPS):
    """x / sqrt(sum(x^2) + eps) over the last axis."""
    x = _f64(x)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)
