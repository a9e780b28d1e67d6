"""Expected results of the three hot-path calls, from the fp64 primitives.

TEST INFRASTRUCTURE ONLY (see the package docstring).  These helpers only
gather one (layer, head) chain's tokens out of the packed token-major layout
that the library uses and then call the plain primitives of this package; no
arithmetic of the method lives here beyond what the primitives do.

Packed layout (numpy arrays, any float dtype; bf16 values arrive already
widened):
    q, k, v : [L, N, H, d]
    alpha   : gated delta [L, N, H]; diagonal gate [L, N, H, d_k];
              scalar decay [L, H] (one gamma per head)
    beta    : [L, N, H] (gated delta only)
    conv_w  : [L, 3, H, d, K] (q, k, v channels; lag j multiplies x_{t-j})
Segments are given by offsets seg_off[0..n_seg] into the token axis; a
request is an order of segment indices.  Each segment's first min(w, len)
tokens are its seam window; the cached pair covers the rest (the body).
HYPIC pages (article “小红书联合北大、上交提出 HYPIC：混合注意力大模型首 Token 延迟降低 3.25 倍，实现位置无关缓存”, section "全注意力层"; article “Xiaohongshu, Peking University, Shanghai Jiao Tong University Unveil HYPIC to Slash First Token Latency by 3.25x in Hybrid Attention Models”,
seam-window paragraph): seam tokens are not cached and are re-run under the
full prefix, advancing the running state and emitting per-token outputs.
"""
import numpy as np

from . import (GATED_DELTA, SCALAR_DECAY, DIAG_GATE, KDA, recurrence, pair,
               causal_conv, l2_normalize, silu)


def _np(x):
    if hasattr(x, "detach"):
        x = x.detach().float().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def chain_stream(tok, mode, l, h, idx, conv_k=0, conv_act=0):
    """q, k, v, a, b of chain (l, h) over token indices idx (a stream that
    starts a request: conv history before idx[0] is zero).

    With conv_k > 0 the tokens are raw: q, k, v are convolved along the
    stream (then passed through SiLU when conv_act == 1), then q and k are
    L2-normalised per token.
    """
    idx = np.asarray(idx, dtype=np.int64)
    q = _np(tok["q"][l, idx, h, :]) if tok.get("q") is not None else None
    k = _np(tok["k"][l, idx, h, :])
    v = _np(tok["v"][l, idx, h, :])
    if conv_k:
        w = _np(tok["conv_w"][l, :, h, :, :])  # [3, d, K]
        act = silu if conv_act == 1 else (lambda x: x)
        q = l2_normalize(act(causal_conv(q, w[0]))) if q is not None else None
        k = l2_normalize(act(causal_conv(k, w[1])))
        v = act(causal_conv(v, w[2]))
    if mode == SCALAR_DECAY:
        a = np.full(len(idx), float(_np(tok["alpha"][l, h])))
    else:
        a = _np(tok["alpha"][l, idx, h])
    b = _np(tok["beta"][l, idx, h]) if mode in (GATED_DELTA, KDA) else None
    return q, k, v, a, b


def seam_len(seg_off, s, w):
    return int(min(w, seg_off[s + 1] - seg_off[s]))


def pair_reference(desc, tok, seg_off, items):
    """Dense fp64 (T, S) of the body of segment s for each (l, s, h) in items.

    The body is the segment minus its first min(w, len) seam tokens, taken as
    the segment's own first prefill (a stream that starts at the segment).
    Returns T [n_items, dk, dk], S [n_items, dk, dv].
    """
    mode, w, ck = desc["mode"], desc["seam_w"], desc.get("conv_k", 0)
    Ts, Ss = [], []
    for (l, s, h) in items:
        lo, hi = int(seg_off[s]), int(seg_off[s + 1])
        q, k, v, a, b = chain_stream(tok, mode, l, h, np.arange(lo, hi), ck, desc.get("conv_act", 0))
        sw = seam_len(seg_off, s, w)
        T, S = pair(mode, k[None, sw:], v[None, sw:], a[None, sw:],
                    None if b is None else b[None, sw:])
        Ts.append(T[0])
        Ss.append(S[0])
    return np.stack(Ts), np.stack(Ss)


def layer_arrays(tok, l):
    """One layer of the packed token tensors as float32 numpy arrays
    (q, k, v [N, H, d]; alpha, beta as laid out; conv_w [3, H, d, K]).
    Gathering only: the values are the bf16 / fp32 inputs, widened."""
    out = {}
    for key in ("q", "k", "v", "alpha", "beta", "conv_w"):
        x = tok.get(key)
        out[key] = None if x is None else x[l].detach().float().cpu().numpy()
    return out


def segment_pairs(desc, arrs, seg_off, s):
    """Dense fp64 (T, S) of segment s's body for every head of one layer, in
    one call of the primitive (the heads are independent chains).

    arrs: one layer from :func:`layer_arrays`.  The body is the segment minus
    its first min(w, len) seam tokens, taken as the segment's own first
    prefill (conv history from the segment itself).
    Returns T [H, dk, dk], S [H, dk, dv].
    """
    mode, w, ck = desc["mode"], desc["seam_w"], desc.get("conv_k", 0)
    act = silu if desc.get("conv_act", 0) == 1 else (lambda x: x)
    lo, hi = int(seg_off[s]), int(seg_off[s + 1])
    H = arrs["k"].shape[1]
    sw = seam_len(seg_off, s, w)
    ks, vs, as_, bs = [], [], [], []
    for h in range(H):
        k = np.asarray(arrs["k"][lo:hi, h, :], dtype=np.float64)
        v = np.asarray(arrs["v"][lo:hi, h, :], dtype=np.float64)
        if ck:
            wts = np.asarray(arrs["conv_w"][:, h, :, :], dtype=np.float64)
            k = l2_normalize(act(causal_conv(k, wts[1])))
            v = act(causal_conv(v, wts[2]))
        if mode == SCALAR_DECAY:
            a = np.full(hi - lo, float(arrs["alpha"][h]))
        else:
            a = np.asarray(arrs["alpha"][lo:hi, h], dtype=np.float64)
        ks.append(k[sw:])
        vs.append(v[sw:])
        as_.append(a[sw:])
        if mode in (GATED_DELTA, KDA):
            bs.append(np.asarray(arrs["beta"][lo:hi, h], dtype=np.float64)[sw:])
    return pair(mode, np.stack(ks), np.stack(vs), np.stack(as_),
                np.stack(bs) if bs else None)


def body_output_reference(desc, tok, seg_off, items):
    """Per-token outputs of the body of segment s from a zero state, for each
    (l, s, h) in items: the segment's own first prefill (conv history from
    the segment itself), o_t = S_t^T q_t over the body tokens.
    Returns a list of [n_body, dv] arrays.
    """
    mode, w, ck = desc["mode"], desc["seam_w"], desc.get("conv_k", 0)
    outs = []
    for (l, s, h) in items:
        lo, hi = int(seg_off[s]), int(seg_off[s + 1])
        q, k, v, a, b = chain_stream(tok, mode, l, h, np.arange(lo, hi), ck, desc.get("conv_act", 0))
        sw = seam_len(seg_off, s, w)
        if hi - lo - sw == 0:
            outs.append(np.zeros((0, v.shape[1])))
            continue
        _, o, _ = recurrence(mode, q[None, sw:], k[None, sw:], v[None, sw:], a[None, sw:],
                             None if b is None else b[None, sw:], want_o=True)
        outs.append(o[0])
    return outs


def request_reference(desc, tok, seg_off, order, chains, S_init=None, want_naive=False):
    """Run the recurrence over the whole request (segments in `order`) for
    each chain (l, h) in chains.

    Returns dict with
      S_prefix [n_chain, n_order, dk, dv]: state before each entry's first token
      o_seam   [n_chain, n_order, w, dv]: outputs of each entry's seam tokens
                (rows past the seam length are zero)
      S_final  [n_chain, dk, dv]
      S_naive  [n_chain, dk, dv] (want_naive only): sum of the entries'
                zero-initial final states (the straw man that drops T)
    """
    mode, w, ck = desc["mode"], desc["seam_w"], desc.get("conv_k", 0)
    order = [int(s) for s in order]
    idx = np.concatenate([np.arange(seg_off[s], seg_off[s + 1]) for s in order]
                         ) if order else np.zeros(0, np.int64)
    starts = np.cumsum([0] + [int(seg_off[s + 1] - seg_off[s]) for s in order])
    out = {"S_prefix": [], "o_seam": [], "S_final": [], "S_naive": []}
    if not chains:
        return {key: np.zeros(0) for key in out}
    streams = [chain_stream(tok, mode, l, h, idx, ck, desc.get("conv_act", 0)) for (l, h) in chains]
    q, k, v, a = (np.stack([st[i] for st in streams]) for i in range(4))
    b = None if mode not in (GATED_DELTA, KDA) else np.stack([st[4] for st in streams])
    dk, dv = k.shape[2], v.shape[2]
    S0 = None if S_init is None else np.stack([_np(x) for x in S_init])
    # all chains in one call: independent chains run in parallel
    Sf, o, Srec = recurrence(mode, q, k, v, a, b, S0=S0, record_at=starts[:-1], want_o=True)
    for ci in range(len(chains)):
        oseam = np.zeros((len(order), w, dv))
        naive = np.zeros((dk, dv))
        for e, s in enumerate(order):
            sw = seam_len(seg_off, s, w)
            oseam[e, :sw] = o[ci, starts[e]:starts[e] + sw]
            if want_naive:
                lo, hi = starts[e], starts[e + 1]
                _, Sz = pair(mode, k[ci:ci + 1, lo:hi], v[ci:ci + 1, lo:hi], a[ci:ci + 1, lo:hi],
                             None if b is None else b[ci:ci + 1, lo:hi])
                naive += Sz[0]
        out["S_prefix"].append(Srec[ci])
        out["o_seam"].append(oseam)
        out["S_final"].append(Sf[ci])
        out["S_naive"].append(naive)
    return {key: np.stack(val) for key, val in out.items()}


def seam_reference(desc, tok, seg_off, order, chains, S_in, entries):
    """Seam tokens of the given entries re-run from given states.

    S_in[c][j] is the state before entry entries[j]'s seam for chain c.
    Returns (o [n_chain, n_entries, w, dv], S_out [n_chain, n_entries, dk, dv]).
    With conv, the seam's convolution history is the previous entry's last
    K-1 raw tokens (zero for the first entry): the stream is the request.
    """
    mode, w, ck = desc["mode"], desc["seam_w"], desc.get("conv_k", 0)
    order = [int(s) for s in order]
    idx = np.concatenate([np.arange(seg_off[s], seg_off[s + 1]) for s in order])
    starts = np.cumsum([0] + [int(seg_off[s + 1] - seg_off[s]) for s in order])
    os_, ss_ = [], []
    for ci, (l, h) in enumerate(chains):
        q, k, v, a, b = chain_stream(tok, mode, l, h, idx, ck, desc.get("conv_act", 0))
        dv = v.shape[1]
        o_c, s_c = [], []
        for j, e in enumerate(entries):
            sw = seam_len(seg_off, order[e], w)
            lo = starts[e]
            S0 = _np(S_in[ci][j])[None]
            Sf, o, _ = recurrence(mode, q[None, lo:lo + sw], k[None, lo:lo + sw],
                                  v[None, lo:lo + sw], a[None, lo:lo + sw],
                                  None if b is None else b[None, lo:lo + sw],
                                  S0=S0, want_o=True)
            op = np.zeros((w, dv))
            op[:sw] = o[0]
            o_c.append(op)
            s_c.append(Sf[0])
        os_.append(np.stack(o_c))
        ss_.append(np.stack(s_c))
    return np.stack(os_), np.stack(ss_)


def rel_fro(x, ref, floor=0.0):
    """Relative Frobenius error of one block: |x - ref|_F / max(|ref|_F, floor)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = max(float(np.linalg.norm(ref)), floor)
    num = float(np.linalg.norm(x - ref))
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return num / den
