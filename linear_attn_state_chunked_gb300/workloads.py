"""Seeded synthetic inputs for the hot path's workloads.

This module only draws and lays out inputs; it holds none of the method's
arithmetic.  Both the CUDA path (tests, benchmark) and the fp64 oracle (through
copies the tests make) consume what it returns.

Recipes (token tensors are drawn in fp32 and then stored in the workload's
input dtype; bf16 rounding happens here, so both sides see the same values):

* q, k ~ N(0, 1), L2-normalised per (token, head) -- except for workloads
  with a causal conv, whose q/k/v are raw N(0, 1) tokens (the library
  convolves and normalises them);
* v ~ N(0, 1);
* gated delta: alpha = exp(-softplus(z)), beta = sigmoid(z'), z, z' ~ N(0, 1);
  the slow-gate stress variant uses alpha = exp(-softplus(z) / 64), plain
  DeltaNet alpha = 1;
* scalar decay (RetNet): gamma_h = 1 - 2^(-5-h);
* diagonal gate: alpha_t[c] = exp(-softplus(z)) per channel;
* KDA: alpha_t[c] = exp(-softplus(z) / 16) per channel, beta = sigmoid(z');
* conv weights ~ N(0, 1) / 2.

Segment lengths, orders and seeds:

* tiny_gdn      1 layer, 1 head, d=16, fp32, 4 x 64 tokens, seed 0, w=0
* decay_retnet  1 layer, 8 heads, d=64, fp32, 16 x 256 tokens, seed 1, w=0
* decay_diag    same shape, diagonal gate, seed 1, w=0
* gdn_bf16      1 layer, 32 heads, d=128, bf16, 64 segments with lengths
                uniform on [512, 2048], seed 2, w=8
* warm_30l      30 layers, 32 heads, d=128, bf16, 128 segments with lengths
                uniform on [512, 1050] rescaled to sum to 100,000; layer l is
                drawn from seed 3*1000+l; request order is a permutation drawn
                from seed 3*10^6+r; w=8
* cold_30l      30 layers, 32 heads, d=128, bf16, 200 segments with lognormal
                lengths (median 512, sigma 0.8) clipped to [64, 4096] and
                rescaled to sum to 100,000 (re-clipped, remainder on the
                longest), conv taps 4, seed 4 (layer l from 4*1000+l), w=8,
                request order = segment order (a cold prompt)
* stress_tiny / stress_gdn  the tiny_gdn / gdn_bf16 shapes with the slow gate
                (seeds 5 and 6), so that T_C stays far from zero.
* stress_cold   the cold_30l shape (200 lognormal segments up to 4096 tokens,
                conv taps 4, w=8) with the slow gate, 2 layers, seed 10: the
                longest bodies under a gate that keeps T_C large.
* deltanet      plain DeltaNet (gated delta with alpha = 1): 1 layer, 2 heads,
                d=32, fp32, 6 x 50 tokens, seed 9, w=8
* kda_tiny      KDA, 1 layer, 2 heads, d=16, fp32, 4 x 64 tokens, seed 7, w=0
* kda_bf16      KDA, 1 layer, 4 heads, d=64, bf16, 12 segments with lengths
                uniform on [40, 300], conv taps 4, seed 8, w=8
"""
from dataclasses import dataclass, field

import numpy as np
import torch

GATED_DELTA, SCALAR_DECAY, DIAG_GATE, KDA = 0, 1, 2, 3
F32, BF16 = 0, 1

_TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}


@dataclass
class Workload:
    name: str
    desc: dict                    # n_layers, n_heads, d_k, d_v, seam_w, conv_k, mode, in_dtype
    seg_off: np.ndarray           # int64 [n_seg + 1]
    order: np.ndarray             # int32 [n_order]
    tok: dict = field(default_factory=dict)  # q, k, v, alpha, beta, conv_w tensors

    @property
    def n_tokens(self):
        return int(self.seg_off[-1])

    @property
    def n_seg(self):
        return len(self.seg_off) - 1

    @property
    def lengths(self):
        return np.diff(self.seg_off)


def _rescale(lengths, total, lo, hi):
    """Scale integer lengths to sum to `total`, re-clip to [lo, hi] and put the
    remainder on the longest segment."""
    x = np.asarray(lengths, dtype=np.float64)
    x = np.rint(x * (total / x.sum())).astype(np.int64)
    x = np.clip(x, lo, hi)
    x[int(np.argmax(x))] += total - int(x.sum())
    return x


def segment_lengths(name):
    if name in ("tiny_gdn", "stress_tiny"):
        return np.full(4, 64, np.int64)
    if name in ("decay_retnet", "decay_diag"):
        return np.full(16, 256, np.int64)
    if name in ("gdn_bf16", "stress_gdn"):
        seed = 2 if name == "gdn_bf16" else 6
        return np.random.default_rng(seed).integers(512, 2049, size=64).astype(np.int64)
    if name == "warm_30l":
        raw = np.random.default_rng(3).integers(512, 1051, size=128)
        return _rescale(raw, 100_000, 512, 1050)
    if name == "deltanet":
        return np.full(6, 50, np.int64)
    if name == "kda_tiny":
        return np.full(4, 64, np.int64)
    if name == "kda_bf16":
        return np.random.default_rng(8).integers(40, 301, size=12).astype(np.int64)
    if name in ("cold_30l", "stress_cold"):
        raw = np.random.default_rng(4).lognormal(np.log(512.0), 0.8, size=200)
        raw = np.clip(np.rint(raw), 64, 4096)
        return _rescale(raw, 100_000, 64, 4096)
    raise KeyError(name)


_SPECS = {
    #  name            mode          L   H   d   dtype  seed w  conv gate divisor (0: alpha = 1)
    "tiny_gdn":     (GATED_DELTA,  1,  1, 16, F32,  0,   0, 0, 1.0),
    "decay_retnet": (SCALAR_DECAY, 1,  8, 64, F32,  1,   0, 0, 1.0),
    "decay_diag":   (DIAG_GATE,    1,  8, 64, F32,  1,   0, 0, 1.0),
    "gdn_bf16":     (GATED_DELTA,  1, 32, 128, BF16, 2,  8, 0, 1.0),
    "warm_30l":     (GATED_DELTA, 30, 32, 128, BF16, 3,  8, 0, 1.0),
    "cold_30l":     (GATED_DELTA, 30, 32, 128, BF16, 4,  8, 4, 1.0),
    "stress_tiny":  (GATED_DELTA,  1,  1, 16, F32,  5,   0, 0, 64.0),
    "stress_gdn":   (GATED_DELTA,  1, 32, 128, BF16, 6,  8, 0, 64.0),
    "stress_cold":  (GATED_DELTA,  2, 32, 128, BF16, 10, 8, 4, 64.0),
    "deltanet":     (GATED_DELTA,  1,  2, 32, F32,  9,   8, 0, 0.0),
    "kda_tiny":     (KDA,          1,  2, 16, F32,  7,   0, 0, 16.0),
    "kda_bf16":     (KDA,          1,  4, 64, BF16, 8,   8, 4, 16.0),
}

NAMES = tuple(_SPECS)


def describe(name, **over):
    mode, L, H, d, dt, seed, w, ck, gdiv = _SPECS[name]
    desc = dict(n_layers=L, n_heads=H, d_k=d, d_v=d, seam_w=w, conv_k=ck,
                mode=mode, in_dtype=dt, conv_act=0)
    desc.update(over)
    return desc


def request_order(name, r=0):
    n = len(segment_lengths(name))
    if name == "warm_30l":
        return np.random.default_rng(3 * 10**6 + r).permutation(n).astype(np.int32)
    return np.arange(n, dtype=np.int32)


def _layer_seed(name, seed, l, L):
    # single-layer workloads keep their seed for layer 0; extra layers drawn
    # for tests (and every layer of a stack) use seed*1000 + l
    return seed if (L == 1 and l == 0) else seed * 1000 + l


def make(name, device="cpu", layers=None, lengths=None, order=None,
         **desc_over):
    """Draw the named workload on `device`.

    layers: draw only this many layers (a prefix of the stack; the per-layer
    seeds make the first layers identical to the full workload's).
    lengths / order: override the segment lengths / request order (edge-case
    tests); desc_over overrides descriptor fields (e.g. n_heads).
    """
    mode, L, H, d, dt, seed, w, ck, gdiv = _SPECS[name]
    L_spec = L
    desc = describe(name, **desc_over)
    if layers is not None:
        desc["n_layers"] = L = int(layers)
    H, d = desc["n_heads"], desc["d_k"]
    lens = segment_lengths(name) if lengths is None else np.asarray(lengths, np.int64)
    seg_off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    N = int(seg_off[-1])
    if order is None:
        order = request_order(name) if lengths is None else np.arange(len(lens), dtype=np.int32)
    tdt = _TORCH_DTYPE[desc["in_dtype"]]
    dev = torch.device(device)
    conv = desc["conv_k"]
    q = torch.empty((L, N, H, d), dtype=tdt, device=dev)
    k = torch.empty_like(q)
    v = torch.empty_like(q)
    if mode == GATED_DELTA:
        alpha = torch.empty((L, N, H), dtype=tdt, device=dev)
        beta = torch.empty((L, N, H), dtype=tdt, device=dev)
    elif mode == DIAG_GATE:
        alpha = torch.empty((L, N, H, d), dtype=tdt, device=dev)
        beta = None
    elif mode == KDA:
        alpha = torch.empty((L, N, H, d), dtype=tdt, device=dev)
        beta = torch.empty((L, N, H), dtype=tdt, device=dev)
    else:
        alpha = torch.empty((L, H), dtype=tdt, device=dev)
        beta = None
    conv_w = torch.empty((L, 3, H, d, conv), dtype=torch.float32, device=dev) if conv else None
    for l in range(L):
        g = torch.Generator(device=dev)
        g.manual_seed(_layer_seed(name, seed, l, L_spec))
        for x, normed in ((q, True), (k, True), (v, False)):
            z = torch.randn((N, H, d), generator=g, device=dev, dtype=torch.float32)
            if normed and not conv:
                z = z / torch.linalg.vector_norm(z, dim=-1, keepdim=True)
            x[l].copy_(z)
            del z
        if mode == GATED_DELTA:
            z = torch.randn((N, H), generator=g, device=dev, dtype=torch.float32)
            sp = torch.nn.functional.softplus(z)
            alpha[l].copy_(torch.exp(-sp / gdiv) if gdiv > 0 else torch.ones_like(sp))
            z = torch.randn((N, H), generator=g, device=dev, dtype=torch.float32)
            beta[l].copy_(torch.sigmoid(z))
        elif mode == KDA:
            z = torch.randn((N, H, d), generator=g, device=dev, dtype=torch.float32)
            alpha[l].copy_(torch.exp(-torch.nn.functional.softplus(z) / gdiv))
            z = torch.randn((N, H), generator=g, device=dev, dtype=torch.float32)
            beta[l].copy_(torch.sigmoid(z))
        elif mode == DIAG_GATE:
            z = torch.randn((N, H, d), generator=g, device=dev, dtype=torch.float32)
            alpha[l].copy_(torch.exp(-torch.nn.functional.softplus(z)))
        else:
            hh = torch.arange(H, device=dev, dtype=torch.float64)
            alpha[l].copy_((1.0 - torch.pow(2.0, -5.0 - hh)).to(torch.float32))
        if conv:
            conv_w[l].copy_(torch.randn((3, H, d, conv), generator=g, device=dev,
                                        dtype=torch.float32) * 0.5)
    tok = dict(q=q, k=k, v=v, alpha=alpha, beta=beta, conv_w=conv_w)
    return Workload(name=name, desc=desc, seg_off=seg_off,
                    order=np.asarray(order, dtype=np.int32), tok=tok)
