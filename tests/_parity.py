"""Shared helpers of the GPU parity tests: run the hot path through the C ABI
and compare it block by block with the fp64 oracle.

Error metric: for every compared block X (one T_C, one S(C|0), one prefix or
final state of a (layer, head), or one seam's outputs [w, d_v]) the relative
Frobenius error |X - X_ref|_F / max(|X_ref|_F, floor); floor = 1e-30 for T
(the fp32 pair underflows to zero where the fp64 one is ~1e-45 or smaller),
0 elsewhere.  The bar is the maximum over blocks: 1e-5 for fp32 inputs, 2e-3
for bf16 inputs with fp32 state.
"""
import numpy as np
import torch

from linear_attn_state_chunked_gb300 import hypic
from oracle import reference as ref

TOL = {hypic.F32: 1e-5, hypic.BF16: 2e-3}
T_FLOOR = 1e-30


def tol_of(desc):
    return TOL[desc["in_dtype"]]


def alloc_outputs(desc, n_seg, n_order, device="cuda", prefix=True):
    L, H, D, w = desc["n_layers"], desc["n_heads"], desc["d_k"], desc["seam_w"]
    tshape, sshape = hypic.pair_shapes(desc, n_seg)
    f32 = dict(dtype=torch.float32, device=device)
    out = dict(T=torch.full(tshape, float("nan"), **f32),
               S=torch.full(sshape, float("nan"), **f32),
               S_final=torch.full((L, H, D, D), float("nan"), **f32),
               ws=torch.empty(hypic.workspace_size(desc), dtype=torch.uint8, device=device))
    out["S_prefix"] = torch.full((L, n_order, H, D, D), float("nan"), **f32) if prefix else None
    out["o"] = torch.full((L, n_order, max(w, 1), H, D), float("nan"), **f32) if w else None
    return out


def run_pipeline(wl, prefix=True, device="cuda"):
    """Build every pair, then compose the request with fused seams."""
    out = alloc_outputs(wl.desc, wl.n_seg, len(wl.order), device, prefix)
    hypic.segment_build(wl.desc, wl.tok, wl.seg_off, out["T"], out["S"], out["ws"])
    hypic.compose(wl.desc, wl.tok, wl.seg_off, wl.order, out["T"], out["S"], out["S_final"],
                  S_prefix_out=out["S_prefix"], o_out=out["o"])
    torch.cuda.synchronize()
    return out


def dense_T(desc, T):
    """GPU T block (dense / diagonal / scalar) as a dense numpy matrix."""
    T = np.asarray(T, dtype=np.float64)
    D = desc["d_k"]
    if desc["mode"] in (hypic.GATED_DELTA, hypic.KDA):
        return T
    if desc["mode"] == hypic.DIAG_GATE:
        return np.diag(T)
    return float(T) * np.eye(D)


class Worst:
    def __init__(self):
        self.err, self.where = 0.0, None

    def add(self, err, where):
        if not np.isfinite(err) or err > self.err:
            self.err, self.where = (err if np.isfinite(err) else float("inf")), where

    def check(self, tol, what=""):
        assert self.err <= tol, "%s max rel Frobenius error %.3e > %.1e at %s" % (
            what, self.err, tol, self.where)
        return self.err


def check_pairs(wl, out, items, tol):
    """Compare T/S of each (l, s, h) in items with the oracle's pair."""
    Tref, Sref = ref.pair_reference(wl.desc, wl.tok, wl.seg_off, items)
    T = out["T"].cpu().numpy()
    S = out["S"].cpu().numpy()
    wt, ws_ = Worst(), Worst()
    for i, (l, s, h) in enumerate(items):
        if wl.desc["mode"] == hypic.GATED_DELTA:
            tg = T[l, s, h]
        elif wl.desc["mode"] == hypic.DIAG_GATE:
            tg = T[l, s, h]
        else:
            tg = T[l, s, h]
        wt.add(ref.rel_fro(dense_T(wl.desc, tg), Tref[i], T_FLOOR), ("T", l, s, h))
        ws_.add(ref.rel_fro(S[l, s, h], Sref[i]), ("S", l, s, h))
    return wt.check(tol, "T"), ws_.check(tol, "S")


def check_request(wl, out, chains, tol, S_init=None):
    """Compare prefix states, seam outputs and the final state of each chain."""
    exp = ref.request_reference(wl.desc, wl.tok, wl.seg_off, wl.order, chains, S_init=S_init)
    Sf = out["S_final"].cpu().numpy()
    Sp = out["S_prefix"].cpu().numpy() if out.get("S_prefix") is not None else None
    o = out["o"].cpu().numpy() if out.get("o") is not None else None
    wf, wp, wo = Worst(), Worst(), Worst()
    for ci, (l, h) in enumerate(chains):
        wf.add(ref.rel_fro(Sf[l, h], exp["S_final"][ci]), ("S_final", l, h))
        for e in range(len(wl.order)):
            if Sp is not None:
                wp.add(ref.rel_fro(Sp[l, e, h], exp["S_prefix"][ci, e]), ("S_prefix", l, e, h))
            if o is not None:
                wo.add(ref.rel_fro(o[l, e, :, h, :], exp["o_seam"][ci, e]), ("o", l, e, h))
    return dict(final=wf.check(tol, "S_final"), prefix=wp.check(tol, "S_prefix"),
                o=wo.check(tol, "seam o"), exp=exp)
