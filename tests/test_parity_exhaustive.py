"""GPU parity on EVERY block, not a sample: each (layer, segment, head) pair
of a build, and each chain of a request, against the fp64 oracle.

* stress_gdn  -- the gated-delta bf16 shape (32 heads, d = 128, 64 segments of
  512-2048 tokens) under the slow gate, where T_C stays far from zero: every
  one of its 2,048 pairs, and every chain of the request (prefix states,
  seam outputs, final state).
* stress_cold -- the cold prompt's shape (200 lognormal segments up to 4,096
  tokens, causal conv of 4 taps) under the slow gate, 2 layers: every pair.
* cold_30l    -- the full 30-layer cold prompt built in the launch the
  benchmark times; every pair of its first and last layers.

The oracle runs all heads of one segment in one call (independent chains in
parallel on the host cores)."""
import numpy as np
import pytest
import torch

from linear_attn_state_chunked_gb300 import hypic, workloads as W
from oracle import reference as ref
from _parity import run_pipeline, check_request, tol_of, T_FLOOR, Worst

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _all_pairs(wl, out, layers):
    """Max relative Frobenius error of T and of S over every pair of `layers`."""
    d = wl.desc
    wt, ws_ = Worst(), Worst()
    for l in layers:
        arrs = ref.layer_arrays(wl.tok, l)
        T = out["T"][l].cpu().numpy()
        S = out["S"][l].cpu().numpy()
        for s in range(wl.n_seg):
            Tr, Sr = ref.segment_pairs(d, arrs, wl.seg_off, s)
            for h in range(d["n_heads"]):
                wt.add(ref.rel_fro(T[s, h], Tr[h], T_FLOOR), ("T", l, s, h))
                ws_.add(ref.rel_fro(S[s, h], Sr[h]), ("S", l, s, h))
        del arrs, T, S
    return wt, ws_


@pytest.mark.parametrize("name", ["stress_gdn", "stress_cold"])
def test_every_pair_slow_gate(name):
    wl = W.make(name, device="cuda")
    out = run_pipeline(wl, prefix=True)
    tol = tol_of(wl.desc)
    for key in ("T", "S", "S_final", "S_prefix", "o"):
        assert torch.isfinite(out[key]).all(), key
    # the slow gate keeps T_C well away from zero, so T is really compared
    assert out["T"].abs().amax().item() > 1e-5
    wt, ws_ = _all_pairs(wl, out, range(wl.desc["n_layers"]))
    msg = "\nevery pair of %s (%d): T %.3e at %s, S %.3e at %s (tol %.0e)" % (
        name, wl.desc["n_layers"] * wl.n_seg * wl.desc["n_heads"], wt.err, wt.where, ws_.err,
        ws_.where, tol)
    if name == "stress_gdn":
        chains = [(0, h) for h in range(wl.desc["n_heads"])]
        r = check_request(wl, out, chains, tol)
        msg += "; every chain: S_final %.3e, S_prefix %.3e, seam o %.3e" % (
            r["final"], r["prefix"], r["o"])
    print(msg)
    wt.check(tol, "T")
    ws_.check(tol, "S")


def test_every_pair_cold_first_last_layer():
    wl = W.make("cold_30l", device="cuda")
    out = run_pipeline(wl, prefix=False)
    L = wl.desc["n_layers"]
    tol = tol_of(wl.desc)
    assert torch.isfinite(out["T"]).all() and torch.isfinite(out["S"]).all()
    wt, ws_ = _all_pairs(wl, out, (0, L - 1))
    print("\nevery pair of cold_30l layers 0 and %d (%d): T %.3e at %s, S %.3e at %s (tol %.0e)"
          % (L - 1, 2 * wl.n_seg * wl.desc["n_heads"], wt.err, wt.where, ws_.err, ws_.where, tol))
    wt.check(tol, "T")
    ws_.check(tol, "S")
