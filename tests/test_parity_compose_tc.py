"""GPU parity of the tensor-core compose path (gated delta, bf16, d = 128)
on the branches the benchmark workloads do not reach: a nonzero initial
state with prefix states, no seams (w = 0), seams shorter than the window
and than the conv history, segments shorter than the seam, repeated and
shuffled request entries, and the empty request."""
import numpy as np
import pytest
import torch

from linear_attn_state_chunked_gb300 import hypic, workloads as W
from oracle import reference as ref
from _parity import check_pairs, check_request, tol_of, alloc_outputs

pytestmark = pytest.mark.gpu

LENGTHS = [0, 1, 2, 3, 5, 8, 9, 64, 65, 130, 300]
ORDER = [4, 0, 10, 2, 2, 7, 1, 9, 3, 6, 5, 8, 4]


def _items(wl):
    d = wl.desc
    return [(l, s, h) for l in range(d["n_layers"]) for s in range(wl.n_seg) for h in range(d["n_heads"])]


def _chains(wl):
    d = wl.desc
    return [(l, h) for l in range(d["n_layers"]) for h in range(d["n_heads"])]


def _run(wl, S0=None):
    d = wl.desc
    out = alloc_outputs(d, wl.n_seg, len(wl.order))
    hypic.segment_build(d, wl.tok, wl.seg_off, out["T"], out["S"], out["ws"])
    hypic.compose(d, wl.tok, wl.seg_off, wl.order, out["T"], out["S"], out["S_final"],
                  S_init=S0, S_prefix_out=out["S_prefix"], o_out=out["o"])
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("w,conv", [(8, 4), (8, 0), (3, 4), (5, 0), (0, 0)])
def test_tc_compose_branches(w, conv):
    base = "cold_30l" if conv else "stress_gdn"
    wl = W.make(base, device="cuda", layers=2, lengths=LENGTHS, order=ORDER, n_heads=3,
                seam_w=w)
    d = wl.desc
    assert d["d_k"] == 128 and d["in_dtype"] == hypic.BF16
    g = torch.Generator(device="cuda").manual_seed(11)
    S0 = 0.3 * torch.randn((d["n_layers"], d["n_heads"], 128, 128), generator=g, device="cuda")
    out = _run(wl, S0)
    tol = tol_of(d)
    check_pairs(wl, out, _items(wl), tol)
    res = [check_request(wl, out, [(l, h)], tol, S_init=[S0[l, h].cpu().numpy()])
           for (l, h) in _chains(wl)]
    print("\ncompose tc w=%d conv=%d: worst S_final %.2e S_prefix %.2e o %.2e" % (
        w, conv, max(r["final"] for r in res), max(r["prefix"] for r in res),
        max(r["o"] for r in res)))


def test_tc_compose_empty_request():
    wl = W.make("stress_gdn", device="cuda", lengths=[40, 70], n_heads=2)
    d = wl.desc
    out = alloc_outputs(d, wl.n_seg, 1)
    hypic.segment_build(d, wl.tok, wl.seg_off, out["T"], out["S"], out["ws"])
    S0 = torch.randn((1, 2, 128, 128), device="cuda")
    Sf = torch.full_like(S0, float("nan"))
    hypic.compose(d, wl.tok, wl.seg_off, [], out["T"], out["S"], Sf, S_init=S0)
    torch.cuda.synchronize()
    assert torch.equal(Sf, S0)
    Z = torch.full_like(S0, 7.0)
    hypic.compose(d, wl.tok, wl.seg_off, [], out["T"], out["S"], Z)
    torch.cuda.synchronize()
    assert torch.count_nonzero(Z).item() == 0


@pytest.mark.parametrize("case", ["big_state", "tiny_state", "scaled_qk"])
def test_tc_compose_far_from_unit_scale(case):
    """Requests whose state or seam operands sit far from unit scale, where
    a tensor-core operand format with a narrow exponent range would lose
    precision or overflow: a state of order 1e5 (until the decays bring it
    back), a request whose values and state are all of order 1e-6, and,
    without the conv (so q and k reach the seams unnormalised), q of order
    1e3 and k of order 1e-2."""
    conv = case != "scaled_qk"
    base = "cold_30l" if conv else "stress_gdn"
    wl = W.make(base, device="cuda", layers=1, lengths=LENGTHS, order=ORDER, n_heads=3)
    d = wl.desc
    g = torch.Generator(device="cuda").manual_seed(12)
    S0 = torch.randn((d["n_layers"], d["n_heads"], 128, 128), generator=g, device="cuda")
    if case == "big_state":
        S0 *= 1e5
    elif case == "tiny_state":
        S0 *= 1e-6
        wl.tok["v"].mul_(1e-6)
    else:
        wl.tok["q"].mul_(1e3)
        wl.tok["k"].mul_(1e-2)
    out = _run(wl, S0)
    res = [check_request(wl, out, [(l, h)], tol_of(d), S_init=[S0[l, h].cpu().numpy()])
           for (l, h) in _chains(wl)]
    print("\ncompose tc %s: worst S_final %.2e S_prefix %.2e o %.2e" % (
        case, max(r["final"] for r in res), max(r["prefix"] for r in res), max(r["o"] for r in res)))
