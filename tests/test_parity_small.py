"""GPU parity on the small workloads and edge cases: every output block of
the C-ABI calls against the fp64 oracle, element by element."""
import numpy as np
import pytest
import torch

from linear_attn_state_chunked_gb300 import hypic, workloads as W
from oracle import reference as ref
from _parity import (run_pipeline, check_pairs, check_request, tol_of, alloc_outputs,
                     T_FLOOR)

pytestmark = pytest.mark.gpu


def _all_items(wl):
    d = wl.desc
    return [(l, s, h) for l in range(d["n_layers"]) for s in range(wl.n_seg)
            for h in range(d["n_heads"])]


def _all_chains(wl):
    d = wl.desc
    return [(l, h) for l in range(d["n_layers"]) for h in range(d["n_heads"])]


@pytest.mark.parametrize("name", ["tiny_gdn", "stress_tiny", "decay_retnet", "decay_diag", "deltanet",
                                  "kda_tiny", "kda_bf16"])
def test_small_workloads(name):
    """tiny_gdn: build per segment, compose in order, against the sequential
    recurrence over all 256 tokens; decay_*: scalar-decay and diagonal-gate
    specialisations; stress_tiny: slow gate so that T_C matters; deltanet:
    plain DeltaNet (alpha = 1); kda_*: the delta rule with a per-channel
    decay (fp32, and bf16 with conv warm-up and seams)."""
    wl = W.make(name, device="cuda")
    out = run_pipeline(wl)
    tol = tol_of(wl.desc)
    et, es = check_pairs(wl, out, _all_items(wl), tol)
    res = check_request(wl, out, _all_chains(wl), tol)
    print("\nparity %s: T %.2e  S %.2e  S_final %.2e  S_prefix %.2e  seam o %.2e  (tol %.0e)"
          % (name, et, es, res["final"], res["prefix"], res["o"], tol))
    if name == "stress_tiny":
        # the composition term is far from negligible here
        T = out["T"].cpu().numpy()
        assert np.abs(T).max() > 1e-3


@pytest.mark.parametrize("name", ["decay_retnet", "decay_diag", "stress_tiny", "kda_tiny"])
def test_naive_addition_is_wrong(name):
    """Negative control: summing the GPU's zero-initial states (dropping T)
    misses the recurrence by far more than the tolerance."""
    wl = W.make(name, device="cuda")
    out = run_pipeline(wl)
    S = out["S"].cpu().numpy()
    Sf = out["S_final"].cpu().numpy()
    tol = tol_of(wl.desc)
    errs = []
    for (l, h) in _all_chains(wl):
        naive = S[l, :, h].sum(axis=0)
        errs.append(ref.rel_fro(naive, Sf[l, h]))
    assert min(errs) > 100 * tol


EDGE_LENGTHS = [0, 1, 5, 8, 9, 70, 130, 3, 64, 65]
EDGE_ORDER = [5, 0, 9, 2, 2, 7, 1, 6, 3, 4, 8, 5]


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", [hypic.F32, hypic.BF16])
@pytest.mark.parametrize("mode", [hypic.GATED_DELTA, hypic.SCALAR_DECAY, hypic.DIAG_GATE, hypic.KDA])
def test_edge_cases_ragged_seams_order(d, dtype, mode):
    """Empty, one-token, shorter-than-seam and ragged segments, a shuffled
    request order with a repeated segment, seams of w = 8, two layers."""
    name = {hypic.GATED_DELTA: "stress_tiny", hypic.SCALAR_DECAY: "decay_retnet",
            hypic.DIAG_GATE: "decay_diag", hypic.KDA: "kda_tiny"}[mode]
    wl = W.make(name, device="cuda", layers=2, lengths=EDGE_LENGTHS, order=EDGE_ORDER,
                n_heads=2, d_k=d, d_v=d, seam_w=8, in_dtype=dtype)
    out = run_pipeline(wl)
    tol = tol_of(wl.desc)
    check_pairs(wl, out, _all_items(wl), tol)
    check_request(wl, out, _all_chains(wl), tol)


@pytest.mark.parametrize("d", [16, 64, 128])
def test_conv_warmup_small(d):
    """Causal conv (4 taps) with warm-up across segment boundaries, including
    segments shorter than the conv history, in a shuffled order."""
    wl = W.make("cold_30l", device="cuda", layers=2, lengths=[9, 40, 3, 1, 25, 12, 0, 17],
                order=[4, 2, 3, 0, 7, 5, 1, 6], n_heads=2, d_k=d, d_v=d)
    out = run_pipeline(wl)
    tol = tol_of(wl.desc)
    check_pairs(wl, out, _all_items(wl), tol)
    check_request(wl, out, _all_chains(wl), tol)


def test_nonzero_initial_state_and_empty_request():
    wl = W.make("stress_tiny", device="cuda", n_heads=3)
    d = wl.desc
    L, H, D = d["n_layers"], d["n_heads"], d["d_k"]
    g = torch.Generator(device="cuda").manual_seed(77)
    S0 = torch.randn((L, H, D, D), generator=g, device="cuda")
    out = alloc_outputs(d, wl.n_seg, len(wl.order))
    hypic.segment_build(d, wl.tok, wl.seg_off, out["T"], out["S"], out["ws"])
    hypic.compose(d, None, wl.seg_off, wl.order, out["T"], out["S"], out["S_final"],
                  S_init=S0, S_prefix_out=out["S_prefix"])
    torch.cuda.synchronize()
    chains = [(0, h) for h in range(H)]
    check_request(wl, out, chains, tol_of(d), S_init=S0[0].cpu().numpy())
    # empty request: S_final = S_init, in place
    Sx = S0.clone()
    hypic.compose(d, None, wl.seg_off, [], out["T"], out["S"], Sx, S_init=Sx)
    torch.cuda.synchronize()
    assert torch.equal(Sx, S0)
    Z = torch.full_like(S0, 5.0)
    hypic.compose(d, None, wl.seg_off, [], out["T"], out["S"], Z)
    torch.cuda.synchronize()
    assert torch.count_nonzero(Z).item() == 0


@pytest.mark.parametrize("conv", [False, True, "kda"])
def test_seam_advance_matches_compose(conv):
    """All seams in parallel from the prefix states equal the fused pass and
    the oracle; S_out may alias S_in."""
    if conv == "kda":
        wl = W.make("kda_bf16", device="cuda", layers=2, lengths=[9, 40, 3, 1, 25, 12, 17],
                    order=[4, 2, 3, 0, 5, 1, 6], n_heads=2, d_k=32, d_v=32)
    elif conv:
        wl = W.make("cold_30l", device="cuda", layers=2, lengths=[9, 40, 3, 1, 25, 12, 17],
                    order=[4, 2, 3, 0, 5, 1, 6], n_heads=2, d_k=32, d_v=32)
    else:
        wl = W.make("stress_tiny", device="cuda", lengths=EDGE_LENGTHS, order=EDGE_ORDER,
                    n_heads=2, seam_w=8, in_dtype=hypic.BF16, d_k=64, d_v=64)
    d = wl.desc
    out = run_pipeline(wl)
    o2 = torch.full_like(out["o"], float("nan"))
    S_after = out["S_prefix"].clone()
    hypic.seam_advance(d, wl.tok, wl.seg_off, wl.order, S_after, o2, S_out=S_after)
    torch.cuda.synchronize()
    tol = tol_of(d)
    if conv == "kda":
        # token by token in both calls: the same arithmetic
        assert torch.equal(o2, out["o"])
    else:
        # gated delta: one pass over the state per seam here, token by token
        # in the fused pass; the two agree to rounding
        assert not torch.isnan(o2).any()
        for l in range(d["n_layers"]):
            for e in range(len(wl.order)):
                for h in range(d["n_heads"]):
                    assert ref.rel_fro(o2[l, e, :, h].cpu().numpy(),
                                       out["o"][l, e, :, h].cpu().numpy()) <= tol
    # oracle: seams re-run from the oracle's own prefix states
    chains = [(l, h) for l in range(d["n_layers"]) for h in range(d["n_heads"])]
    exp = ref.request_reference(d, wl.tok, wl.seg_off, wl.order, chains)
    entries = list(range(len(wl.order)))
    Sa = S_after.cpu().numpy()
    for ci, (l, h) in enumerate(chains):
        o_ref, s_ref = ref.seam_reference(d, wl.tok, wl.seg_off, wl.order, [(l, h)],
                                          [exp["S_prefix"][ci]], entries)
        for e in entries:
            assert ref.rel_fro(Sa[l, e, h], s_ref[0, e]) <= tol
            assert ref.rel_fro(o2[l, e, :, h].cpu().numpy(), o_ref[0, e]) <= tol


@pytest.mark.parametrize("d,dtype,ck,w", [
    (16, hypic.F32, 0, 13), (32, hypic.F32, 4, 20), (64, hypic.BF16, 4, 8), (64, hypic.F32, 3, 9),
    (128, hypic.BF16, 4, 8), (128, hypic.F32, 0, 64), (128, hypic.BF16, 4, 17),
    (128, hypic.F32, 4, 3), (128, hypic.BF16, 0, 8), (128, hypic.F32, 2, 6), (128, hypic.BF16, 3, 8)])
@pytest.mark.parametrize("with_out", [False, True])
def test_seam_advance_from_given_states(d, dtype, ck, w, with_out):
    """Gated delta seams from random prefix states (not produced by compose)
    against the oracle's seam re-run from the same states: seams of up to 8
    tokens in one pass over the state and longer ones in several passes;
    empty, one-token and shorter-than-seam segments; a repeated segment;
    the conv history crossing several short entries."""
    _seam_from_states(d, dtype, ck, w, with_out)


@pytest.mark.parametrize("d,dtype,ck,w", [(128, hypic.BF16, 4, 8), (128, hypic.F32, 0, 5), (32, hypic.BF16, 4, 12)])
def test_seam_advance_in_place(d, dtype, ck, w):
    """S_out aliasing S_in (the state advanced in place) gives the same
    outputs and states as separate buffers."""
    over = dict(conv_k=ck) if ck else {}
    wl = W.make("cold_30l" if ck else "stress_tiny", device="cuda", layers=2, lengths=EDGE_LENGTHS,
                order=EDGE_ORDER, n_heads=2, d_k=d, d_v=d, seam_w=w, in_dtype=dtype, **over)
    desc = wl.desc
    L, H, n_ord = desc["n_layers"], desc["n_heads"], len(wl.order)
    g = torch.Generator(device="cuda").manual_seed(4242 + d)
    S_in = 0.5 * torch.randn((L, n_ord, H, d, d), generator=g, device="cuda")
    o1 = torch.empty((L, n_ord, w, H, d), device="cuda")
    S1 = torch.empty_like(S_in)
    hypic.seam_advance(desc, wl.tok, wl.seg_off, wl.order, S_in, o1, S_out=S1)
    S2 = S_in.clone()
    o2 = torch.empty_like(o1)
    hypic.seam_advance(desc, wl.tok, wl.seg_off, wl.order, S2, o2, S_out=S2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(S1, S2)


@pytest.mark.parametrize("d,dtype,ck,w", [(128, hypic.BF16, 4, 8), (64, hypic.F32, 3, 9)])
def test_seam_advance_conv_silu(d, dtype, ck, w):
    """The same with SiLU between the conv and the normalisation."""
    _seam_from_states(d, dtype, ck, w, True, act=hypic.ACT_SILU)


def _seam_from_states(d, dtype, ck, w, with_out, act=0):
    over = dict(conv_k=ck, conv_act=act) if ck else {}
    wl = W.make("cold_30l" if ck else "stress_tiny", device="cuda", layers=2, lengths=EDGE_LENGTHS,
                order=EDGE_ORDER, n_heads=2, d_k=d, d_v=d, seam_w=w, in_dtype=dtype, **over)
    desc = wl.desc
    L, H, n_ord = desc["n_layers"], desc["n_heads"], len(wl.order)
    g = torch.Generator(device="cuda").manual_seed(1000 + d + w)
    S_in = 0.5 * torch.randn((L, n_ord, H, d, d), generator=g, device="cuda")
    S_keep = S_in.clone()
    o = torch.full((L, n_ord, w, H, d), float("nan"), device="cuda")
    S_out = torch.full_like(S_in, float("nan")) if with_out else None
    hypic.seam_advance(desc, wl.tok, wl.seg_off, wl.order, S_in, o, S_out=S_out)
    torch.cuda.synchronize()
    assert torch.equal(S_in, S_keep)
    tol = tol_of(desc)
    chains = _all_chains(wl)
    Sn = S_in.cpu().numpy()
    entries = list(range(n_ord))
    on = o.cpu().numpy()
    Son = S_out.cpu().numpy() if with_out else None
    worst = 0.0
    for ci, (l, h) in enumerate(chains):
        o_ref, s_ref = ref.seam_reference(desc, wl.tok, wl.seg_off, wl.order, [(l, h)],
                                          [[Sn[l, e, h] for e in entries]], entries)
        for e in entries:
            err = ref.rel_fro(on[l, e, :, h], o_ref[0, e])
            worst = max(worst, err)
            assert err <= tol, ("o", l, e, h, err)
            if with_out:
                assert ref.rel_fro(Son[l, e, h], s_ref[0, e]) <= tol, ("S", l, e, h)
    print("\nseam advance d=%d w=%d: worst o %.2e (tol %.0e)" % (d, w, worst, tol))


@pytest.mark.parametrize("d,dtype", [(128, hypic.BF16), (64, hypic.BF16), (32, hypic.F32)])
def test_conv_silu(d, dtype):
    """Causal conv followed by SiLU before the L2 normalisation (the
    tensor-core path at d = 128 bf16, the CUDA-core path otherwise): every
    pair, and composition with seams, against the oracle; negative control:
    the oracle without the activation misses the GPU result by far more than
    the tolerance."""
    wl = W.make("cold_30l", device="cuda", layers=2, lengths=[9, 40, 3, 1, 25, 12, 0, 17, 300, 70],
                order=[4, 2, 3, 0, 7, 5, 1, 6, 8, 9], n_heads=2, d_k=d, d_v=d, in_dtype=dtype,
                conv_act=hypic.ACT_SILU)
    out = run_pipeline(wl)
    tol = tol_of(wl.desc)
    et, es = check_pairs(wl, out, _all_items(wl), tol)
    res = check_request(wl, out, _all_chains(wl), tol)
    print("\nconv+SiLU d=%d: T %.2e  S %.2e  S_final %.2e  seam o %.2e  (tol %.0e)"
          % (d, et, es, res["final"], res["o"], tol))
    plain = ref.request_reference(dict(wl.desc, conv_act=0), wl.tok, wl.seg_off, wl.order, [(1, 1)])
    assert ref.rel_fro(out["S_final"][1, 1].cpu().numpy(), plain["S_final"][0]) > 100 * tol


@pytest.mark.parametrize("name,over", [
    ("tiny_gdn", {}), ("decay_retnet", {}), ("decay_diag", {}), ("kda_tiny", {}), ("deltanet", {}),
    ("stress_tiny", dict(d_k=128, d_v=128, in_dtype=hypic.BF16, seam_w=8, n_heads=2)),
    ("cold_30l", dict(d_k=64, d_v=64, n_heads=2, conv_act=hypic.ACT_SILU))])
def test_segment_forward(name, over):
    """Per-token outputs of every segment body from a zero state against the
    oracle's prefill of that body; seam rows untouched; the pair written
    alongside equals the oracle's; without T and S the outputs are bitwise
    the same (the forward alone)."""
    kw = dict(over)
    if name in ("stress_tiny", "cold_30l"):
        kw.update(layers=2, lengths=EDGE_LENGTHS if name == "stress_tiny" else [9, 40, 3, 1, 25, 70, 0, 17],
                  order=EDGE_ORDER if name == "stress_tiny" else None)
    wl = W.make(name, device="cuda", **kw)
    d = wl.desc
    L, H, D, N = d["n_layers"], d["n_heads"], d["d_k"], wl.n_tokens
    o = torch.full((L, N, H, D), float("nan"), device="cuda")
    tshape, sshape = hypic.pair_shapes(d, wl.n_seg)
    T = torch.empty(tshape, device="cuda")
    S = torch.empty(sshape, device="cuda")
    hypic.segment_forward(d, wl.tok, wl.seg_off, o, T_out=T, S_out=S)
    o2 = torch.full_like(o, float("nan"))
    hypic.segment_forward(d, wl.tok, wl.seg_off, o2)
    torch.cuda.synchronize()
    assert torch.equal(torch.nan_to_num(o, nan=7.0), torch.nan_to_num(o2, nan=7.0))
    tol = tol_of(d)
    items = _all_items(wl)
    check_pairs(wl, {"T": T, "S": S}, items, tol)
    refs = ref.body_output_reference(d, wl.tok, wl.seg_off, items)
    on = o.cpu().numpy()
    worst = 0.0
    for (l, s, h), r in zip(items, refs):
        lo, hi = int(wl.seg_off[s]), int(wl.seg_off[s + 1])
        sw = min(d["seam_w"], hi - lo)
        assert np.isnan(on[l, lo:lo + sw, h]).all()  # seam rows untouched
        if len(r):
            err = ref.rel_fro(on[l, lo + sw:hi, h], r)
            worst = max(worst, err)
            assert err <= tol, (l, s, h, err)
    print("\nsegment forward %s: worst o %.2e (tol %.0e)" % (name, worst, tol))


@pytest.mark.parametrize("d,dtype", [(128, hypic.BF16), (32, hypic.F32)])
def test_maximum_segment_count(d, dtype):
    """The request table at its limit: as many segments as the library takes
    (0 to 40 tokens each: empty ones, ones shorter than the seam or the conv
    history) and a request order of the same length with repeats; every pair
    of two sampled heads' items, the two chains over the whole order (every
    prefix state, seam output and the final state), and all seams in
    parallel from the prefix states, against the oracle."""
    rng = np.random.default_rng(99)
    n = hypic.MAX_SEGMENTS
    lengths = rng.integers(0, 41, size=n)
    order = rng.integers(0, n, size=n).astype(np.int32)
    wl = W.make("cold_30l", device="cuda", layers=1, lengths=lengths, order=order, n_heads=2,
                d_k=d, d_v=d, in_dtype=dtype)
    out = run_pipeline(wl)
    tol = tol_of(wl.desc)
    pick = sorted(set([int(np.argmax(lengths)), int(np.argmin(lengths)), 0, n - 1] +
                      [int(x) for x in rng.integers(0, n, size=12)]))
    check_pairs(wl, out, [(0, s, h) for s in pick for h in range(2)], tol)
    res = check_request(wl, out, [(0, 0), (0, 1)], tol)
    o2 = torch.full_like(out["o"], float("nan"))
    hypic.seam_advance(wl.desc, wl.tok, wl.seg_off, wl.order, out["S_prefix"], o2)
    torch.cuda.synchronize()
    num = (o2.double() - out["o"].double()).pow(2).sum(dim=(2, 4)).sqrt()
    den = out["o"].double().pow(2).sum(dim=(2, 4)).sqrt()
    assert (torch.where(den > 0, num / den.clamp_min(1e-300), num) <= tol).all()
    print("\nmax segments d=%d: S_final %.2e  S_prefix %.2e  seam o %.2e" % (d, res["final"], res["prefix"], res["o"]))
