"""The oracle's layout helpers (oracle.reference) agree with the composition
law and with one another on tiny seeded workloads, including seams, a random
request order, a causal conv and ragged / empty / shorter-than-seam segments.
CPU only."""
import numpy as np
import pytest

import oracle
from oracle import reference as ref
from linear_attn_state_chunked_gb300 import workloads as W


def _pairs_all(wl, l, h):
    items = [(l, s, h) for s in range(wl.n_seg)]
    return ref.pair_reference(wl.desc, wl.tok, wl.seg_off, items)


@pytest.mark.parametrize("name,over", [
    ("tiny_gdn", {}),
    ("stress_tiny", {}),
    ("decay_retnet", dict(n_heads=2, d_k=8, d_v=8)),
    ("decay_diag", dict(n_heads=2, d_k=8, d_v=8)),
    ("stress_tiny", dict(seam_w=5)),
    ("cold_30l", dict(n_heads=2, d_k=8, d_v=8)),
])
def test_request_equals_composed_pairs(name, over):
    lengths = None
    order = None
    if name == "cold_30l":
        lengths = [9, 40, 3, 0, 25, 12]
    elif "seam_w" in over:
        lengths = [20, 3, 0, 31, 8, 17]
        order = [3, 0, 5, 1, 2, 4, 0]
    wl = W.make(name, layers=1, lengths=lengths, order=order, **over)
    d, w = wl.desc, wl.desc["seam_w"]
    chains = [(0, h) for h in range(d["n_heads"])]
    out = ref.request_reference(d, wl.tok, wl.seg_off, wl.order, chains)
    for ci, (l, h) in enumerate(chains):
        T, S = _pairs_all(wl, l, h)
        state = np.zeros((d["d_k"], d["d_v"]))
        for e, s in enumerate(wl.order):
            np.testing.assert_allclose(out["S_prefix"][ci, e], state, atol=1e-11, rtol=0)
            if w:
                o, Sw = ref.seam_reference(d, wl.tok, wl.seg_off, wl.order, [(l, h)],
                                           [[state]], [e])
                np.testing.assert_allclose(o[0, 0], out["o_seam"][ci, e], atol=1e-11, rtol=0)
                state = Sw[0, 0]
            state = oracle.compose(T[s][None], S[s][None], state[None])[0]
        np.testing.assert_allclose(out["S_final"][ci], state, atol=1e-11, rtol=0)


def test_workload_shapes_and_recipes():
    wl = W.make("tiny_gdn")
    assert wl.tok["k"].shape == (1, 256, 1, 16)
    kn = np.linalg.norm(wl.tok["k"].numpy(), axis=-1)
    np.testing.assert_allclose(kn, 1.0, rtol=1e-5)
    a = wl.tok["alpha"].numpy()
    assert np.all((a > 0) & (a < 1))
    r = W.make("decay_retnet")
    np.testing.assert_array_equal(r.tok["alpha"][0].numpy(),
                                  (1.0 - 2.0 ** (-5.0 - np.arange(8))).astype(np.float32))
    assert W.segment_lengths("cold_30l").sum() == 100_000
    assert W.segment_lengths("cold_30l").min() >= 64
    assert W.segment_lengths("warm_30l").sum() == 100_000
    assert len(W.segment_lengths("warm_30l")) == 128
    l2 = W.segment_lengths("gdn_bf16")
    assert len(l2) == 64 and l2.min() >= 512 and l2.max() <= 2048
    # per-layer seeds: a prefix of the stack equals the full stack's first layers
    a2 = W.make("cold_30l", layers=2, lengths=[10, 6], n_heads=1, d_k=8, d_v=8)
    a1 = W.make("cold_30l", layers=1, lengths=[10, 6], n_heads=1, d_k=8, d_v=8)
    assert np.array_equal(a2.tok["k"][0].float().numpy(), a1.tok["k"][0].float().numpy())
    assert not np.array_equal(a2.tok["k"][1].float().numpy(), a1.tok["k"][0].float().numpy())
