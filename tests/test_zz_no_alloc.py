"""The allocation-free segment build (hypic_segment_build_noalloc) gives the
same pairs as hypic_segment_build.

That entry point exists for callers that may not allocate device memory (for
instance a plugin inside a host inference engine that owns every device
buffer, or a latency-critical path that must not call cudaMalloc): it runs
the build on a scratch block compiled into the library instead of a
caller-provided workspace.  Two calls in a row on different requests check
that the shared scratch carries nothing over from one call to the next.

This file is named so that pytest collects it last; it also passes when run
alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from linear_attn_state_chunked_gb300 import hypic, workloads as W
from oracle import reference as ref
from _parity import tol_of, T_FLOOR

pytestmark = pytest.mark.gpu


def _requests():
    # gated delta, bf16, d = 128 (tensor-core build), slow gate, ragged segments
    yield W.make("stress_gdn", device="cuda", lengths=[700, 64, 9, 0, 130, 1500, 3],
                 n_heads=4)
    # the conv workload shape (conv warm-up in the bodies), two layers
    yield W.make("cold_30l", device="cuda", layers=2, lengths=[300, 40, 1000, 8, 77],
                 n_heads=3)


def _pairs(wl, fn):
    tshape, sshape = hypic.pair_shapes(wl.desc, wl.n_seg)
    T = torch.full(tshape, float("nan"), device="cuda")
    S = torch.full(sshape, float("nan"), device="cuda")
    fn(T, S)
    torch.cuda.synchronize()
    return T.cpu().numpy(), S.cpu().numpy()


def test_noalloc_build_matches_workspace_build_twice():
    for wl in _requests():
        d = wl.desc
        ws = torch.empty(hypic.workspace_size(d), dtype=torch.uint8, device="cuda")
        T0, S0 = _pairs(wl, lambda T, S: hypic.segment_build(d, wl.tok, wl.seg_off, T, S, ws))
        T1, S1 = _pairs(wl, lambda T, S: hypic.segment_build_noalloc(d, wl.tok, wl.seg_off, T, S))
        hypic.noalloc_status()  # raises if a device-side wait of that build gave up
        hypic.workspace_status(ws)
        assert np.isfinite(T1).all() and np.isfinite(S1).all()
        tol = tol_of(d)
        worst = 0.0
        for l in range(d["n_layers"]):
            for s in range(wl.n_seg):
                for h in range(d["n_heads"]):
                    worst = max(worst, ref.rel_fro(T1[l, s, h], T0[l, s, h], T_FLOOR),
                                ref.rel_fro(S1[l, s, h], S0[l, s, h]))
        assert worst <= tol, worst
