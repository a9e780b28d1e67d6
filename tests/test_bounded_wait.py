"""Failure detection without a fault: the bounded device-side wait that the
pipelined kernels use gives up on a barrier that nothing completes, reports
through the workspace status word, lets a second waiter leave on the CTA's
abort flag, and leaves the device usable."""
import time

import pytest
import torch

from linear_attn_state_chunked_gb300 import hypic, workloads as W
from _parity import run_pipeline, check_pairs, tol_of

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    max_cycles = 20_000_000  # ~10 ms; the second waiter's own limit is 64x that (~0.6 s)
    hypic.selftest_bounded_wait(ws, 1000)  # load the module before timing
    with pytest.raises(hypic.HypicError):
        hypic.workspace_status(ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    hypic.selftest_bounded_wait(ws, max_cycles)
    with pytest.raises(hypic.HypicError) as ei:
        hypic.workspace_status(ws)
    dt = time.perf_counter() - t0
    assert ei.value.status == 7 and "status 3" in str(ei.value), str(ei.value)
    assert dt < 0.3, dt  # the second waiter left on the flag, not on its own limit

    # the device is still usable, and the next build on the workspace clears the word
    wl = W.make("tiny_gdn", device="cuda")
    d = wl.desc
    tshape, sshape = hypic.pair_shapes(d, wl.n_seg)
    T = torch.empty(tshape, device="cuda")
    S = torch.empty(sshape, device="cuda")
    hypic.segment_build(d, wl.tok, wl.seg_off, T, S, ws)
    hypic.workspace_status(ws)
    out = run_pipeline(wl)
    items = [(l, s, h) for l in range(d["n_layers"]) for s in range(wl.n_seg) for h in range(d["n_heads"])]
    check_pairs(wl, out, items, tol_of(d))
    assert torch.equal(out["T"], T) and torch.equal(out["S"], S)


def test_async_status_reports_and_clears():
    """Calls without a workspace (compose, seam advance) report a bounded wait
    that gave up through the device's status word: the self-test writes into
    it, the query raises HYPIC_ERR_TIMEOUT once and clears it, and a compose
    afterwards leaves it clear."""
    try:  # whatever an earlier call left is reported once and cleared
        hypic.async_status()
    except hypic.HypicError:
        pass
    try:
        hypic.async_status()
    except hypic.HypicError:
        pytest.fail("the first query did not clear the word")
    hypic.selftest_bounded_wait(None, 20_000_000)
    with pytest.raises(hypic.HypicError) as ei:
        hypic.async_status()
    assert ei.value.status == 7 and "status 3" in str(ei.value), str(ei.value)
    hypic.async_status()  # cleared by the query above
    out = run_pipeline(W.make("stress_tiny", device="cuda", seam_w=8, in_dtype=W.BF16, d_k=128, d_v=128,
                              n_heads=2, lengths=[64, 9, 40, 64], order=[2, 0, 3, 1]))
    assert torch.isfinite(out["S_final"]).all()
    hypic.async_status()
