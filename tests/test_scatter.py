"""Segment-level scatter / combine across ranks, on CPU: the LPT partition,
the packing of a worker's segments, and two gloo ranks that each build their
share of the pairs and stream them to the combine rank, which then holds the
pairs of the whole request and composes them.  The per-rank build function
here is the fp64 oracle (the GPU library plays that part on a GPU rank), so
the combined pairs must equal the single-process ones exactly."""
import os
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

from linear_attn_state_chunked_gb300 import scatter  # noqa: E402


def test_lpt_assign_by_hand():
    # 7 -> r0, 5 -> r1, 4 -> r1 (5 < 7), 3 -> r0 (7 < 9), 3 -> r1 (9 < 10), 2 -> r0 (10 < 12)
    owner = scatter.lpt_assign([7, 5, 4, 3, 3, 2], 2)
    assert owner.tolist() == [0, 1, 1, 0, 1, 0]
    rng = np.random.default_rng(3)
    for ranks in (2, 3, 8):
        work = rng.integers(64, 4097, size=200)
        owner = scatter.lpt_assign(work, ranks)
        loads = np.bincount(owner, weights=work, minlength=ranks)
        assert loads.max() - loads.min() <= work.max()  # LPT's guarantee
        assert sorted(set(owner.tolist())) == list(range(ranks))


def test_schedule_covers_every_segment_once():
    seg_off = np.concatenate([[0], np.cumsum([70, 9, 0, 300, 41, 8, 1000, 3, 64])])
    owner, plan = scatter.schedule(seg_off, 8, 3, 2)
    flat = [s for r in range(3) for b in plan[r] for s in b]
    assert sorted(flat) == list(range(len(seg_off) - 1))
    for r in range(3):
        assert all(owner[s] == r for b in plan[r] for s in b)
        assert all(len(b) <= 2 for b in plan[r])


def test_compact_request_packs_rows():
    L, N, H, d = 2, 30, 3, 4
    q = torch.arange(L * N * H * d, dtype=torch.float32).reshape(L, N, H, d)
    alpha = torch.arange(L * N * H, dtype=torch.float32).reshape(L, N, H)
    seg_off = [0, 10, 14, 30]
    tok, off = scatter.compact_request({"q": q, "alpha": alpha, "conv_w": None}, seg_off, [2, 0])
    assert off.tolist() == [0, 16, 26]
    assert torch.equal(tok["q"][:, :16], q[:, 14:30]) and torch.equal(tok["q"][:, 16:], q[:, 0:10])
    assert torch.equal(tok["alpha"][:, 16:], alpha[:, 0:10])


def _oracle_build(desc, tok, seg_off):
    """Pairs of every segment of a (compact) request from the fp64 oracle, laid
    out like the library writes them: T, S [L][n_seg][H][d][d] float32."""
    from oracle import reference as ref
    L, H, d = desc["n_layers"], desc["n_heads"], desc["d_k"]
    n = len(seg_off) - 1
    T = torch.zeros((L, n, H, d, d))
    S = torch.zeros((L, n, H, d, d))
    items = [(l, s, h) for l in range(L) for s in range(n) for h in range(H)]
    if items:
        Tr, Sr = ref.pair_reference(desc, tok, seg_off, items)
        for i, (l, s, h) in enumerate(items):
            T[l, s, h] = torch.from_numpy(Tr[i]).float()
            S[l, s, h] = torch.from_numpy(Sr[i]).float()
    return T, S


def _shapes(desc, n):
    L, H, d = desc["n_layers"], desc["n_heads"], desc["d_k"]
    return (L, n, H, d, d), (L, n, H, d, d)


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from linear_attn_state_chunked_gb300 import workloads as W
    import oracle
    from oracle import reference as ref
    lens = [70, 9, 0, 300, 41, 8, 120, 3, 64]
    wl = W.make("stress_tiny", device="cpu", lengths=lens, seam_w=8, n_heads=2, layers=2)
    res = scatter.scatter_build_combine(wl.desc, wl.tok, wl.seg_off, _oracle_build, _shapes, combine_rank=0,
                                        batch=2)
    if rank == 0:
        T, S = res
        T1, S1 = _oracle_build(wl.desc, wl.tok, wl.seg_off)
        out["pairs_equal"] = bool(torch.equal(T, T1) and torch.equal(S, S1))
        # the combine rank composes the gathered pairs (seams re-run from the
        # running state) and must land on the recurrence over the request
        d = wl.desc
        order = [int(s) for s in wl.order]
        chains = [(l, h) for l in range(d["n_layers"]) for h in range(d["n_heads"])]
        exp = ref.request_reference(d, wl.tok, wl.seg_off, order, chains)
        worst = 0.0
        for ci, (l, h) in enumerate(chains):
            idx = np.concatenate([np.arange(wl.seg_off[s], wl.seg_off[s + 1]) for s in order])
            q, k, v, a, b = ref.chain_stream(wl.tok, d["mode"], l, h, idx)
            starts = np.cumsum([0] + [int(wl.seg_off[s + 1] - wl.seg_off[s]) for s in order])
            Sx = np.zeros((1, d["d_k"], d["d_v"]))
            for e, s in enumerate(order):
                lo = starts[e]
                sw = min(d["seam_w"], starts[e + 1] - lo)
                Sx, _, _ = oracle.recurrence(d["mode"], q[None, lo:lo + sw], k[None, lo:lo + sw],
                                             v[None, lo:lo + sw], a[None, lo:lo + sw], b[None, lo:lo + sw],
                                             S0=Sx, want_o=True)
                Sx = oracle.compose(T[l, s, h].double().numpy()[None], S[l, s, h].double().numpy()[None], Sx)
            worst = max(worst, ref.rel_fro(Sx[0], exp["S_final"][ci]))
        out["final_err"] = worst
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_scatter_combine():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = 30500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    assert out["pairs_equal"]
    assert out["final_err"] < 1e-6, out["final_err"]
