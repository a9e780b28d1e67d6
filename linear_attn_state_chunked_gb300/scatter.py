"""Segment-level scatter / combine of a cold request across ranks.

HYPIC pages (article “小红书联合北大、上交提出 HYPIC：混合注意力大模型首 Token
延迟降低 3.25 倍，实现位置无关缓存”, section "段并行"; article “Xiaohongshu,
Peking University, Shanghai Jiao Tong University Unveil HYPIC to Slash First
Token Latency by 3.25x in Hybrid Attention Models”, segment-level parallelism
paragraph): a router hands the cache-miss segments of a request to scatter
workers, balancing their load by longest-processing-time-first (LPT) on
segment length; each worker prefills its segments independently -- their
pairs depend on nothing outside the segment -- and the results stream to a
combine worker, which assembles the running state in request order while
later segments are still being computed.

This module is the host-side orchestration of that exchange and nothing
else: which rank builds which segment, the order in which batches of pairs
are sent and received, and where each lands in the combine rank's pair cache.
The pairs themselves come from a caller-supplied build function (the
library's ``hypic.segment_build`` on a GPU rank), and the exchange uses
``torch.distributed`` point-to-point calls, so it runs on any backend that
supports them.  The unit of work is a whole segment (all its layers and
heads), as the pages' segment-level parallelism assigns it.
"""
import numpy as np
import torch
import torch.distributed as dist


def body_lengths(seg_off, seam_w):
    """Tokens of each segment after its first min(w, len) seam tokens: the
    part whose pair a worker builds."""
    lens = np.diff(np.asarray(seg_off, dtype=np.int64))
    return lens - np.minimum(lens, seam_w)


def lpt_assign(work, n_ranks):
    """Greedy LPT: items in decreasing work (ties: lower index first), each to
    the rank with the least work so far (ties: lower rank).  Returns the rank
    of every item."""
    work = np.asarray(work, dtype=np.int64)
    order = sorted(range(len(work)), key=lambda i: (-int(work[i]), i))
    load = [0] * n_ranks
    owner = np.zeros(len(work), dtype=np.int64)
    for i in order:
        r = min(range(n_ranks), key=lambda k: (load[k], k))
        owner[i] = r
        load[r] += int(work[i])
    return owner


def schedule(seg_off, seam_w, n_ranks, batch):
    """The build and transfer plan every rank derives identically: for each
    rank, its segments longest body first, cut into batches of at most
    `batch` segments (a batch is built, then sent while the next is built)."""
    work = body_lengths(seg_off, seam_w)
    owner = lpt_assign(work, n_ranks)
    plan = []
    for r in range(n_ranks):
        mine = sorted((s for s in range(len(work)) if owner[s] == r), key=lambda s: (-int(work[s]), s))
        plan.append([mine[i:i + batch] for i in range(0, len(mine), batch)])
    return owner, plan


def compact_request(tok, seg_off, segs):
    """The token rows of segments `segs` (in that order) packed back to back,
    with their new offsets: the part of the request a scatter worker
    receives.  tok: dict of [L][N][H]... tensors (alpha of the scalar-decay
    mode, [L][H], and conv weights are passed through)."""
    rows = [(int(seg_off[s]), int(seg_off[s + 1])) for s in segs]
    idx = torch.cat([torch.arange(a, b, dtype=torch.long) for a, b in rows]) if rows else \
        torch.zeros(0, dtype=torch.long)
    out = {}
    for key, x in tok.items():
        if x is None or key == "conv_w" or x.dim() < 3:
            out[key] = x
        else:
            out[key] = x.index_select(1, idx.to(x.device)).contiguous()
    off = np.concatenate([[0], np.cumsum([b - a for a, b in rows])]).astype(np.int64)
    return out, off


def scatter_build_combine(desc, tok, seg_off, build_fn, pair_shapes, combine_rank=0, batch=4,
                          group=None, device="cpu"):
    """Build every segment's pair on the rank LPT assigns it to and gather the
    pairs on `combine_rank`.

    build_fn(desc, tok_compact, off_compact) -> (T, S), the pairs of the
    compact request's segments ([L][n][H]... as ``hypic.segment_build``
    writes them); pair_shapes(desc, n_seg) -> (T shape, S shape).  Each rank
    builds its batches in order and sends each one as soon as it is built
    (isend), so transfers overlap the next batch's build; the combine rank
    posts its receives in the same plan order and drops each batch into the
    request's segment slots.  Returns (T, S) of the whole request on the
    combine rank, None elsewhere.
    """
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    n_seg = len(seg_off) - 1
    _, plan = schedule(seg_off, desc["seam_w"], world, batch)
    # the combine rank posts every receive first, so that the other ranks'
    # batches land while it builds its own
    recvs = []
    if rank == combine_rank:
        for r in range(world):
            if r == combine_rank:
                continue
            for segs in plan[r]:
                tb, sb = pair_shapes(desc, len(segs))
                T = torch.empty(tb, dtype=torch.float32, device=device)
                S = torch.empty(sb, dtype=torch.float32, device=device)
                recvs.append((segs, T, S, dist.irecv(T, r, group=group), dist.irecv(S, r, group=group)))
    sends = []
    mine = []
    for segs in plan[rank]:
        t_c, off_c = compact_request(tok, seg_off, segs)
        T, S = build_fn(desc, t_c, off_c)
        if rank == combine_rank:
            mine.append((segs, T, S))
        else:
            T, S = T.contiguous(), S.contiguous()
            sends.append((dist.isend(T, combine_rank, group=group), dist.isend(S, combine_rank, group=group), T, S))
    if rank != combine_rank:
        for rq in sends:
            rq[0].wait()
            rq[1].wait()
        return None
    tshape, sshape = pair_shapes(desc, n_seg)
    T_all = torch.empty(tshape, dtype=torch.float32, device=device)
    S_all = torch.empty(sshape, dtype=torch.float32, device=device)
    for segs, T, S in mine:
        T_all[:, segs] = T
        S_all[:, segs] = S
    for segs, T, S, rq_t, rq_s in recvs:
        rq_t.wait()
        rq_s.wait()
        T_all[:, segs] = T
        S_all[:, segs] = S
    return T_all, S_all
