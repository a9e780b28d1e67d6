"""Benchmark of the linear-attention PIC hot path on one GB300.

A step is one pass of the whole hot path over the cold 100k-token prompt of a
30-layer stack (32 heads, d = 128, bf16 q/k/v/alpha/beta, fp32 state, causal
conv of 4 taps, w = 8, 200 lognormal segments, all cache misses):

  1. hypic_segment_build -- the (T_C, S(C|0)) pair of every segment body x
     layer x head, conv warm-up inside each body, one launch;
  2. hypic_compose       -- the running state over the request, every seam
     re-run under its prefix (conv warm-up across segment boundaries), one
     launch.

value = tokens x layers processed per second (Mtok/s, all heads), inputs
resident in HBM.  The JSON line also carries each call's own throughput
(build Mtok/s, compose segs/s), the dominant kernel's roofline, an end-to-end
figure through the C ABI from pinned host buffers, SM clocks sampled during
the timed region, and the fp64 oracle timed on the host cores on a bounded
sample of the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the fp64 CPU oracle (the only other implementation of
this path) on a bounded sample of the same workload, per step.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "cold_30l"
# the fp64 oracle's bounded sample, the same in both of its legs (the GPU arm's
# cpu_baseline and --impl reference): layer 0, every head, the request's first
# ORACLE_SEGS segments (~19k tokens of the cold prompt, a few seconds per run)
ORACLE_HEADS, ORACLE_SEGS = 32, 40
METRIC = "segment-build Mtok/s and compose segs/s per layer, % of roofline (1 GB300)"
UNIT = "Mtok/s"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16=d["bf16_tflops"],
                    bf16_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    sm_max_mhz=d.get("sm_max_mhz", 2070.0), source="measured")
    return dict(hbm_gbs=6800.0, bf16=1900.0, bf16_sustained=1700.0, sm_max_mhz=2070.0,
                source="fallback")


# DRAM bytes of one build launch on the 1-layer case (dram__bytes.sum.per_second
# x gpu__time_duration.sum of one ncu capture: 1.492755 TB/s x 1.689440 ms),
# and the SHA-256 of the kernel source they were taken on; reported only while
# the source is unchanged.
BUILD_TRAFFIC = {"source_sha256": "7abc9020af409a1d75cab0afe8e4639c0488548d2f9336e5422365a0ca9d12a2",
                 "bytes_per_layer": 2521920007}


def _build_traffic(n_layers):
    import hashlib
    src = os.path.join(ROOT, "linear_attn_state_chunked_gb300", "csrc", "build_tc.cu")
    with open(src, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    if BUILD_TRAFFIC["source_sha256"] != sha or BUILD_TRAFFIC["bytes_per_layer"] is None:
        return None
    return BUILD_TRAFFIC["bytes_per_layer"] * n_layers


def _config():
    from linear_attn_state_chunked_gb300 import workloads as W
    d = W.describe(WORKLOAD)
    lens = W.segment_lengths(WORKLOAD)
    n = int(lens.sum())
    in_bytes = d["n_layers"] * n * d["n_heads"] * (3 * d["d_k"] * 2 + 2 * 2)
    return {
        "workload": "cold_30l: cold 100k-token prompt, %d layers x %d heads, d_k=d_v=%d, "
                    "%d lognormal segments (median %d, clipped [64,4096], sum %d), "
                    "causal conv %d taps, seam w=%d, bf16 q/k/v/alpha/beta, fp32 state; "
                    "step = batched build of every segment pair + compose with fused seams"
                    % (d["n_layers"], d["n_heads"], d["d_k"], len(lens), int(np.median(lens)), n,
                       d["conv_k"], d["seam_w"]),
        "tokens": n, "layers": d["n_layers"], "heads": d["n_heads"], "d": d["d_k"],
        "segments": int(len(lens)),
        "l2": "inputs larger than L2 (%.1f GB of token inputs per step)" % (in_bytes / 1e9),
    }


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _reduce_max(x, ws):
    """Max of x over the ranks (each rank times its own replica; the job's
    time is the slowest rank's)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------
# fp64 oracle on a bounded sample (cpu_baseline leg and --impl reference)

def oracle_sample(wl, n_heads, n_segments):
    """Time the oracle on layer 0, heads [0, n_heads), the first n_segments of
    the request: conv + normalisation, every body pair, the compose chain and
    every seam.  Returns (seconds, layer-tokens covered)."""
    import oracle
    from oracle import reference as ref
    d = wl.desc
    order = [int(s) for s in wl.order[:n_segments]]
    off = wl.seg_off
    idx = np.concatenate([np.arange(off[s], off[s + 1]) for s in order])
    starts = np.cumsum([0] + [int(off[s + 1] - off[s]) for s in order])
    # inputs leave the device before the clock starts
    cpu_tok = {k: (None if v is None else v.detach().cpu()) for k, v in wl.tok.items()}
    w = d["seam_w"]
    t0 = time.perf_counter()
    streams = [ref.chain_stream(cpu_tok, d["mode"], 0, h, idx, d["conv_k"], d.get("conv_act", 0)) for h in range(n_heads)]
    q, k, v, a = (np.stack([s[i] for s in streams]) for i in range(4))
    b = np.stack([s[4] for s in streams])
    C, D = n_heads, d["d_k"]
    S = np.zeros((C, D, D))
    for e in range(len(order)):
        lo, hi = starts[e], starts[e + 1]
        sw = min(w, hi - lo)
        S, _, _ = oracle.recurrence(d["mode"], q[:, lo:lo + sw], k[:, lo:lo + sw], v[:, lo:lo + sw],
                                    a[:, lo:lo + sw], b[:, lo:lo + sw], S0=S, want_o=True)
        T, Sc = oracle.pair(d["mode"], k[:, lo + sw:hi], v[:, lo + sw:hi], a[:, lo + sw:hi],
                            b[:, lo + sw:hi])
        S = oracle.compose(T, Sc, S)
    dt = time.perf_counter() - t0
    layer_tokens = len(idx) * n_heads / d["n_heads"]
    return dt, layer_tokens


def _compose_bytes(wl):
    """Algorithmic bytes of one compose with fused seams: every entry's pair
    read (T and S, fp32), each seam token's raw q, k, v (bf16) and gates read
    and its fp32 outputs written, the final state written."""
    d = wl.desc
    L, H, D, w = d["n_layers"], d["n_heads"], d["d_k"], d["seam_w"]
    n_ord = len(wl.order)
    pair_bytes = L * n_ord * H * 2 * D * D * 4
    seam_tok = int(sum(min(w, int(wl.lengths[s])) for s in wl.order))
    seam_bytes = L * seam_tok * H * (3 * D * 2 + 2 * 2 + D * 4)
    return pair_bytes, pair_bytes + seam_bytes + L * H * D * D * 4


def _config_leg(name, args, peaks, dev, stream):
    """Build, compose with seams and compose alone on one named workload, each
    timed with CUDA events over repeated calls (inputs larger than L2)."""
    import torch
    from linear_attn_state_chunked_gb300 import hypic, workloads as W
    wl = W.make(name, device=dev)
    d = wl.desc
    L, H, D, w = d["n_layers"], d["n_heads"], d["d_k"], d["seam_w"]
    n_ord = len(wl.order)
    tshape, sshape = hypic.pair_shapes(d, wl.n_seg)
    T = torch.empty(tshape, device=dev)
    S = torch.empty(sshape, device=dev)
    Sf = torch.empty((L, H, D, D), device=dev)
    o = torch.empty((L, n_ord, max(w, 1), H, D), device=dev)
    wsp = torch.empty(hypic.workspace_size(d), dtype=torch.uint8, device=dev)
    d0 = dict(d, seam_w=0, conv_k=0)
    reps = max(3, min(args.steps, 10))

    def timed(fn):
        for _ in range(2):
            fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    build_ms = timed(lambda: hypic.segment_build(d, wl.tok, wl.seg_off, T, S, wsp, stream=stream))
    comp_ms = timed(lambda: hypic.compose(d, wl.tok, wl.seg_off, wl.order, T, S, Sf, o_out=o, stream=stream))
    scan_ms = timed(lambda: hypic.compose(d0, wl.tok, wl.seg_off, wl.order, T, S, Sf, stream=stream))
    hypic.workspace_status(wsp, stream)
    hypic.async_status(stream)
    body_tokens = int(sum(max(0, int(x) - min(w, int(x))) for x in wl.lengths))
    flops = body_tokens * L * H * 4.0 * D * (2 * D)
    tf32_peak = peaks["bf16_sustained"] * 1.1 / 2.25
    pair_bytes, comp_bytes = _compose_bytes(wl)
    out = {
        "workload": "%s: %d layer(s) x %d heads, d=%d, %d segments (%d tokens), seam w=%d, order %s"
                    % (name, L, H, D, wl.n_seg, wl.n_tokens, w,
                       "random" if name == "warm_30l" else "in sequence"),
        "build": {"ms": build_ms, "mtok_s_per_layer": body_tokens * L / (build_ms * 1e-3) / 1e6,
                  "tflops": flops / (build_ms * 1e-3) / 1e12,
                  "frac_tf32": flops / (build_ms * 1e-3) / 1e12 / tf32_peak},
        "compose_with_seams": {"ms": comp_ms, "segs_s_per_layer": n_ord * L / (comp_ms * 1e-3),
                               "gbs": comp_bytes / (comp_ms * 1e-3) / 1e9,
                               "hbm_frac": comp_bytes / (comp_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                               "algorithmic_bytes": comp_bytes},
        "compose_alone": {"ms": scan_ms, "gbs": pair_bytes / (scan_ms * 1e-3) / 1e9,
                          "hbm_frac": pair_bytes / (scan_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]},
    }
    del T, S, Sf, o, wsp, wl
    torch.cuda.empty_cache()
    return out


def _small_leg(name, args, dev, stream):
    """Build and compose (with its seams, if the workload has any) on one of
    the small fp32 workloads that run on the exact-fp32 token-serial CUDA-core
    kernels (d < 128 or fp32 inputs), each timed with CUDA events over
    repeated calls.  These calls take microseconds: the times are launch- and
    latency-bound and are reported as such, with no roofline fraction."""
    import torch
    from linear_attn_state_chunked_gb300 import hypic, workloads as W
    wl = W.make(name, device=dev)
    d = wl.desc
    L, H, Dk, Dv, w = d["n_layers"], d["n_heads"], d["d_k"], d["d_v"], d["seam_w"]
    n_ord = len(wl.order)
    tshape, sshape = hypic.pair_shapes(d, wl.n_seg)
    T = torch.empty(tshape, device=dev)
    S = torch.empty(sshape, device=dev)
    Sf = torch.empty((L, H, Dk, Dv), device=dev)
    o = torch.empty((L, n_ord, max(w, 1), H, Dv), device=dev)
    wsp = torch.empty(hypic.workspace_size(d), dtype=torch.uint8, device=dev)
    reps = 50

    def timed(fn):
        for _ in range(3):
            fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    build_ms = timed(lambda: hypic.segment_build(d, wl.tok, wl.seg_off, T, S, wsp, stream=stream))
    comp_ms = timed(lambda: hypic.compose(d, wl.tok, wl.seg_off, wl.order, T, S, Sf,
                                          o_out=o if w > 0 else None, stream=stream))
    hypic.workspace_status(wsp, stream)
    hypic.async_status(stream)
    body_tokens = int(sum(max(0, int(x) - min(w, int(x))) for x in wl.lengths))
    mode = {hypic.GATED_DELTA: "gated delta", hypic.SCALAR_DECAY: "scalar decay (RetNet)",
            hypic.DIAG_GATE: "diagonal gate (Mamba2 / GLA)"}.get(d["mode"], str(d["mode"]))
    out = {
        "workload": "%s: %s, %d layer(s) x %d heads, d_k=d_v=%d, %d segments (%d tokens), fp32 inputs, seam w=%d"
                    % (name, mode, L, H, Dk, wl.n_seg, wl.n_tokens, w),
        "path": "exact-fp32 token-serial CUDA-core kernels",
        "build": {"ms": build_ms, "mtok_s_per_layer": body_tokens * L / (build_ms * 1e-3) / 1e6},
        "compose": {"ms": comp_ms, "segs_s_per_layer": n_ord * L / (comp_ms * 1e-3)},
        "note": "microsecond calls: launch- and latency-bound, no roofline fraction claimed",
    }
    del T, S, Sf, o, wsp, wl
    return out


def _q_rows_read(wl):
    """Token rows of q that the calls read: each request entry's seam tokens
    and the conv history before them (the previous entries' last conv_k - 1
    tokens in request order), merged into sorted ranges [r0, r1)."""
    d = wl.desc
    w, hist = d["seam_w"], max(0, d.get("conv_k", 0) - 1)
    off, order = wl.seg_off, [int(x) for x in wl.order]
    stream = np.concatenate([np.arange(off[s], off[s + 1]) for s in order]) if order else np.zeros(0, np.int64)
    starts = np.cumsum([0] + [int(off[s + 1] - off[s]) for s in order])
    rows = set()
    for e, s in enumerate(order):
        sw = min(w, int(off[s + 1] - off[s]))
        lo = max(0, int(starts[e]) - hist)
        rows.update(int(x) for x in stream[lo:int(starts[e]) + sw])
    ranges = []
    for r in sorted(rows):
        if ranges and ranges[-1][1] == r:
            ranges[-1][1] = r + 1
        else:
            ranges.append([r, r + 1])
    return [tuple(x) for x in ranges]


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args):
    ws, rank, local = _dist()
    if rank != 0:
        return 0
    import torch
    from linear_attn_state_chunked_gb300 import workloads as W
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    wl = W.make(WORKLOAD, device=dev, layers=1)
    heads, segs = ORACLE_HEADS, ORACLE_SEGS
    for _ in range(args.warmup):
        oracle_sample(wl, heads, segs)
    tot_t, tot_tok = 0.0, 0.0
    for _ in range(args.steps):
        dt, lt = oracle_sample(wl, heads, segs)
        tot_t += dt
        tot_tok += lt
    value = tot_tok / tot_t / 1e6
    sample = ("fp64 oracle, layer 0, heads 0-%d, first %d segments of the request (%d tokens): "
              "conv, every body pair, compose, seams" % (heads - 1, segs, int(tot_tok / args.steps * W.describe(WORKLOAD)["n_heads"] / heads)))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": _cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------------
# GPU arm

def run_gpu(args):
    import torch
    from linear_attn_state_chunked_gb300 import hypic, workloads as W

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = _peaks()

    wl = W.make(WORKLOAD, device=dev, layers=args.layers)
    d = wl.desc
    L, H, D, w = d["n_layers"], d["n_heads"], d["d_k"], d["seam_w"]
    n_seg, n_ord = wl.n_seg, len(wl.order)
    tshape, sshape = hypic.pair_shapes(d, n_seg)
    T = torch.empty(tshape, device=dev)
    S = torch.empty(sshape, device=dev)
    Sf = torch.empty((L, H, D, D), device=dev)
    o = torch.empty((L, n_ord, w, H, D), device=dev)
    wsp = torch.empty(hypic.workspace_size(d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        hypic.segment_build(d, wl.tok, wl.seg_off, T, S, wsp, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        hypic.compose(d, wl.tok, wl.seg_off, wl.order, T, S, Sf, o_out=o, stream=stream)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    _barrier(ws)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.4)  # let the sampler emit its first line
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    _barrier(ws)
    ms_total = _reduce_max(start.elapsed_time(end), ws)
    build_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    comp_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)

    # compose alone (the scan over the pairs without seams), same pairs
    d0 = dict(d, seam_w=0, conv_k=0)  # no seams: the conv warm-up has nothing to do
    for _ in range(2):
        hypic.compose(d0, wl.tok, wl.seg_off, wl.order, T, S, Sf, stream=stream)
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for _ in range(args.steps):
        hypic.compose(d0, wl.tok, wl.seg_off, wl.order, T, S, Sf, stream=stream)
    c1.record(stream)
    torch.cuda.synchronize()
    scan_ms = c0.elapsed_time(c1) / args.steps

    # seam advance alone (all seams of the request in parallel from given
    # prefix states): prefix states from one compose, then timed
    Sp = torch.empty((L, n_ord, H, D, D), device=dev)
    hypic.compose(d, wl.tok, wl.seg_off, wl.order, T, S, Sf, o_out=o, S_prefix_out=Sp, stream=stream)
    for _ in range(2):
        hypic.seam_advance(d, wl.tok, wl.seg_off, wl.order, Sp, o, stream=stream)
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(args.steps):
        hypic.seam_advance(d, wl.tok, wl.seg_off, wl.order, Sp, o, stream=stream)
    a1.record(stream)
    torch.cuda.synchronize()
    seam_ms = a0.elapsed_time(a1) / args.steps
    del Sp

    # segment forward (per-token body outputs from a zero state: the segment's
    # first prefill) on the first layer, with and without the pair -- the
    # pair's cost next to the linear layer's own prefill, on the exact-fp32
    # token-serial CUDA-core build that serves the forward
    d1 = dict(d, n_layers=1)
    tok1 = {k: (None if v is None else v[:1]) for k, v in wl.tok.items()}
    o1 = torch.empty((1, wl.n_tokens, H, D), device=dev)
    T1 = torch.empty((1,) + tuple(tshape[1:]), device=dev)
    S1 = torch.empty((1,) + tuple(sshape[1:]), device=dev)
    fwd = {}
    for key, kw in (("outputs_only", {}), ("with_pair", dict(T_out=T1, S_out=S1))):
        hypic.segment_forward(d1, tok1, wl.seg_off, o1, stream=stream, **kw)
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(2):
            hypic.segment_forward(d1, tok1, wl.seg_off, o1, stream=stream, **kw)
        f1.record(stream)
        torch.cuda.synchronize()
        fwd[key] = f0.elapsed_time(f1) / 2
    del o1, T1, S1

    tokens = wl.n_tokens
    body_tokens = int(sum(max(0, int(x) - min(w, int(x))) for x in wl.lengths))
    ms_step = ms_total / args.steps
    value = tokens * L * ws / (ms_step * 1e-3) / 1e6
    build_mtok = body_tokens * L / (build_ms * 1e-3) / 1e6
    comp_segs = n_ord * L / (comp_ms * 1e-3)

    # roofline of the dominant kernel (the build, a tf32 tensor-core
    # contraction): algorithmic flops of the recurrence, 4 d_k (d_k + d_v) =
    # 131,072 per body token and head, against the dense tf32 peak taken as
    # the measured sustained bf16 peak x the nominal tf32/bf16 ratio 1.1/2.25
    # (the build runs ~70 ms inside a longer step).  DRAM traffic per launch:
    # from the ncu capture of the 1-layer case scaled by the layer count
    # (traffic grows in proportion), or null if not supplied.
    flops = body_tokens * L * H * 4.0 * D * (2 * D)
    achieved = flops / (build_ms * 1e-3) / 1e12
    tf32_peak = peaks["bf16_sustained"] * 1.1 / 2.25
    traffic = _build_traffic(L)
    # full roofline time of the build: the recurrence's flops at tf32, the
    # chunk overhead C (2 d_k + d_v) + C^2 / 3 per token-head at bf16, or the
    # algorithmic bytes at HBM speed, whichever is longer
    C = 64
    f_bf16 = body_tokens * L * H * (C * (2.0 * D + D) + C * C / 3.0)
    b_build = (body_tokens * L * H * (2 * D * 2 * (C + 3) / C + 4) + L * n_seg * H * 2 * D * D * 4)
    t_roof = max(flops / (tf32_peak * 1e12) + f_bf16 / (peaks["bf16_sustained"] * 1e12),
                 b_build / (peaks["hbm_gbs"] * 1e9))
    roof = {"kernel": "build_tc_kernel", "bound": "tensor", "achieved": achieved,
            "peak": tf32_peak, "unit": "TFLOP/s", "frac": achieved / tf32_peak, "traffic": traffic,
            "peak_source": "%s sustained bf16 %.1f TFLOP/s x 1.1/2.25 (tf32)"
                           % (peaks["source"], peaks["bf16_sustained"]),
            "algorithmic": "131072 flop per body token-head x %d token-heads" % (body_tokens * L * H),
            "t_roof_ms": t_roof * 1e3, "frac_of_t_roof": t_roof * 1e3 / build_ms,
            "frac_vs_bf16_peak": achieved / peaks["bf16_sustained"],
            "t_roof_note": "max(tf32 flops / tf32 peak + chunk-overhead flops (26k per token-head) / bf16 "
                           "peak, algorithmic bytes / HBM)"}
    # compose + seams: HBM-bound; algorithmic bytes = pairs read + seam inputs + outputs
    pair_bytes = L * n_ord * H * (2 * D * D) * 4
    seam_tok = int(sum(min(w, int(wl.lengths[s])) for s in wl.order))
    # seam tokens: raw q, k, v (bf16) and alpha, beta in; fp32 outputs out
    seam_bytes = L * seam_tok * H * (3 * D * 2 + 2 * 2 + D * 4)
    comp_bytes = pair_bytes + seam_bytes + L * H * D * D * 4
    comp_gbs = comp_bytes / (comp_ms * 1e-3) / 1e9

    # end to end through the C ABI from pinned host buffers (h2d inputs,
    # d2h final state and seam outputs inside the timed region).  The layers
    # are independent, so the step streams them in groups: the inputs of
    # group g + 1 cross the host link while group g is built and composed
    # (token tensors are layer-major, so a group is one contiguous slab).
    e2e = None
    if not args.no_e2e:
        host = {}
        for key, v in wl.tok.items():
            if v is not None:
                host[key] = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                host[key].copy_(v)
        h_Sf = torch.empty(Sf.shape, dtype=Sf.dtype, pin_memory=True)
        h_o = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        # q is read only for the seam tokens and their conv history: those rows
        # alone cross the link (one contiguous copy per layer and range); the
        # other q rows on the device are poisoned with NaN first, so a kernel
        # that read them would show in the outputs checked below
        q_ranges = _q_rows_read(wl)
        q_rows = sum(r1 - r0 for r0, r1 in q_ranges)
        wl.tok["q"].fill_(float("nan"))
        row_bytes = H * D * wl.tok["q"].element_size()
        h2d = sum(v.numel() * v.element_size() for k_, v in host.items() if k_ != "q") + L * q_rows * row_bytes
        d2h = Sf.numel() * 4 + o.numel() * 4
        n_e2e = max(1, min(args.steps, 3))
        n_groups = min(L, args.e2e_groups)
        bounds = [round(g * L / n_groups) for g in range(n_groups + 1)]
        groups = [(bounds[g], bounds[g + 1]) for g in range(n_groups) if bounds[g + 1] > bounds[g]]
        cs_in = torch.cuda.Stream(dev)
        cs_out = torch.cuda.Stream(dev)

        def e2e_step():
            start_ev = torch.cuda.Event()
            start_ev.record(stream)
            cs_in.wait_event(start_ev)
            ev_in = []
            for (l0, l1) in groups:
                with torch.cuda.stream(cs_in):
                    for key, hv in host.items():
                        if key == "q":
                            for l in range(l0, l1):
                                for r0, r1 in q_ranges:
                                    wl.tok["q"][l, r0:r1].copy_(hv[l, r0:r1], non_blocking=True)
                        else:
                            wl.tok[key][l0:l1].copy_(hv[l0:l1], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cs_in)
                ev_in.append(ev)
            for (l0, l1), ev in zip(groups, ev_in):
                stream.wait_event(ev)
                dg = dict(d, n_layers=l1 - l0)
                tg = {k: (None if v is None else v[l0:l1]) for k, v in wl.tok.items()}
                hypic.segment_build(dg, tg, wl.seg_off, T[l0:l1], S[l0:l1], wsp, stream=stream)
                hypic.compose(dg, tg, wl.seg_off, wl.order, T[l0:l1], S[l0:l1], Sf[l0:l1],
                              o_out=o[l0:l1], stream=stream)
                done = torch.cuda.Event()
                done.record(stream)
                cs_out.wait_event(done)
                with torch.cuda.stream(cs_out):
                    h_Sf[l0:l1].copy_(Sf[l0:l1], non_blocking=True)
                    h_o[l0:l1].copy_(o[l0:l1], non_blocking=True)
            end_ev = torch.cuda.Event()
            end_ev.record(cs_out)
            stream.wait_event(end_ev)

        e2e_step()
        torch.cuda.synchronize()
        _barrier(ws)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms_e2e = _reduce_max(e0.elapsed_time(e1), ws) / n_e2e
        # the end-to-end outputs are those of the device-resident step
        o_dev, Sf_dev = o.clone(), Sf.clone()
        hypic.segment_build(d, wl.tok, wl.seg_off, T, S, wsp, stream=stream)
        hypic.compose(d, wl.tok, wl.seg_off, wl.order, T, S, Sf, o_out=o, stream=stream)
        torch.cuda.synchronize()
        same = bool(torch.equal(h_o, o.cpu()) and torch.equal(h_Sf, Sf.cpu()) and torch.isfinite(h_o).all()
                    and torch.isfinite(h_Sf).all())
        del o_dev, Sf_dev
        wl.tok["q"].copy_(host["q"])  # the whole q again, for the legs below
        e2e = {"value": tokens * L * ws / (ms_e2e * 1e-3) / 1e6, "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": n_e2e, "ms_per_step": ms_e2e,
               "h2d_gbs": h2d / (ms_e2e * 1e-3) / 1e9,
               "outputs_match_device_step": same,
               "schedule": "%d layer groups; group g+1's inputs copy while group g computes; k, v, alpha, "
                           "beta, conv weights whole, q only for the %d rows the seams read (seam tokens and "
                           "conv history)" % (len(groups), q_rows)}
        del host

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        heads, segs = ORACLE_HEADS, ORACLE_SEGS
        dt, lt = oracle_sample(wl, heads, segs)
        cpu = {"value": lt / dt / 1e6, "unit": UNIT, "cores": _cores(), "kind": "oracle",
               "sample": "fp64 oracle on layer 0, all %d heads, first %d segments of the request "
                         "(%d tokens): conv, body pairs, compose, seams; %.1f s"
                         % (heads, segs, int(lt * d["n_heads"] / heads), dt)}

    # the other configurations of the workload set, each on its own after the
    # cold prompt's tensors are released: the single-layer gated-delta request
    # (build, compose with seams, compose alone), the warm-cache 30-layer
    # request (its pairs built once, then the compose with seams it is about)
    # and the small fp32 workloads of the CUDA-core paths (tiny gated delta,
    # RetNet decay, diagonal gate)
    configs = None
    if rank == 0 and not args.layers and not args.no_configs:
        del T, S, Sf, o, wsp, wl
        torch.cuda.empty_cache()
        configs = {name: _config_leg(name, args, peaks, dev, stream)
                   for name in ("gdn_bf16", "warm_30l")}
        configs.update({name: _small_leg(name, args, dev, stream)
                        for name in ("tiny_gdn", "decay_retnet", "decay_diag")})

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "tf32", "data": "synthetic",
            "config": dict(_config(), **({"layers": L, "subset": "first %d layers only" % L}
                                         if args.layers else {})),
            "components": {
                "build": {"mtok_s_per_layer": build_mtok, "ms": build_ms, "launches_per_step": 1},
                "compose_alone": {"segs_s_per_layer": n_ord * L / (scan_ms * 1e-3), "ms": scan_ms,
                                  "gbs": pair_bytes / (scan_ms * 1e-3) / 1e9,
                                  "hbm_frac": pair_bytes / (scan_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                  "launches_per_step": 1},
                "seam_advance": {"seams_s_per_layer": n_ord * L / (seam_ms * 1e-3), "ms": seam_ms,
                                 "gbs": (L * n_ord * H * D * D * 4 + seam_bytes) / (seam_ms * 1e-3) / 1e9,
                                 "hbm_frac": (L * n_ord * H * D * D * 4 + seam_bytes) / (seam_ms * 1e-3) / 1e9
                                             / peaks["hbm_gbs"],
                                 "launches_per_step": 1,
                                 "note": "prefix states in, seam outputs out; state not written back"},
                "segment_forward_layer0": {"ms_outputs_only": fwd["outputs_only"],
                                           "ms_with_pair": fwd["with_pair"],
                                           "pair_overhead": fwd["with_pair"] / fwd["outputs_only"] - 1.0,
                                           "note": "per-token body outputs of layer 0 from a zero state on the "
                                                   "exact-fp32 token-serial CUDA-core build, alone and with "
                                                   "(T_C, S(C|0)); the linear layer only, not a whole model"},
                "compose_with_seams": {"segs_s_per_layer": comp_segs, "ms": comp_ms,
                                       "gbs": comp_gbs, "hbm_frac": comp_gbs / peaks["hbm_gbs"],
                                       "launches_per_step": 1}},
            "configs": configs,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "clocks": clk,
            "gpu_launches": 2 * args.steps,
            "peaks": peaks,
        }
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the single-layer gated-delta and warm-cache 30-layer legs")
    ap.add_argument("--e2e-groups", type=int, default=6,
                    help="layer groups of the end-to-end step (copies overlap compute)")
    ap.add_argument("--layers", type=int, default=None,
                    help="first N layers of the workload only (small cases for profiling; "
                         "not a bench line)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
