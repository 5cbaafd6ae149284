#!/usr/bin/env python
"""Benchmark of the hybrid W4A16 MoE layer on GB300.

Headline workload: decode on the 256-expert hybrid layer. H=6144, I=2048,
E=256, top-8 softmax routing. The 64 experts with the largest weight norm
are NVFP4 and the other 192 are NF3. There are M=8 tokens per batch. A step
is one pass of the hot path over one batch: hmoe_plan_routes (top-k, gates,
permutation, offsets) and then hmoe_forward (both GEMMs, SwiGLU, gate-weighted
sum, bf16 output).

value = HBM GB/s. The bytes are the packed weights and scales of the experts
a batch touches, counted once per expert from the routed ids, divided by the
device time of the step. The same line reports:
- a per-M table (M = 1, 2, 4, 8; us per layer and GB/s);
- the prefill point (M = 4096, skewed routing): tokens/s, TFLOP/s and the
  fraction of the bf16 peak;
- the dominant kernel's roofline;
- the CPU oracle's time on a bounded sample.

L2 hygiene: the packed layer is replicated 4 times (4 x 4.30 GB). Step i uses
replica i % 4 and batch i % 4, so no step finds its weights in the 129 MB L2.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
N > 1 runs one independent replica per GPU (the layer does not shard:
replicas only). It is launched through torch.distributed.run.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "hybrid MoE layer µs & HBM GB/s at M≤8; tokens/s & % bf16 peak at M=4096"
SHAPE = synth.HYBRID_256
KEPT = 64
REPLICAS = 4
FMT_NF3, FMT_NVFP4 = 3, 4
BYTES_PER_EXPERT = {4: 21_233_664, 5: 20_054_016, 3: 15_335_424}
W13_BYTES = {4: 14_155_776, 5: 13_369_344, 3: 10_223_616}
TIER_NAMES = {0: "one_launch", 1: "kept_first", 2: "nf3_first"}
# The stream kernel's sources: the traffic figure committed under profiles/ is
# used only while these are unchanged since the capture.
STREAM_SOURCES = ("nf3_moe_gb300/csrc/stream.cu", "nf3_moe_gb300/csrc/common.cuh")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks
def nvsmi_gpu_id(device):
    """The nvidia-smi selector of the torch device: its UUID ("GPU-..."). nvidia-smi numbers
    GPUs physically and ignores CUDA_VISIBLE_DEVICES, so a CUDA ordinal could name another
    user's GPU on a shared machine; the UUID cannot."""
    try:
        u = str(torch.cuda.get_device_properties(device).uuid)
    except (AttributeError, RuntimeError):
        return None
    if not u:
        return None
    return u if u.startswith("GPU-") else "GPU-" + u


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples of one GPU (selected by UUID) while it is under load."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.gpu = nvsmi_gpu_id(device)
        self.proc = None
        self.lines = []

    def start(self):
        try:
            if self.gpu is None:
                return
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", self.gpu], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0,
                    "gpu": self.gpu}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "gpu": self.gpu}


# ------------------------------------------------------------------ helpers
def max_over_ranks(t_ms, world, device):
    """The slowest rank's time, returned on every rank (N > 1 runs one independent
    replica per rank; the whole job takes as long as its slowest replica)."""
    if world <= 1:
        return float(t_ms)
    tt = torch.tensor([float(t_ms)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
    return float(tt.item())


def whole_job_gbs(bytes_per_rank, world, t_ms):
    """GB/s over all ranks: every rank moved bytes_per_rank in the (max-over-ranks) time t_ms."""
    return bytes_per_rank * world / (t_ms * 1e-3) / 1e9


def touched(ids_cpu, fmts):
    es = np.unique(np.asarray(ids_cpu).reshape(-1))
    total = sum(BYTES_PER_EXPERT[fmts[e]] for e in es)
    w13 = sum(W13_BYTES[fmts[e]] for e in es)
    return int(total), int(w13), len(es)


def make_layer(device):
    return synth.make_layer(**SHAPE, kept=KEPT, device=device)


def expert_tuples(L):
    return [(e["w13"][0], e["w13"][1], e["w13"][2], e["w2"][0], e["w2"][1], e["w2"][2]) for e in L.experts]


def oracle_sample(L_host_experts, H, I, x_row, ids_row, gates_row):
    """The oracle on one token. Returns seconds and bytes of its experts."""
    from oracle import layer as olayer
    fmts = {e: L_host_experts[e]["fmt"] for e in L_host_experts}
    t0 = time.perf_counter()
    olayer.moe_forward(x_row[None, :].astype(np.float64), ids_row[None, :], gates_row[None, :].astype(np.float64),
                       lambda e: L_host_experts[e], H, I)
    dt = time.perf_counter() - t0
    return dt, sum(BYTES_PER_EXPERT[fmts[int(e)]] for e in np.unique(ids_row))


def host_experts(L, ids):
    return {int(e): L.expert_numpy(int(e)) for e in np.unique(ids)}


def sources_sha16(paths):
    import hashlib
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def stream_traffic(M):
    """(DRAM bytes per stream-kernel launch, where the figure comes from). The figure is an
    ncu capture committed under profiles/, scaled to this workload; it is used only while
    the kernel's sources are those it was captured on, else (None, reason)."""
    tpath = os.path.join(ROOT, "profiles", "stream_gemm_traffic.json")
    try:
        tj = json.load(open(tpath))
    except (OSError, ValueError):
        return None, "no capture committed"
    if tj.get("M") != M:
        return None, f"capture is for M={tj.get('M')}"
    if tj.get("source_sha16") != sources_sha16(STREAM_SOURCES):
        return None, "stale: the stream kernel changed since the ncu capture"
    return tj.get("dram_bytes_per_launch"), tj.get("how", "ncu capture, scaled")


# ------------------------------------------------------------------ reference arm
def run_reference(args, rank, world):
    if rank != 0:
        return None
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    L = make_layer(dev)
    M = args.m
    x = synth.gen_x(M, SHAPE["H"], seed=1000, device=dev)
    logits = synth.gen_logits(M, SHAPE["E"], seed=1000, device=dev)
    from oracle import route as oroute
    ids, gates, _, _ = oroute.plan(logits.cpu().numpy(), SHAPE["topk"])
    exps = host_experts(L, ids[:1])
    xr = x.float().cpu().numpy()[0]
    del L
    # A step is one routed (token, expert) pair of the batch's first token,
    # cycling over its k experts: about 0.6 s of oracle work, so that
    # --steps K --warmup W ends within a few minutes for the K a bench uses.
    k = SHAPE["topk"]

    def one(i):
        j = i % k
        return oracle_sample(exps, SHAPE["H"], SHAPE["I"], xr, ids[0, j:j + 1], gates[0, j:j + 1])

    for i in range(args.warmup):
        one(i)
    tot_t, tot_b = 0.0, 0
    for i in range(args.steps):
        dt, b = one(i)
        tot_t += dt
        tot_b += b
    value = tot_b / tot_t / 1e9
    cores = len(os.sched_getaffinity(0))
    sample = (f"one routed (token, expert) pair per step, cycling over the {k} experts of the first token of "
              f"an M={M} batch (each dequantised in float64 and multiplied), NumPy on the host")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * tot_t / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"hybrid MoE decode (oracle), H=6144 I=2048 E=256 top-8, 64 NVFP4 + 192 NF3, M={M}",
                   "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world):
    import nf3_moe_gb300 as hm
    from nf3_moe_gb300 import _lib
    if not os.path.exists(_lib.LIB_PATH):
        from nf3_moe_gb300 import build
        build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    H, I, E, k = SHAPE["H"], SHAPE["I"], SHAPE["E"], SHAPE["topk"]
    pk = peaks()

    L = make_layer(dev)
    bit_map = [int(b) for b in L.bit_map]
    experts = expert_tuples(L)
    desc = hm.LayerDesc(H, I, E, k, hm.FMT_NVFP4)
    reps = []
    for _ in range(REPLICAS):
        kb, nb = hm.hmoe_packed_size(desc, bit_map)
        kbuf = torch.empty(kb, dtype=torch.uint8, device=dev)
        nbuf = torch.empty(nb, dtype=torch.uint8, device=dev)
        reps.append(hm.hmoe_pack_weights(desc, bit_map, experts, kbuf, nbuf))
    fmts = [reps[0].expert_info(e)[0] for e in range(E)]
    max_tokens = max(args.m, 8, 0 if args.skip_prefill else args.prefill_m)
    ws = torch.empty(hm.hmoe_workspace_size(desc, max_tokens), dtype=torch.uint8, device=dev)
    hm.hmoe_workspace_init(ws)

    def batches(M, seed0):
        out = []
        for r in range(REPLICAS):
            x = synth.gen_x(M, H, seed=seed0 + r, device=dev)
            lg = synth.gen_logits(M, E, seed=seed0 + r, device=dev)
            bufs = dict(ids=torch.empty((M, k), dtype=torch.int32, device=dev),
                        gates=torch.empty((M, k), dtype=torch.float32, device=dev),
                        perm=torch.empty((M * k,), dtype=torch.int32, device=dev),
                        offsets=torch.empty((E + 1,), dtype=torch.int32, device=dev),
                        out=torch.empty((M, H), dtype=torch.bfloat16, device=dev))
            out.append((x, lg, bufs))
        return out

    def step(i, bl, evs=None, tier_order=hm.TIERS_ONE_LAUNCH):
        r = i % REPLICAS
        x, lg, b = bl[r]
        hm.hmoe_plan_routes(reps[r], lg, b["ids"], b["gates"], b["perm"], b["offsets"], ws)
        hm.hmoe_forward(reps[r], x, b["ids"], b["gates"], b["perm"], b["offsets"], b["out"], ws,
                        stage_events=evs, tier_order=tier_order)

    def batch_bytes(bl):
        res = []
        for r in range(REPLICAS):
            step(r, bl)
        torch.cuda.synchronize()
        for r in range(REPLICAS):
            res.append(touched(bl[r][2]["ids"].cpu().numpy(), fmts))
        return res

    M = args.m
    bl = batches(M, 1000)
    tb = batch_bytes(bl)
    hm.hmoe_check_device_status(ws)

    # Each replica's step (plan + forward) is captured once into a CUDA graph,
    # as a serving engine replays a decode step; the graph holds exactly the
    # library's kernels. A second graph per replica adds two stage events
    # around the GEMM launch (W13 and W2 fused into one stream-kernel launch
    # at M <= 8). Event nodes split a graph and cost about 11 us per replay
    # at M=8 (they also stop the launch from overlapping the routing kernel
    # through programmatic dependent launch), so only the last replay of each
    # replica inside the timed region uses the event graph.
    def capture(bl_, tier_order=hm.TIERS_ONE_LAUNCH, events=False):
        graphs, per_step = [], 0
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for r in range(REPLICAS):
                step(r, bl_, tier_order=tier_order)     # warm the launch path outside capture
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        for r in range(REPLICAS):
            evs = None
            if events:
                evs = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
                for e in evs:
                    e.record()
                torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            n0 = hm.hmoe_launch_count()
            with torch.cuda.graph(g):
                step(r, bl_, evs=evs, tier_order=tier_order)
            per_step = hm.hmoe_launch_count() - n0
            graphs.append((g, evs))
        return graphs, per_step

    graphs, launches_per_step = capture(bl)
    graphs_ev, launches_per_step_ev = capture(bl, events=True)
    assert launches_per_step_ev == launches_per_step

    # warm-up (untimed) and clock soak
    clock = ClockSampler(dev)
    for i in range(args.warmup):
        graphs[i % REPLICAS][0].replay()
    for r in range(REPLICAS):
        graphs_ev[r][0].replay()
    clock.start()
    t_soak = time.perf_counter()
    i = 0
    while time.perf_counter() - t_soak < args.soak_s:
        graphs[i % REPLICAS][0].replay()
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()

    # timed region: exactly K steps, barrier + synchronize on both sides; the
    # last min(K, REPLICAS) steps replay the event graphs
    K = args.steps
    nlast = min(K, REPLICAS)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for i in range(K):
        (graphs_ev if i >= K - nlast else graphs)[i % REPLICAS][0].replay()
    ev1.record()
    torch.cuda.synchronize()
    launches = launches_per_step * K
    if world > 1:
        torch.distributed.barrier()
    clocks = clock.stop()
    t_ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    hm.hmoe_check_device_status(ws)
    bytes_steps = sum(tb[i % REPLICAS][0] for i in range(K))
    value = whole_job_gbs(bytes_steps, world, t_ms)
    # GEMM launch time (W13 + W2, one fused stream-kernel launch) of the
    # event-graph replays at the end of the timed region.
    ev_reps = [i % REPLICAS for i in range(K - nlast, K)]
    gemm_ms = [graphs_ev[r][1][0].elapsed_time(graphs_ev[r][1][1]) for r in ev_reps]
    gemm_avg = sum(gemm_ms) / nlast
    gemm_bytes = sum(tb[r][0] for r in ev_reps) / nlast
    gemm_gbs = gemm_bytes / (gemm_avg * 1e-3) / 1e9

    # per-M table (extra)
    per_m = {}
    for Mm in (1, 2, 4, 8):
        blm = batches(Mm, 2000 + Mm)
        tbm = batch_bytes(blm)
        gm, _ = capture(blm)
        for j in range(8):
            gm[j % REPLICAS][0].replay()
        n = 64
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for j in range(n):
            gm[j % REPLICAS][0].replay()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / n
        byt = sum(tbm[j % REPLICAS][0] for j in range(n)) / n
        per_m[str(Mm)] = {"us_per_layer": round(ms * 1e3, 2), "hbm_gbs": round(byt / (ms * 1e-3) / 1e9, 1),
                          "frac_hbm": round(byt / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                          "touched_experts": round(sum(tbm[j][2] for j in range(REPLICAS)) / REPLICAS, 1)}
        del gm

    # e2e through the public API with host buffers (pinned), copies inside the timed region
    hx = [bl[r][0].cpu().pin_memory() for r in range(REPLICAS)]
    hl = [bl[r][1].cpu().pin_memory() for r in range(REPLICAS)]
    hout = torch.empty((M, H), dtype=torch.bfloat16).pin_memory()
    dx = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    dl = torch.empty((M, E), dtype=torch.float32, device=dev)

    def e2e_step(i):
        r = i % REPLICAS
        b = bl[r][2]
        dx.copy_(hx[r], non_blocking=True)
        dl.copy_(hl[r], non_blocking=True)
        hm.hmoe_plan_routes(reps[r], dl, b["ids"], b["gates"], b["perm"], b["offsets"], ws)
        hm.hmoe_forward(reps[r], dx, b["ids"], b["gates"], b["perm"], b["offsets"], b["out"], ws)
        hout.copy_(b["out"], non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for i in range(args.warmup):
        e2e_step(i)
    t0 = time.perf_counter()
    for i in range(K):
        e2e_step(i)
    e2e_s = time.perf_counter() - t0
    e2e_eager = bytes_steps / e2e_s / 1e9

    # The same step as a serving loop runs it: the input copies, the two API
    # calls and the output copy captured once per replica in a CUDA graph
    # (both calls are graph-safe), replayed and synchronized every step, so
    # the copies still run every step and the host waits for each result.
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for r in range(REPLICAS):
            e2e_step(r)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    e2e_graphs = []
    for r in range(REPLICAS):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            b = bl[r][2]
            dx.copy_(hx[r], non_blocking=True)
            dl.copy_(hl[r], non_blocking=True)
            hm.hmoe_plan_routes(reps[r], dl, b["ids"], b["gates"], b["perm"], b["offsets"], ws)
            hm.hmoe_forward(reps[r], dx, b["ids"], b["gates"], b["perm"], b["offsets"], b["out"], ws)
            hout.copy_(b["out"], non_blocking=True)
        e2e_graphs.append(g)
    for i in range(args.warmup):
        e2e_graphs[i % REPLICAS].replay()
        torch.cuda.current_stream().synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        e2e_graphs[i % REPLICAS].replay()
        torch.cuda.current_stream().synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_val = bytes_steps / e2e_s / 1e9
    hm.hmoe_check_device_status(ws)
    del e2e_graphs

    # tier strategy at decode M=8: one launch per GEMM with per-expert format
    # dispatch, or one launch per tier (kept first / NF3 first); graph replay
    tiers = {"decode_m8_us": {}, "prefill_m4096_ms": {}}
    if world == 1 and not args.skip_tiers:
        for order in (hm.TIERS_ONE_LAUNCH, hm.TIERS_KEPT_FIRST, hm.TIERS_NF3_FIRST):
            gs = capture(bl, tier_order=order)[0]
            for j in range(8):
                gs[j % REPLICAS][0].replay()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a_.record()
            for j in range(64):
                gs[j % REPLICAS][0].replay()
            b_.record()
            torch.cuda.synchronize()
            tiers["decode_m8_us"][TIER_NAMES[order]] = round(a_.elapsed_time(b_) / 64 * 1e3, 2)
            del gs

    # prefill point: M = 4096 with skewed routing
    prefill = None
    if not args.skip_prefill:
        Mp = args.prefill_m
        beta, ratio = synth.calibrate_zipf_beta(Mp, E, k, device=dev, iters=24)
        xp = synth.gen_x(Mp, H, seed=3000, device=dev)
        lp = synth.gen_logits(Mp, E, device=dev) + synth.zipf_bias(E, beta, device=dev)
        bp = dict(ids=torch.empty((Mp, k), dtype=torch.int32, device=dev),
                  gates=torch.empty((Mp, k), dtype=torch.float32, device=dev),
                  perm=torch.empty((Mp * k,), dtype=torch.int32, device=dev),
                  offsets=torch.empty((E + 1,), dtype=torch.int32, device=dev),
                  out=torch.empty((Mp, H), dtype=torch.bfloat16, device=dev))

        def pstep(r, order=hm.TIERS_ONE_LAUNCH):
            hm.hmoe_plan_routes(reps[r], lp, bp["ids"], bp["gates"], bp["perm"], bp["offsets"], ws)
            hm.hmoe_forward(reps[r], xp, bp["ids"], bp["gates"], bp["perm"], bp["offsets"], bp["out"], ws,
                            path=args.prefill_path, tier_order=order)

        def ptime(n, order=hm.TIERS_ONE_LAUNCH):
            # each forward uses the next weight replica, so no forward finds its weights in L2
            for r in range(2):
                pstep(r, order)
            torch.cuda.synchronize()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record()
            for r in range(n):
                pstep(r % REPLICAS, order)
            b_.record()
            torch.cuda.synchronize()
            return a_.elapsed_time(b_) / n

        pclock = ClockSampler(dev)
        pclock.start()
        ms = ptime(args.prefill_steps)
        pclocks = pclock.stop()
        hm.hmoe_check_device_status(ws)
        if world == 1 and not args.skip_tiers:
            for order in (hm.TIERS_ONE_LAUNCH, hm.TIERS_KEPT_FIRST, hm.TIERS_NF3_FIRST):
                tiers["prefill_m4096_ms"][TIER_NAMES[order]] = round(ptime(3, order), 3)
        flops = 2.0 * k * 3 * H * I * Mp
        tfs = flops / (ms * 1e-3) / 1e12
        cnt = torch.bincount(bp["ids"].reshape(-1).long(), minlength=E).float()
        prefill = {"workload": f"hybrid MoE prefill M={Mp}, Zipf(1.1)-biased router logits "
                               f"(beta={beta:.3f}, hottest expert {float(cnt.max() / cnt.mean()):.1f}x mean)",
                   "ms_per_layer": round(ms, 3), "tokens_per_s": round(Mp / (ms * 1e-3), 1),
                   "tflops": round(tfs, 2), "frac_bf16_peak": round(tfs / pk["bf16_tflops"], 4),
                   "peak_used": "bf16_tflops, burst (" + pk["source"] + "): the layer is timed alone, "
                                f"{args.prefill_steps} forwards",
                   "frac_bf16_sustained_peak": round(tfs / pk["bf16_tflops_sustained"], 4),
                   "timing": "eager plan + forward, CUDA events; each forward on the next of 4 weight replicas",
                   "clocks": pclocks,
                   "path": {0: "auto", 1: "stream", 2: "grouped"}[args.prefill_path]}
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            # The oracle on a bounded sample of the same batch: its first two tokens.
            from oracle import layer as olayer
            nt = 2
            ids_p = bp["ids"][:nt].cpu().numpy()
            g_p = bp["gates"][:nt].cpu().numpy().astype(np.float64)
            x_p = xp[:nt].float().cpu().numpy().astype(np.float64)
            exps_p = host_experts(L, ids_p)
            t0 = time.perf_counter()
            olayer.moe_forward(x_p, ids_p, g_p, lambda e: exps_p[e], H, I)
            dt = time.perf_counter() - t0
            prefill["cpu_baseline"] = {
                "value": round(nt / dt, 4), "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
                "kind": "oracle", "tflops": round(2.0 * k * 3 * H * I * nt / dt / 1e12, 6),
                "sample": f"the first {nt} tokens of the M={Mp} batch ({len(exps_p)} experts), float64 NumPy "
                          f"dequantise-then-matmul, {dt:.1f} s"}

    # CPU oracle on a bounded sample (rank 0, N=1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # The first two tokens of the batch, one oracle call each (about 10 s):
        # each call dequantises its token's experts, so the bytes add up per call.
        nt = 2
        ids0 = bl[0][2]["ids"].cpu().numpy()
        g0 = bl[0][2]["gates"].cpu().numpy()
        exps = host_experts(L, ids0[:nt])
        xs = bl[0][0].float().cpu().numpy()
        dt, byt = 0.0, 0
        for t in range(nt):
            d_, b_ = oracle_sample(exps, H, I, xs[t], ids0[t], g0[t])
            dt += d_
            byt += b_
        cpu = {"value": round(byt / dt / 1e9, 4), "unit": "GB/s", "cores": len(os.sched_getaffinity(0)),
               "kind": "oracle",
               "sample": f"the first {nt} tokens of the M={M} batch, one oracle call each ({len(exps)} distinct "
                         f"experts, {byt / 1e6:.0f} MB packed in all), float64 NumPy dequantise-then-matmul, "
                         f"{dt:.1f} s"}

    traffic, traffic_source = stream_traffic(M)
    sweep = None
    if world == 1 and not args.skip_sweep:
        del graphs, graphs_ev
        torch.cuda.empty_cache()
        sweep = sweep_points(dev, pk, steps=args.sweep_steps, warmup=3)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(t_ms / K, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"hybrid MoE decode, H=6144 I=2048 E=256 top-8, 64 NVFP4 + 192 NF3, M={M}",
                   "us_per_layer": round(t_ms / K * 1e3, 2),
                   "frac_hbm": round(value / world / pk["hbm_gbs"], 4),
                   "bytes_per_step": int(bytes_steps / K),
                   "l2": f"{REPLICAS} rotating weight replicas and batches; each step touches > L2 (129 MB)",
                   "timing": "CUDA-graph replay of plan + forward per step; CUDA events on the replay stream; "
                             "the last replay of each replica carries the stage events of the roofline timing",
                   "parallelism": "replicas only" if world > 1 else "1 GPU",
                   "peaks": pk, "per_m": per_m, "prefill": prefill, "tiers": tiers, "sweep": sweep},
        "clocks": clocks,
        "e2e": {"value": round(e2e_val, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(M * H * 2 + M * E * 4), "d2h_bytes_per_step": int(M * H * 2),
                "timing": "host clock over K steps, each: pinned-host copies of x and the router logits in, "
                          "hmoe_plan_routes + hmoe_forward, the output copied back, all captured once per replica "
                          "in a CUDA graph and replayed, then a stream synchronize",
                "eager_value": round(e2e_eager, 2),
                "eager_timing": "the same step issued eagerly from Python (ctypes calls and torch copies) each step"},
        "gpu_launches": int(launches),
        "roofline": {"kernel": "stream_gemm_kernel (W13 + W2 in one launch: dequant + mma, SwiGLU, slot store)",
                     "bound": "hbm",
                     "achieved": round(gemm_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(gemm_gbs / pk["hbm_gbs"], 4), "traffic": traffic,
                     "traffic_source": traffic_source,
                     "algorithmic_bytes_per_launch": int(gemm_bytes), "avg_launch_us": round(gemm_avg * 1e3, 2),
                     "timing": "stage events around the launch in a second graph per replica, replayed as the last "
                               "step of each replica inside the timed region"},
        "cpu_baseline": cpu,
    }
    return line if rank == 0 else None


def run_profile_case(args):
    """A small, fixed case for ncu captures. It prints nothing timed.

    The layer has the 256-expert shape with fewer experts (--experts;
    H=6144, I=2048, top-8, --kept experts kept NVFP4, a quarter by default).
    It runs --steps forwards at M = --m tokens in tier order --tier-order:
    the stream kernel for M <= 8, the tcgen05 grouped kernel above that.
    """
    import nf3_moe_gb300 as hm
    dev = torch.device("cuda", torch.cuda.current_device())
    E, M = args.experts, args.m
    L = synth.make_layer(SHAPE["H"], SHAPE["I"], E, SHAPE["topk"], kept=args.kept or max(1, E // 4), device=dev)
    moe = hm.HybridMoELayer(L.H, L.I, E, L.topk, [int(b) for b in L.bit_map], expert_tuples(L), max_tokens=M)
    x = synth.gen_x(M, L.H, device=dev)
    lg = synth.gen_logits(M, E, device=dev)
    ids, gates, perm, off = moe.plan(lg)
    out = torch.empty((M, L.H), dtype=torch.bfloat16, device=dev)
    for _ in range(args.steps):
        hm.hmoe_forward(moe.layer, x, ids, gates, perm, off, out, moe.ws, tier_order=args.tier_order)
    torch.cuda.synchronize()
    hm.hmoe_check_device_status(moe.ws)
    fmts = [moe.layer.expert_info(e)[0] for e in range(E)]
    tb, _, ne = touched(ids.cpu().numpy(), fmts)
    print(json.dumps({"profile_case": {"experts": E, "m": M, "steps": args.steps, "tier_order": args.tier_order,
                                       "touched_experts": ne,
                                       "touched_packed_bytes": tb}}))


def sweep_points(dev, pk, steps=10, warmup=3):
    """The other configurations, one point at a time, timed like the headline.

    - the 256-expert shape with the kept tier in MXFP4 (64 MXFP4 + 192 NF3),
      M in {64, 512}, uniform N(0,1) logits;
    - the uniform NVFP4 layer (H=2048, I=768, E=128, top-8, no bit map),
      M in {1, 8, 128, 1024, 8192};
    - the headline 256-expert hybrid layer (64 NVFP4 + 192 NF3) with fp16
      activations, M in {8, 4096};
    - the same layer as W4A4 (activations quantised to NVFP4, static global
      scales 5 / 2688 for x and 24 / 2688 for h), M in {8, 4096}.
    A step is plan + forward on the automatic path, captured once in a CUDA
    graph and replayed. Before every replay a 512 MB buffer is written,
    outside the event bracket, so no step finds its weights in the 129 MB L2.
    Returns one entry per point (median of ``steps`` replays after ``warmup``).
    """
    import nf3_moe_gb300 as hm
    bpw = {FMT_NVFP4: 0.5625, 5: 0.53125, FMT_NF3: 0.40625}
    cases = [
        ("hybrid MXFP4 kept tier, H=6144 I=2048 E=256 top-8, 64 MXFP4 + 192 NF3",
         dict(**SHAPE, kept=KEPT, kept_format=synth.FMT_MXFP4), (64, 512)),
        ("uniform NVFP4, H=2048 I=768 E=128 top-8", dict(**synth.UNIFORM_128, uniform=True),
         (1, 8, 128, 1024, 8192)),
        ("hybrid NVFP4 + NF3 with fp16 activations, H=6144 I=2048 E=256 top-8, 64 NVFP4 + 192 NF3",
         dict(**SHAPE, kept=KEPT, act="f16"), (8, 4096)),
        ("hybrid NVFP4 + NF3, W4A4 (NVFP4 activations), H=6144 I=2048 E=256 top-8, 64 NVFP4 + 192 NF3",
         dict(**SHAPE, kept=KEPT), (8, 4096)),
    ]
    w4a4_globals = (5.0 / (6 * 448), 24.0 / (6 * 448))
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    points = []
    for name, kw, ms in cases:
        L = synth.make_layer(device=dev, **kw)
        bm = None if L.bit_map is None else [int(b) for b in L.bit_map]
        w4a4 = "W4A4" in name
        moe = hm.HybridMoELayer(L.H, L.I, L.E, L.topk, bm, expert_tuples(L), kept_format=L.kept_format,
                                max_tokens=max(ms), act_dtype=hm.ACT_F16 if L.act == "f16" else hm.ACT_BF16,
                                act_globals=w4a4_globals if w4a4 else None)
        fmts = [moe.layer.expert_info(e)[0] for e in range(L.E)]
        per_w = 3 * L.H * L.I
        for M in ms:
            x = synth.gen_x(M, L.H, seed=4000 + M, device=dev, dtype=L.x_dtype)
            lg = synth.gen_logits(M, L.E, seed=4000 + M, device=dev)
            ids = torch.empty((M, L.topk), dtype=torch.int32, device=dev)
            gates = torch.empty((M, L.topk), dtype=torch.float32, device=dev)
            perm = torch.empty((M * L.topk,), dtype=torch.int32, device=dev)
            off = torch.empty((L.E + 1,), dtype=torch.int32, device=dev)
            out = torch.empty((M, L.H), dtype=moe.dtype, device=dev)

            def fwd():
                hm.hmoe_plan_routes(moe.layer, lg, ids, gates, perm, off, moe.ws)
                hm.hmoe_forward(moe.layer, x, ids, gates, perm, off, out, moe.ws)

            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                fwd()
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fwd()
            ts = []
            for i in range(warmup + steps):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                g.replay()
                b.record()
                torch.cuda.synchronize()
                if i >= warmup:
                    ts.append(a.elapsed_time(b))
            hm.hmoe_check_device_status(moe.ws)
            ms_ = statistics.median(ts)
            es = np.unique(ids.cpu().numpy().reshape(-1))
            byt = sum(per_w * bpw[fmts[int(e)]] for e in es)
            tfs = 2.0 * L.topk * per_w * M / (ms_ * 1e-3) / 1e12
            path = "stream" if hm.hmoe_auto_path(moe.desc, M) == hm.PATH_STREAM else "grouped"
            points.append({"workload": f"{name}, M={M}", "path": path, "act": L.act,
                           "act_quant": "nvfp4" if w4a4 else None,
                           "us_per_layer": round(ms_ * 1e3, 2), "touched_experts": int(len(es)),
                           "touched_bytes": int(byt), "hbm_gbs": round(byt / (ms_ * 1e-3) / 1e9, 1),
                           "frac_hbm": round(byt / (ms_ * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                           "tokens_per_s": round(M / (ms_ * 1e-3), 1),
                           "tflops": round(tfs, 2), "frac_bf16_peak": round(tfs / pk["bf16_tflops"], 4)})
            del g
        del moe, L
        torch.cuda.empty_cache()
    del flush
    torch.cuda.empty_cache()
    return points


def run_sweep(args):
    """The sweep of sweep_points() alone, printed as one JSON object."""
    dev = torch.device("cuda", torch.cuda.current_device())
    pk = peaks()
    points = sweep_points(dev, pk, steps=args.steps, warmup=args.warmup)
    print(json.dumps({"sweep": points, "steps": args.steps, "warmup": args.warmup, "peaks": pk,
                      "timing": "CUDA-graph replay of plan + forward, CUDA events, L2 flushed before each "
                                "replay; median"}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--m", type=int, default=8)
    ap.add_argument("--prefill-m", type=int, default=4096)
    ap.add_argument("--prefill-steps", type=int, default=5)
    ap.add_argument("--prefill-path", type=int, default=0)
    ap.add_argument("--skip-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--soak-s", type=float, default=1.0)
    ap.add_argument("--profile", action="store_true", help="run the small fixed case used for ncu captures")
    ap.add_argument("--experts", type=int, default=64, help="experts in the --profile case")
    ap.add_argument("--tier-order", type=int, default=0, choices=(0, 1, 2),
                    help="tier_order of the --profile case's forwards (0 one launch, 1 kept first, 2 NF3 first)")
    ap.add_argument("--kept", type=int, default=0, help="kept experts in the --profile case (0: a quarter)")
    ap.add_argument("--sweep", action="store_true", help="time only the MXFP4-kept and uniform NVFP4 configurations")
    ap.add_argument("--skip-sweep", action="store_true", help="leave the other configurations out of the line")
    ap.add_argument("--sweep-steps", type=int, default=10)
    ap.add_argument("--skip-tiers", action="store_true", help="leave the tier-order timings out of the line")
    args = ap.parse_args()
    if args.profile:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        run_profile_case(args)
        return
    if args.sweep:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        args.warmup = max(args.warmup, 3)
        run_sweep(args)
        return
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    if world > 1:
        if args.impl == "reference":
            if rank != 0:
                return
        else:
            torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    line = run_reference(args, rank, world) if args.impl == "reference" else run_ours(args, rank, world)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl != "reference":
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
