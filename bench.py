"""Benchmark of the Kimi-K3 routed-expert MoE layer forward on GB300.

One step = one kmoe_forward over one batch: routing -> MXFP8 quantisation ->
expert permutation -> FC1 (+SiTU +requant) -> FC2 -> combine, with the layer's
inputs (x, router logits, correction bias) and the 896 experts' MXFP4 weights
resident in HBM.  Headline: tokens/s of the T=8192 prefill-chunk layer
(H=7168, I=3584, E=896, top-16), with TFLOP/s and the T=16 decode layer's
microseconds per layer alongside.  Inputs are synthetic and seeded.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the float64 CPU oracle (a deliberately slow program)
on the host cores, on a bounded token sample per step.
Under torchrun (N > 1) every rank runs its own replica of the layer (the path
does not shard; replicas only) and rank 0 prints one JSON line with the
whole-job throughput (tokens of all ranks / slowest rank's time).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "Kimi-K3 MoE layer tokens/s & TFLOP/s at T=8192; µs/layer at T=16 (1×GB300)"
HEADLINE = "prefill"     # T=8192 layer
DECODE = "decode"        # T=16 layer
BIG_TILE_ROWS_ABOVE = 64  # experts with more rows than this take the 224-row CTA-pair tiles


def kernel_launches(w) -> int:
    """Kernels of this library one forward launches: routing; the permutation
    (rank + scan, or one block when R <= 1024); quantise-scatter; FC1 and FC2
    (each a CTA-pair launch for the big-tile experts, left out when no expert
    can exceed 64 rows (T <= 64), and a small-tile launch); combine."""
    fc = 2 if w.T > BIG_TILE_ROWS_ABOVE else 1
    return 1 + (2 if w.R > 1024 else 1) + 1 + 2 * fc + 1
ROUNDS = 5               # interleaved timing rounds (median reported)
# the five seeded workloads, timed in turn within every round; the small ones
# (inputs that fit in L2) with the L2 flushed before every timed forward
INTERLEAVED = ("prefill", "decode", "skewed", "reduced", "tiny")
FLUSHED = ("reduced", "tiny")


def headline_config(world_size: int) -> dict:
    """The `config` block of the headline line (both arms print the same)."""
    wp = W.WORKLOADS[HEADLINE]
    return {"workload": "Kimi-K3 MoE layer prefill chunk T=8192 H=7168 I=3584 E=896 top-16 (SiTU 4/25)",
            "global_batch": wp.T * world_size, "seq_len": wp.T,
            "parallelism": "replicas" if world_size > 1 else "single-gpu",
            "l2": "inputs larger than L2 (36.7 GB of expert weights streamed every step)"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
        return dist
    return None


def reduce_max(dist, v, device):
    if dist is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def job_throughput(dist, world_size, tokens_per_rank_step, steps, rank_ms, device):
    """Whole-job tokens/s: the tokens of all ranks over the slowest rank's time
    (every rank runs its own replica of the layer; no data-path collective)."""
    slowest_ms = reduce_max(dist, rank_ms, device)
    return world_size * tokens_per_rank_step * steps / (slowest_ms / 1e3), slowest_ms


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (100 ms period), started before the warm-up so that
    it is running when the timed region begins; only samples stamped inside
    the timed region [begin(), end()] are kept (the nearest one if none is)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None
        # raw samples go to a scratch directory (the summary goes into the JSON line)
        d = os.environ.get("KMOE_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(d, f"kmoe_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def begin(self):
        self.t0 = time.time()

    def end(self):
        self.t1 = time.time()

    @staticmethod
    def _stamp(text):
        import datetime
        try:
            return datetime.datetime.strptime(text, "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((self._stamp(parts[0]), float(parts[2]), float(parts[3]),
                             {n for n, v in zip(names, parts[6:10]) if v.lower() == "active"}))
            except ValueError:
                continue
        inside = [r for r in rows if r[0] is not None and self.t0 is not None and self.t1 is not None
                  and self.t0 <= r[0] <= self.t1]
        note = None
        if not inside and rows:
            mid = 0.5 * (self.t0 + self.t1) if self.t0 is not None and self.t1 is not None else None
            dated = [r for r in rows if r[0] is not None]
            if mid is not None and dated:
                inside = [min(dated, key=lambda r: abs(r[0] - mid))]
                note = "no sample inside the timed region; nearest sample"
        sm = [r[1] for r in inside]
        reasons = set().union(*[r[3] for r in inside]) if inside else set()
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(r[2] for r in inside) if inside else None,
               "reasons": sorted(reasons), "samples": len(sm)}
        if note:
            out["note"] = note
        return out


# ----------------------------------------------------------------------------- peaks
L2_BYTES = 129 << 20  # GB300 L2 (MB as nvidia reports it, rounded up)

WORKLOAD_TEXT = {
    "tiny": "Tiny MoE layer T=16 H=128 I=128 E=8 top-2",
    "reduced": "Reduced-expert Kimi-K3 layer T=128 H=7168 I=3584 E=64 top-16",
    "decode": "Kimi-K3 MoE layer decode T=16 H=7168 I=3584 E=896 top-16",
    "prefill": "Kimi-K3 MoE layer prefill chunk T=8192 H=7168 I=3584 E=896 top-16",
    "skewed": "Skewed-routing Kimi-K3 layer T=2048 H=7168 I=3584 E=896 top-16 (Zipf s=1.2 bias, max +3.0)",
}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


FC1_KERNEL_SOURCES = ("gemm_pair.cu", "gemm.cu", "gemm_dev.cuh", "gemm.cuh", "ptx.cuh")


def fc1_kernel_sha256():
    """sha256 over the sources of the prefill FC1 kernel (in a fixed order)."""
    h = hashlib.sha256()
    for f in FC1_KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, "mxfp8_mxfp4_moe_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def fc1_traffic_record():
    """DRAM bytes per FC1 launch from a committed ncu summary, if the kernel
    sources it was taken on are unchanged (else null)."""
    path = os.path.join(ROOT, "profiles", "fc1_dram_traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path))
    if rec.get("fc1_kernel_sha256") != fc1_kernel_sha256():
        return None
    return rec


DECODE_KERNEL_SOURCES = ("gemm.cu", "gemm_dev.cuh", "gemm.cuh", "ptx.cuh")


def decode_kernel_sha256():
    """sha256 over the sources of the small-tile (decode) GEMM kernel."""
    h = hashlib.sha256()
    for f in DECODE_KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, "mxfp8_mxfp4_moe_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def decode_traffic_record():
    """DRAM bytes per touched expert of the decode FC1 launch from a committed
    ncu summary, if the kernel sources are unchanged since (else null)."""
    path = os.path.join(ROOT, "profiles", "decode_fc1_dram_traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path))
    if rec.get("decode_kernel_sha256") != decode_kernel_sha256():
        return None
    return rec


# ----------------------------------------------------------------------------- layer set-up
class Layer:
    def __init__(self, w: W.Workload, device, weights=None):
        import torch
        import mxfp8_mxfp4_moe_gb300 as K
        self.K = K
        self.w = w
        self.device = device
        s = W.gen_small_inputs(w)
        self.host = s
        self.x = torch.from_numpy(s["x"].view(np.int16)).view(torch.bfloat16).to(device)
        self.wg = torch.from_numpy(s["wg"].view(np.int16)).view(torch.bfloat16).to(device)
        self.router = False  # True: route from x and the gate weight (kmoe_forward_router)
        self.logits = torch.from_numpy(s["logits"]).to(device)
        self.bias = torch.from_numpy(s["bias"]).to(device)
        self.p = layer_params(K, w)
        if weights is None:
            wts = W.gen_expert_weights_torch(w, device)
            w13_k, w2_k = K.kmoe_prepare_weights(self.p, wts["w13"], wts["w13_sf"], wts["w2"], wts["w2_sf"])
            del wts
            torch.cuda.empty_cache()
            weights = {"w13_k": w13_k, "w2_k": w2_k}
        self.weights = weights
        self.ws = torch.zeros(K.kmoe_workspace_size(self.p), dtype=torch.uint8, device=device)
        self.out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=device)
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
        for e in self.events:
            e.record()
        torch.cuda.synchronize()

    def forward(self, stage_events=False, x=None, logits=None, bias=None, out=None):
        wt = self.weights
        if self.router:
            self.K.kmoe_forward_router(self.p, self.x if x is None else x, self.wg, self.bias if bias is None else bias,
                                       wt["w13_k"], wt["w2_k"], out=self.out if out is None else out,
                                       workspace=self.ws, stage_events=self.events if stage_events else None)
            return
        self.K.kmoe_forward(self.p, self.x if x is None else x, self.logits if logits is None else logits,
                            self.bias if bias is None else bias, wt["w13_k"], wt["w2_k"],
                            out=self.out if out is None else out, workspace=self.ws,
                            stage_events=self.events if stage_events else None)

    def stage_ms(self):
        ev = self.events
        return [ev[i].elapsed_time(ev[i + 1]) for i in range(6)]

    def touched_experts(self):
        v = self.K.stage_views(self.p, self.ws)
        return int((v["counts"] > 0).sum().item())

    def check(self):
        st, word = self.K.kmoe_device_error(self.ws)
        if st != 0:
            raise RuntimeError(f"device error {word:#x}")


def time_layer(layer, steps, warmup, dist, device, clocks=None):
    import torch
    if clocks:
        clocks.start()  # running well before the timed region begins
    for _ in range(warmup):
        layer.forward()
    torch.cuda.synchronize()
    layer.check()
    stream = torch.cuda.current_stream()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    if clocks:
        clocks.begin()
    start.record(stream)
    for _ in range(steps):
        layer.forward()
    end.record(stream)
    torch.cuda.synchronize()
    if clocks:
        clocks.end()
    clk = clocks.stop() if clocks else None
    barrier(dist)
    total_ms = start.elapsed_time(end)
    return total_ms, clk


def time_block(layer, steps):
    """ms per forward over `steps` back-to-back forwards (CUDA events on the
    launching stream, synchronised on both sides)."""
    import torch
    stream = torch.cuda.current_stream()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(steps):
        layer.forward()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def time_flushed(layer, steps, flush):
    """ms per forward, each forward timed alone right after a write of
    `flush` (a buffer twice the size of L2), so no input starts in L2."""
    import torch
    stream = torch.cuda.current_stream()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    tot = 0.0
    for _ in range(steps):
        flush.zero_()
        a.record(stream)
        layer.forward()
        b.record(stream)
        torch.cuda.synchronize()
        tot += a.elapsed_time(b)
    return tot / steps


def time_interleaved(layers, steps, dist, clocks, flush):
    """ROUNDS rounds; in each, every workload of `layers` is timed in turn
    (INTERLEAVED order): the headline for about steps / ROUNDS back-to-back
    forwards (the rounds time exactly `steps` headline forwards), the others
    for a fixed count.  Returns {name: [ms per forward of each round]} and
    {name: [forwards in each round]}."""
    import torch
    # the headline's `steps` forwards split over the rounds (a round left
    # with none, when steps < ROUNDS, times the other workloads only)
    head = [steps // ROUNDS + (1 if r < steps % ROUNDS else 0) for r in range(ROUNDS)]
    counts = {n: (head if n == HEADLINE else [10 if n in FLUSHED else 20] * ROUNDS) for n in layers}
    out = {n: [] for n in layers}
    barrier(dist)
    torch.cuda.synchronize()
    if clocks:
        clocks.begin()
    for r in range(ROUNDS):
        for n, layer in layers.items():
            c = counts[n][r]
            if c == 0:
                continue
            out[n].append(time_flushed(layer, c, flush) if n in FLUSHED else time_block(layer, c))
    torch.cuda.synchronize()
    if clocks:
        clocks.end()
    barrier(dist)
    return out, counts


def time_graph(layer, steps, blocks=3):
    """The layer's forward captured once into a CUDA graph and replayed
    `steps` times back to back (no host launch work between kernels), after
    ten untimed replays; microseconds per forward, the median of `blocks`
    such runs."""
    import torch
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        layer.forward()  # warm-up on the capture stream
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        layer.forward()
    for _ in range(10):
        g.replay()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    runs = []
    for _ in range(blocks):
        s.record()
        for _ in range(steps):
            g.replay()
        e.record()
        torch.cuda.synchronize()
        runs.append(1000.0 * s.elapsed_time(e) / steps)
    return float(np.median(runs))


def time_stages(layer, steps):
    """Per-stage durations from the stage events, averaged over `steps` forwards."""
    import torch
    acc = np.zeros(6)
    for _ in range(steps):
        layer.forward(stage_events=True)
        torch.cuda.synchronize()
        acc += np.array(layer.stage_ms())
    return (acc / steps).tolist()


def mma_peak(device, N=224, iters=500000):
    """Measured tensor-pipe roof of the GEMMs' instruction (kmoe_mma_peak_run):
    block-scaled E2M1 x E4M3 MMAs on resident operands, one CTA per SM."""
    import torch
    import mxfp8_mxfp4_moe_gb300 as K
    ws = torch.zeros(256, dtype=torch.uint8, device=device)
    K.kmoe_mma_peak_run(1000, N, ws)
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record()
    flops = K.kmoe_mma_peak_run(iters, N, ws)
    e.record()
    torch.cuda.synchronize()
    st, word = K.kmoe_device_error(ws)
    if st != 0:
        raise RuntimeError(f"peak kernel device error {word:#x}")
    ms = s.elapsed_time(e)
    return {"tflops": flops / (ms / 1e3) / 1e12, "N": N, "duration_ms": ms,
            "what": "tcgen05.mma kind::mxf8f6f4 block-scaled E2M1 x E4M3, M=128, operands resident in smem, "
                    "one CTA per SM"}


def time_router(w, device, iters=20):
    """The fused router (kmoe_router) alone on workload w, with the L2 flushed
    (a 256 MB write) before every timed launch; beside it, for context, the
    routing kernel alone on the same logits (kmoe_route) and a cuBLAS bf16
    GEMM of the same shape (torch.matmul, bf16 output)."""
    import torch
    import mxfp8_mxfp4_moe_gb300 as K
    s = W.gen_small_inputs(w)
    x = torch.from_numpy(s["x"].view(np.int16)).view(torch.bfloat16).to(device)
    wg = torch.from_numpy(s["wg"].view(np.int16)).view(torch.bfloat16).to(device)
    bias = torch.from_numpy(s["bias"]).to(device)
    logits = torch.empty((w.T, w.E), dtype=torch.float32, device=device)
    ids = torch.empty((w.T, w.k), dtype=torch.int32, device=device)
    wts = torch.empty((w.T, w.k), dtype=torch.float32, device=device)
    ws = torch.zeros(K.kmoe_router_workspace_size(w.T, w.H, w.E), dtype=torch.uint8, device=device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def timed(fn):
        for _ in range(3):
            fn()
        tot = 0.0
        for _ in range(iters):
            flush.zero_()
            ev[0].record()
            fn()
            ev[1].record()
            torch.cuda.synchronize()
            tot += ev[0].elapsed_time(ev[1])
        return tot / iters

    t_router = timed(lambda: K.kmoe_router(x, wg, bias, w.k, logits, ids, wts, ws))
    st, word = K.kmoe_device_error(ws)
    if st != 0:
        raise RuntimeError(f"router device error {word:#x}")
    t_route = timed(lambda: K.kmoe_route(logits, bias, w.k, ids, wts))
    t_cublas = timed(lambda: torch.matmul(x, wg.t()))
    flops = 2.0 * w.T * w.H * w.E
    nbytes = 2.0 * w.T * w.H + 2.0 * w.E * w.H + 4.0 * w.T * w.E + 8.0 * w.T * w.k + 4.0 * w.E
    return {"router_ms": t_router, "route_kernel_only_ms": t_route, "cublas_bf16_gemm_ms": t_cublas,
            "gemm_tflops": flops / (t_router / 1e3) / 1e12, "algorithmic_GBs": nbytes / (t_router / 1e3) / 1e9,
            "flop": flops, "algorithmic_bytes": nbytes}


def e2e_time(layer, steps, warmup):
    """Same metric through the C ABI with host buffers: every step copies its
    x, logits and bias from pinned host memory to the device, runs the
    forward, and reads its output back to pinned host memory, all inside the
    timed region.  Two buffer sets and three streams (copy-in, compute,
    copy-out) let the copies of neighbouring steps overlap a step's compute,
    as a serving loop would; events order every buffer reuse."""
    import torch
    hx = layer.x.cpu().pin_memory()
    hl = layer.logits.cpu().pin_memory()
    hb = layer.bias.cpu().pin_memory()
    hout = [torch.empty(layer.out.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dx = [torch.empty_like(layer.x) for _ in range(2)]
    dl = [torch.empty_like(layer.logits) for _ in range(2)]
    db = [torch.empty_like(layer.bias) for _ in range(2)]
    dout = [torch.empty_like(layer.out) for _ in range(2)]
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for e in comp_done + out_done:
        e.record(torch.cuda.current_stream())
    torch.cuda.synchronize()

    def step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(comp_done[b])          # step i-2 finished reading dx[b]...
            dx[b].copy_(hx, non_blocking=True)
            dl[b].copy_(hl, non_blocking=True)
            db[b].copy_(hb, non_blocking=True)
            in_done[b].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(in_done[b])
            s_comp.wait_event(out_done[b])         # ...and its output was read back
            layer.forward(x=dx[b], logits=dl[b], bias=db[b], out=dout[b])
            comp_done[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            hout[b].copy_(dout[b], non_blocking=True)
            out_done[b].record(s_out)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for i in range(steps):
        step(warmup + i)
    end.record(s_out)  # after the last step's read-back
    torch.cuda.synchronize()
    h2d = hx.numel() * 2 + hl.numel() * 4 + hb.numel() * 4
    d2h = hout[0].numel() * 2
    return start.elapsed_time(end), h2d, d2h


# ----------------------------------------------------------------------------- CPU oracle
def oracle_inputs(w: W.Workload):
    from oracle import moe as O
    s = W.gen_small_inputs(w)
    ids, wts, _ = O.route(s["logits"], s["bias"], w.k)
    return s, ids, wts


def oracle_slot_sample(w: W.Workload, budget_s: float, seed: int, pre):
    """Time the float64 oracle (as it stands) on (token, expert slot) pairs
    of the workload, drawn at random, until `budget_s` of oracle time has
    passed (at least one pair): each pair is the oracle's forward of one
    token with its other slots masked, i.e. 1/k of that token's expert work.
    Returns (tokens/s, token equivalents, seconds, threads)."""
    from oracle import moe as O
    s, ids, wts = pre
    rng = np.random.default_rng(1000 + seed)
    pairs, done_s = 0, 0.0
    while pairs == 0 or done_s < budget_s:
        t = int(rng.integers(w.T))
        j = int(rng.integers(w.k))
        masked = np.full_like(ids, -1)
        masked[t, j] = ids[t, j]
        e = int(ids[t, j])
        weights = W.gen_expert_weights_np(w, [e])       # data generation: outside the timed region
        t0 = time.perf_counter()
        O.forward(w, s["x"], None, None, weights, experts_host=[e], tokens=np.array([t]), ids=masked, topk_w=wts)
        done_s += time.perf_counter() - t0
        pairs += 1
    return (pairs / w.k) / done_s, pairs / w.k, done_s, os.cpu_count()


# ----------------------------------------------------------------------------- main
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = W.WORKLOADS[HEADLINE]
    pre = oracle_inputs(w)
    per_step = []
    for i in range(args.warmup + args.steps):
        tps, ntok, secs, cores = oracle_slot_sample(w, budget_s=args.ref_step_s, seed=i, pre=pre)
        if i >= args.warmup:
            per_step.append((tps, ntok, secs))
    tps = sum(x[1] for x in per_step) / sum(x[2] for x in per_step)
    step_ms = 1000.0 * sum(x[2] for x in per_step) / len(per_step)
    line = {
        "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; random MXFP4 weights of the Kimi-K3 expert shapes)",
        "impl": "reference",
        "config": headline_config(args.gpus),
        "step": "a bounded sample of the layer per step: random (token, expert slot) pairs until "
                f"{args.ref_step_s:g} s of oracle time; ms_per_step is that measured time",
        "ms_per_layer_extrapolated": 1000.0 * w.T / tps,
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{round(sum(x[1] for x in per_step) * w.k)} random (token, expert slot) pairs "
                                   f"over {args.steps} steps = {sum(x[1] for x in per_step):.3g} token equivalents "
                                   f"(float64 numpy oracle: quantise, FC1, SiTU, requantise, FC2, combine of one "
                                   f"slot per pair; the routing of all tokens is done once before the steps)"},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_ours(args):
    import torch
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(ws, "nccl")
    import mxfp8_mxfp4_moe_gb300 as K
    st = K.kmoe_check_device(local)
    if st != 0:
        raise SystemExit(f"kmoe_check_device: {K.kmoe_status_string(st)}")
    peaks, peaks_kind = measured_peaks()

    # ---- the five workloads, timed in interleaved rounds; the headline is T=8192
    wp = W.WORKLOADS[HEADLINE]
    layer = Layer(wp, device)
    weights = layer.weights
    layers = {}
    for n in INTERLEAVED:
        w_ = W.WORKLOADS[n]
        if n == HEADLINE:
            layers[n] = layer
        elif (w_.E, w_.H, w_.I) == (wp.E, wp.H, wp.I):
            layers[n] = Layer(w_, device, weights=weights)   # the same 896 experts
        else:
            layers[n] = Layer(w_, device)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()  # running well before the timed region begins
    for L in layers.values():
        for _ in range(args.warmup):
            L.forward()
    torch.cuda.synchronize()
    for L in layers.values():
        L.check()
    rounds, counts = time_interleaved(layers, args.steps, dist, clocks, flush)
    clk = clocks.stop() if clocks else None
    for L in layers.values():
        L.check()
    med = {n: statistics.median(v) for n, v in rounds.items()}
    tokens_s, ms_step = job_throughput(dist, ws, wp.T, 1, med[HEADLINE], device)
    tflops = wp.flops() / (ms_step / 1e3) / 1e12
    # the FP8 peak: 2 x the measured bf16 burst when the SM clock stayed near
    # its maximum through the timed region, else 2 x the sustained figure
    sm, sm_max = (clk or {}).get("sm_mhz"), (clk or {}).get("sm_max_mhz")
    near_max = bool(sm and sm_max and sm >= 0.97 * sm_max)
    bf16_kind = "bf16_tflops" if near_max else "bf16_tflops_sustained"
    fp8_peak = 2.0 * peaks[bf16_kind]
    peak_source = (f"{peaks_kind}: 2 x {bf16_kind} (nominal FP8/BF16 ratio 2); "
                   f"{'burst' if near_max else 'sustained'} because the median SM clock in the timed region was "
                   f"{sm} MHz of {sm_max} MHz")
    configs = {}
    for n in INTERLEAVED:
        w_, L, m = W.WORKLOADS[n], layers[n], reduce_max(dist, med[n], device)
        touched = L.touched_experts()
        wbytes = touched * w_.expert_weight_bytes()
        alg = wbytes + 2.0 * w_.T * w_.H * 2 + 4.0 * w_.T * w_.E + 4.0 * w_.E
        configs[n] = {
            "workload": WORKLOAD_TEXT[n], "us_per_layer": 1000.0 * m, "tokens_per_s": w_.T / (m / 1e3),
            "tflops": w_.flops() / (m / 1e3) / 1e12, "fp8_frac": w_.flops() / (m / 1e3) / 1e12 / fp8_peak,
            "touched_experts": touched, "algorithmic_bytes": alg, "layer_GBs": alg / (m / 1e3) / 1e9,
            "hbm_frac": alg / (m / 1e3) / 1e9 / peaks["hbm_gbs"],
            "tile_rows": tile_classes(K, L.p),
            "rounds_ms": rounds[n], "forwards_per_round": [c for c in counts[n] if c],
            "timing": ("each forward timed alone after a write of 2 x L2 (inputs fit in L2)" if n in FLUSHED
                       else "back-to-back forwards (weights larger than L2)")}
    # kernels of this library launched in the timed region (kernel_launches per forward)
    gpu_launches = sum(sum(counts[n]) * kernel_launches(W.WORKLOADS[n]) for n in layers)
    stages = time_stages(layer, max(3, min(args.steps, 10)))
    layer.check()
    fc1_ms = stages[3]
    fc1_flops = 4.0 * wp.R * wp.H * wp.I
    fc1_tf = fc1_flops / (fc1_ms / 1e3) / 1e12
    traffic = fc1_traffic_record()
    e2e_ms, h2d, d2h = e2e_time(layer, args.steps, max(1, args.warmup // 2))
    e2e_tok_s, e2e_ms = job_throughput(dist, ws, wp.T, args.steps, e2e_ms, device)
    touched_p = configs[HEADLINE]["touched_experts"]

    # ---- decode: T=16 (same experts, same weights)
    wd = W.WORKLOADS[DECODE]
    dl = layers[DECODE]
    d_us = configs[DECODE]["us_per_layer"]
    d_stages = time_stages(dl, 10)
    touched = configs[DECODE]["touched_experts"]
    dl.check()
    per_expert_w13 = 2 * wd.I * wd.H // 2 + 2 * wd.I * wd.H // 32
    d_fc1_gbs = touched * per_expert_w13 / (d_stages[3] / 1e3) / 1e9
    d_layer_gbs = configs[DECODE]["layer_GBs"]
    d_graph_us = time_graph(dl, 20)
    d_traffic = decode_traffic_record()
    dl.check()
    del dl, layers, flush
    torch.cuda.empty_cache()

    # ---- the SwiGLU control activation on the same prefill layer (same weights)
    wsg = wp.with_(name="prefill_swiglu", activation="swiglu")
    sl = Layer(wsg, device, weights=weights)
    sg_total, _ = time_layer(sl, args.steps, args.warmup, dist, device, None)
    sg_total = reduce_max(dist, sg_total, device)
    sg_ms = sg_total / args.steps
    sg_stages = time_stages(sl, max(3, min(args.steps, 10)))
    sl.check()
    swiglu_control = {
        "workload": "Kimi-K3 MoE layer prefill chunk T=8192 H=7168 I=3584 E=896 top-16, clamped SwiGLU "
                    f"(alpha {wsg.swiglu_alpha}, beta {wsg.swiglu_beta}, limit {wsg.swiglu_limit}) in place of SiTU",
        "ms_per_layer": sg_ms, "tokens_per_s": wsg.T / (sg_ms / 1e3),
        "tflops": wsg.flops() / (sg_ms / 1e3) / 1e12,
        "stages_ms": dict(zip(K.STAGE_NAMES, sg_stages)),
    }
    # ---- the fused router (gate GEMM + routing in one kernel) on the same prefill layer
    rl_ = Layer(wp, device, weights=weights)
    rl_.router = True
    fr_total, _ = time_layer(rl_, args.steps, args.warmup, dist, device, None)
    fr_total = reduce_max(dist, fr_total, device)
    fr_ms = fr_total / args.steps
    fr_stages = time_stages(rl_, max(3, min(args.steps, 10)))
    rl_.check()
    # ---- and on the decode layer: the router's stage inside back-to-back forwards
    # (the previous forward's weight stream leaves the L2 holding clean lines)
    rd_ = Layer(W.WORKLOADS[DECODE], device, weights=weights)
    rd_.router = True
    frd_total, _ = time_layer(rd_, max(args.steps, 20), args.warmup, dist, device, None)
    frd_us = 1000.0 * reduce_max(dist, frd_total, device) / max(args.steps, 20)
    frd_stages = time_stages(rd_, 10)
    rd_.check()
    del sl, rl_, rd_, weights, layer
    torch.cuda.empty_cache()
    r_pre = time_router(wp, device)
    r_dec = time_router(W.WORKLOADS[DECODE], device)
    router = {
        "what": "gate GEMM (bf16 x bf16 -> fp32 logits on tcgen05) and sigmoid + bias top-16 routing in one "
                "kernel; L2 flushed before each timed launch",
        "prefill_T8192": r_pre, "decode_T16": r_dec,
        "layer_with_fused_router_T8192": {"ms_per_layer": fr_ms, "tokens_per_s": wp.T / (fr_ms / 1e3),
                                          "stages_ms": dict(zip(K.STAGE_NAMES, fr_stages))},
        "layer_with_fused_router_T16": {"us_per_layer": frd_us,
                                        "stages_us": {n: 1000 * v for n, v in zip(K.STAGE_NAMES, frd_stages)},
                                        "router_stage": "the route stage is the fused router inside the layer "
                                                        "(stage events around it; L2 not flushed)"},
        "roofline": {"bound": "tensor", "kernel": "router_kernel (prefill T=8192)",
                     "achieved": r_pre["gemm_tflops"], "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": r_pre["gemm_tflops"] / peaks["bf16_tflops"],
                     "peak_source": f"{peaks_kind}: bf16_tflops (burst; the kernel is timed alone)",
                     "algorithmic": "2*T*H*E FLOP per launch"},
        "decode_roofline": {"bound": "hbm", "achieved": r_dec["algorithmic_GBs"], "peak": peaks["hbm_gbs"],
                            "unit": "GB/s", "frac": r_dec["algorithmic_GBs"] / peaks["hbm_gbs"],
                            "algorithmic": "x + gate weight + bias read, logits/ids/weights written"},
    }

    # ---- the real checkpoint's expert shape (3584-wide latent, I=3072): prefill and decode
    wr = W.NEXT_WORKLOADS["real_prefill"]
    rl = Layer(wr, device)
    r_total, _ = time_layer(rl, args.steps, args.warmup, dist, device, None)
    r_total = reduce_max(dist, r_total, device)
    r_ms = r_total / args.steps
    r_stages = time_stages(rl, max(3, min(args.steps, 10)))
    rl.check()
    r_weights = rl.weights
    del rl
    torch.cuda.empty_cache()
    wrd = W.NEXT_WORKLOADS["real_decode"]
    rdl = Layer(wrd, device, weights=r_weights)
    rd_total, _ = time_layer(rdl, max(args.steps, 20), args.warmup, dist, device, None)
    rd_total = reduce_max(dist, rd_total, device)
    rd_us = 1000.0 * rd_total / max(args.steps, 20)
    rd_touched = rdl.touched_experts()
    rdl.check()
    rd_bytes = rd_touched * wrd.expert_weight_bytes() + 2 * wrd.T * wrd.H * 2 + 4 * wrd.T * wrd.E
    del rdl, r_weights
    torch.cuda.empty_cache()
    real_shape = {
        "workload": "Kimi-K3 real checkpoint expert shape H=3584 I=3072 E=896 top-16",
        "prefill_T8192": {"ms_per_layer": r_ms, "tokens_per_s": wr.T / (r_ms / 1e3),
                          "tflops": wr.flops() / (r_ms / 1e3) / 1e12,
                          "frac_of_fp8_peak": wr.flops() / (r_ms / 1e3) / 1e12 / fp8_peak,
                          "stages_ms": dict(zip(K.STAGE_NAMES, r_stages))},
        "decode_T16": {"us_per_layer": rd_us, "touched_experts": rd_touched,
                       "layer_GBs": rd_bytes / (rd_us / 1e6) / 1e9,
                       "layer_hbm_frac": rd_bytes / (rd_us / 1e6) / 1e9 / peaks["hbm_gbs"]},
    }

    peak_mma = mma_peak(device)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        tps, ntok, secs, cores = oracle_slot_sample(wp, args.cpu_budget_s, 0, oracle_inputs(wp))
        cpu = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{round(ntok * wp.k)} random (token, expert slot) pairs of the T=8192 layer = "
                         f"{ntok:.3g} token equivalents ({secs:.1f} s of float64 oracle work: quantise, FC1, "
                         f"SiTU, requantise, FC2, combine of one slot per pair; routing of all tokens done once "
                         f"before)"}

    if rank == 0:
        # `config` is the reference arm's, key for key; the run's details sit beside it
        cfg = headline_config(ws)
        details = {"tile_rows": configs[HEADLINE]["tile_rows"], "touched_experts": touched_p,
                   "timing": f"{ROUNDS} interleaved rounds (each: the five workloads in turn), median; "
                             f"{[c for c in counts[HEADLINE] if c]} back-to-back T=8192 forwards per round"}
        line = {
            "metric": METRIC, "value": tokens_s, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "mxfp8xmxfp4 (e4m3 x e2m1, ue8m0 scales, fp32 accumulate, bf16 out)",
            "data": "synthetic (seeded; random MXFP4 weights of the Kimi-K3 expert shapes)",
            "config": cfg,
            "run": details,
            "tflops": tflops,
            "stages_ms": dict(zip(K.STAGE_NAMES, stages)),
            "roofline": {"bound": "tensor", "kernel": "FC1 grouped GEMM (tcgen05 mxf8f6f4, SiTU+requant epilogue)",
                         "achieved": fc1_tf, "peak": fp8_peak, "unit": "TFLOP/s", "frac": fc1_tf / fp8_peak,
                         "peak_source": peak_source, "sm_mhz_median": sm,
                         "algorithmic": f"4*R*H*I = {fc1_flops:.4g} FLOP per launch",
                         "traffic": (traffic["dram_bytes_per_launch"] if traffic else None),
                         "frac_of_measured_mma_roof": fc1_tf / peak_mma["tflops"],
                         "layer": {"achieved": tflops, "frac": tflops / fp8_peak,
                                   "frac_of_measured_mma_roof": tflops / peak_mma["tflops"],
                                   "algorithmic": "6*R*H*I FLOP per layer"}},
            "configs": configs,
            "mma_peak_measured": peak_mma,
            "real_shape": real_shape,
            "swiglu_control": swiglu_control,
            "router": router,
            "decode": {"workload": "Kimi-K3 MoE layer decode T=16 H=7168 I=3584 E=896 top-16",
                       "us_per_layer": d_us, "us_per_layer_cuda_graph": d_graph_us,
                       "touched_experts": touched, "layer_GBs": d_layer_gbs,
                       "layer_hbm_frac": d_layer_gbs / peaks["hbm_gbs"],
                       "stages_us": {n: 1000 * v for n, v in zip(K.STAGE_NAMES, d_stages)},
                       "roofline": {"bound": "hbm", "kernel": "FC1 grouped GEMM", "achieved": d_fc1_gbs,
                                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                    "frac": d_fc1_gbs / peaks["hbm_gbs"],
                                    "algorithmic": f"touched experts x {per_expert_w13} B of w13 codes+scales",
                                    "traffic": (touched * d_traffic["dram_bytes_per_touched_expert"]
                                                if d_traffic else None)}},
            "e2e": {"value": e2e_tok_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": gpu_launches,
            "clocks": clk,
            "cpu_baseline": cpu,
            "device": torch.cuda.get_device_name(device),
        }
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_profile(args):
    """Lean mode for profiler captures: one workload, warm-up + steps forwards,
    stage times printed as JSON (no clocks, baselines or e2e).  "route:NAME"
    runs only the routing kernel on workload NAME's logits and "router:NAME"
    only the fused router on its x and gate weight (no expert weights on the
    device), for multi-pass captures of those kernels."""
    import torch
    torch.cuda.set_device(0)
    if args.profile.startswith("route:"):
        import mxfp8_mxfp4_moe_gb300 as K
        w = W.WORKLOADS[args.profile.split(":", 1)[1]]
        s = W.gen_small_inputs(w)
        logits = torch.from_numpy(s["logits"]).cuda()
        bias = torch.from_numpy(s["bias"]).cuda()
        ids = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
        wts = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
        for _ in range(args.warmup + args.steps):
            K.kmoe_route(logits, bias, w.k, ids, wts)
        torch.cuda.synchronize()
        print(json.dumps({"profile": args.profile, "T": w.T, "E": w.E, "k": w.k}))
        return 0
    if args.profile.startswith("router:"):
        import mxfp8_mxfp4_moe_gb300 as K
        w = W.WORKLOADS[args.profile.split(":", 1)[1]]
        s = W.gen_small_inputs(w)
        x = torch.from_numpy(s["x"].view(np.int16)).view(torch.bfloat16).cuda()
        wg = torch.from_numpy(s["wg"].view(np.int16)).view(torch.bfloat16).cuda()
        bias = torch.from_numpy(s["bias"]).cuda()
        ws = torch.zeros(K.kmoe_router_workspace_size(w.T, w.H, w.E), dtype=torch.uint8, device="cuda")
        for _ in range(args.warmup + args.steps):
            K.kmoe_router(x, wg, bias, w.k, workspace=ws)
        torch.cuda.synchronize()
        st, word = K.kmoe_device_error(ws)
        print(json.dumps({"profile": args.profile, "T": w.T, "H": w.H, "E": w.E, "k": w.k, "device_error": word}))
        return 0 if st == 0 else 1
    w = {**W.WORKLOADS, **W.PROFILE_WORKLOADS}[args.profile]
    layer = Layer(w, torch.device("cuda", 0))
    for _ in range(args.warmup + args.steps):
        layer.forward(stage_events=True)
    torch.cuda.synchronize()
    layer.check()
    import mxfp8_mxfp4_moe_gb300 as K
    print(json.dumps({"profile": w.name, "stages_ms": dict(zip(K.STAGE_NAMES, layer.stage_ms())),
                      "touched_experts": layer.touched_experts(),
                      "tile_rows": tile_classes(K, layer.p)}))
    return 0


def tile_classes(K, p):
    """Token-tile sizes of a layer: small tiles for experts with at most
    big_rows rows, big (CTA-pair) tiles for the others (0: none possible)."""
    L = K.kmoe_workspace_layout(p)
    return {"small": L.tile_rows, "big": L.tile_rows_big, "big_above_rows": L.big_rows}


def layer_params(K, w):
    return K.make_params(w.T, w.H, w.I, w.E, w.k, w.situ_beta, w.situ_linear_beta, w.routed_scaling_factor,
                         activation=w.activation, swiglu_alpha=w.swiglu_alpha, swiglu_beta=w.swiglu_beta,
                         swiglu_limit=w.swiglu_limit)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--ref-step-s", type=float, default=1.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", default=None, help="lean run of one workload (for profiler captures)")
    args = ap.parse_args(argv)
    if args.profile:
        return run_profile(args)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
