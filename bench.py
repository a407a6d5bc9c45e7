"""Benchmark of the MoE layer step on GB300.

One full-shape layer -- hidden 7168, expert intermediate 1536, 896 routed MXFP4 experts
resident in HBM (15.7 GB), top-16, one bf16 shared expert 7168x1536 -- with seeded
synthetic inputs (synth/).  The default run times, in one process and on one resident
expert pool:

  decode1        1 token per step (the headline: value, e2e, roofline, cpu_baseline);
  decode64_zipf  64 tokens per step, expert popularity Zipf(1.1) through the bias;
  decode64_uniform  64 tokens per step, uniform routing;
  prefill4096    4096 tokens per step, uniform routing, grouped GEMMs on tcgen05;
  stacked8       1 token per step through 8 stacked layers (126 GB of MXFP4 resident),
                 RMSNorm and the residual stream in between;
  latent_decode1 1 token per step through the pages' LatentMoE layer (experts in a
                 3584-wide latent, its own 15.7 GB pool, two shared experts);
  streamed_decode1  1 token per step with the records in pinned host memory and 256
                 device slots in front of them (the LRU expert cache);

the last six as nested entries of the one JSON line (``workloads``; at one GPU only -- a
multi-GPU run times the headline).  ``--workload``
times one of them alone as the line's headline.  Timed regions: blocks of exactly K
steps, each between a barrier and a synchronize, repeated until at least a second of
load has passed so that the clock sampler sees the timed work; every step between CUDA
events on the launching stream; L2 flushed between steps (outside the events) except
for stacked8, whose inputs are larger than L2.

``--impl reference`` times the CPU oracle instead (the reference arm of this
comparison), on the decode1 workload, metric and unit.

N > 1 (torchrun): the layer step does not shard without an exchange step, so every rank
runs an independent replica; value = tokens processed by all ranks / max rank time.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer decode tokens/s & HBM GB/s vs ~8 TB/s; prefill tcgen05 % peak"
WORKLOADS = {
    "decode1": "decode1: 1 token/step through one full-shape MoE layer (hidden 7168, inter "
               "1536, 896 MXFP4 experts top-16, 1 bf16 shared expert 7168x1536)",
    "decode64_zipf": "decode64_zipf: 64 tokens/step through one full-shape MoE layer, expert "
                     "popularity Zipf(1.1) through the correction bias",
    "decode64_uniform": "decode64_uniform: 64 tokens/step through one full-shape MoE layer, "
                        "uniform routing",
    "prefill4096": "prefill4096: 4096 tokens/step through one full-shape MoE layer, uniform "
                   "routing (grouped MXFP4 GEMM on tcgen05)",
    "stacked8": "stacked8: 1 token/step through 8 stacked full-shape MoE layers (126 GB of "
                "MXFP4 resident) with RMSNorm and the residual stream between them",
    "streamed_decode1": "streamed_decode1: 1 token/step through one full-shape MoE layer whose "
                        "896 MXFP4 expert records live in pinned host memory, read over the "
                        "host link into 256 device slots by the LRU expert cache",
    "latent_decode1": "latent_decode1: 1 token/step through the pages' LatentMoE layer (hidden "
                      "7168, 896 MXFP4 experts top-16 in a 3584-wide latent with inter 3072, "
                      "latent RMSNorm, 2 bf16 shared experts of 3072 on the full width)",
}
WORKLOAD = WORKLOADS["decode1"]
DEFAULT_STEPS = {"decode1": 3000, "decode64_zipf": 200, "decode64_uniform": 200,
                 "prefill4096": 40, "stacked8": 256,
                 "latent_decode1": 1000, "streamed_decode1": 200}
MIN_TIMED_SECONDS = 1.0

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu
# capture of the decode kernel, keyed to a hash of the sources it is compiled from (its
# translation unit and the headers that unit includes): a changed kernel reports null
# until it is captured again.
TRAFFIC_SOURCES = ["mxfp4_routed_expert_02_gb300/csrc/k3moe_decode_fused.cu",
                   "mxfp4_routed_expert_02_gb300/csrc/k3moe_kernels.cuh",
                   "mxfp4_routed_expert_02_gb300/csrc/k3moe_device.cuh",
                   "mxfp4_routed_expert_02_gb300/csrc/k3moe_topk.cuh",
                   "include/k3moe.h"]
# k_decode_fused: captured with a 64-expert pool (347,873,280 B read + 2,811,392 B written
# per launch), plus the router rows the full 896-expert pool adds ((896 - 64) x 7168 x 2 B):
# every other byte the kernel reads is the same at both pool sizes (16 selected experts,
# the shared expert).
TRAFFIC_CAPTURED = {"sources": "8f9947976e789b9b",
                    "bytes": {"k_decode_fused": 347873280 + 2811392 + (896 - 64) * 7168 * 2}}


def traffic_of(kernel):
    import hashlib
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    if h.hexdigest()[:16] != TRAFFIC_CAPTURED["sources"]:
        return None
    return TRAFFIC_CAPTURED["bytes"].get(kernel)


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except OSError:
        return None


def step_bytes(cfg, U):
    """Algorithmic bytes of one decode step with U distinct routed experts."""
    H, I, E, SI = cfg.hidden, cfg.inter, cfg.n_experts, cfg.shared_inter
    op = I * H // 2 + I * H // 32            # one MXFP4 operand (packed + scales)
    gate_up = U * 2 * op                    # W1 and W3 of each distinct expert
    down = U * op + H * SI * 2 + H * 4       # W2 of each distinct expert, shared W2s, y
    router = E * H * 2 + 2 * SI * H * 2 + H * 2   # Wr, shared W1s/W3s, x
    return {
        "k_router_shared": router, "k_router_t1": router,
        "k_expert_gateup": gate_up, "k_gateup_t1": gate_up,
        "k_down_combine": down, "k_down_tma": down, "k_down_t1": down,
        "k_decode_fused": router + gate_up + down,  # the whole step in one kernel
    }


class Clocks:
    """nvidia-smi sampling (200 ms) during the timed region."""

    def __init__(self, path):
        self.path = path
        self.p = None

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.p = subprocess.Popen(["nvidia-smi", "--query-gpu=" + q, "--format=csv,noheader",
                                       "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
            t0 = time.time()
            while time.time() - t0 < 3.0 and os.path.getsize(self.path) == 0:
                time.sleep(0.02)  # sampling is running before the timed region starts
        except OSError:
            self.p = None
        return self

    def __exit__(self, *a):
        if self.p is not None:
            self.p.terminate()
            self.p.wait()
            self.f.close()

    def summary(self, dev_index=0):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": []}
        try:
            rows = [l.split(",") for l in open(self.path).read().strip().splitlines()]
        except OSError:
            return out
        mhz, reasons = [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9 or r[0] != str(dev_index):
                continue
            try:
                mhz.append(float(r[1].split()[0]))
                out["sm_max_mhz"] = float(r[2].split()[0])
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if mhz:
            out["sm_mhz"] = statistics.median(mhz)
            out["samples"] = len(mhz)
        out["reasons"] = sorted(reasons)
        return out


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


def cpu_baseline(cfg, seed, n_tokens=2):
    """The oracle, as it stands, on a bounded sample of the same workload."""
    import oracle
    import synth
    w = synth.layer_weights(cfg, seed)
    x = synth.activations(cfg, seed + 1, n_tokens)
    cache = {}

    def rec(e):
        if e not in cache:
            cache[e] = synth.expert_record(cfg, seed, 0, e)
        return cache[e]
    # expert bytes are regenerated outside the timed region
    oi, _, _, _ = oracle.router(x, w["wr"], w["bias"], cfg.topk)
    for e in set(oi.ravel().tolist()):
        rec(int(e))
    nt = oracle.num_threads()
    t0 = time.perf_counter()
    oracle.moe_layer(x, w["wr"], w["bias"], rec, cfg.topk, cfg.hidden, cfg.inter,
                     w["sh_gate"], w["sh_up"], w["sh_down"], nthreads=nt)
    dt = time.perf_counter() - t0
    return {"value": n_tokens / dt, "unit": "tokens/s", "cores": nt, "kind": "oracle",
            "sample": "%d decode tokens through the full decode1 layer (router + 16 experts + "
                      "shared expert, fp64 accumulation)" % n_tokens}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import synth
    cfg = synth.config("decode1")
    for _ in range(args.warmup):
        cpu_baseline(cfg, 0, 1)
    vals = []
    t_all = 0.0
    for s in range(args.steps):
        r = cpu_baseline(cfg, 100 + s, 1)
        vals.append(r["value"])
        t_all += 1.0 / r["value"]
    value = args.steps / t_all
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t_all / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens_per_step": 1},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": r["cores"],
                         "kind": "oracle", "sample": "1 decode token per step, %d steps"
                                                     % args.steps},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def reduce_max(dist, value, device):
    """The largest of the ranks' values, returned on every rank (the value itself when
    there is one rank): the job's time is its slowest rank's."""
    if dist is None:
        return value
    import torch
    tt = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_rate(units_per_rank, world, seconds):
    """Whole-job throughput of independent replicas: the units all ranks processed over
    the slowest rank's time."""
    return units_per_rank * world / seconds


def blocks_needed(block_seconds, min_seconds=MIN_TIMED_SECONDS):
    """Timed blocks of K steps so that the timed work lasts at least min_seconds."""
    if block_seconds <= 0:
        return 1
    return max(1, int(math.ceil(min_seconds / block_seconds)))


class Timer:
    """Timed blocks of exactly K steps, each between a barrier and a synchronize, with
    per-step CUDA events on the launching stream and nvidia-smi sampling throughout."""

    def __init__(self, ctx, tag):
        self.ctx, self.tag = ctx, tag

    def run(self, step, K, W, flush=None):
        import torch
        c = self.ctx
        for s in range(W):
            if flush:
                flush(s)
            step(s)
        torch.cuda.synchronize()
        clocks = Clocks("/tmp/k3moe_bench_clocks_%s_%d_%d.csv" % (self.tag, os.getpid(), c.rank))
        per_step, blocks, nb = [], 0, 1
        with clocks:
            t_wall = time.perf_counter()
            while blocks < nb:
                ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                      for _ in range(K)]
                if c.dist:
                    c.dist.barrier()
                torch.cuda.synchronize()
                tb = time.perf_counter()
                for s in range(K):
                    i = W + blocks * K + s
                    if flush:
                        flush(i)
                    ev[s][0].record(c.stream)
                    step(i)
                    ev[s][1].record(c.stream)
                torch.cuda.synchronize()
                if c.dist:
                    c.dist.barrier()
                per_step += [a.elapsed_time(b) for a, b in ev]
                if blocks == 0:  # every rank runs the slowest rank's number of blocks
                    nb = int(reduce_max(c.dist, blocks_needed(time.perf_counter() - tb,
                                                              c.min_seconds), c.dev))
                blocks += 1
            t_wall = time.perf_counter() - t_wall
        self.blocks, self.wall = blocks, t_wall
        self.clocks = clocks.summary(c.local)
        self.ms = per_step
        # the job's device time: the slowest rank's sum of step times
        self.t_dev = reduce_max(c.dist, sum(per_step) / 1e3, c.dev)
        return self


class Ctx:
    """Device, process group, the resident expert pool and the layer's small weights."""

    def __init__(self, args):
        import torch
        self.rank, self.world, self.local = dist_env()
        torch.cuda.set_device(self.local)
        self.dist = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("nccl")
            self.dist = dist
        import synth
        import synth.device as sd
        import mxfp4_routed_expert_02_gb300 as k3
        self.k3, self.synth, self.sd = k3, synth, sd
        self.dev = torch.device("cuda", self.local)
        self.stream = torch.cuda.current_stream()
        self.seed = 0
        cfg = synth.config("decode1")
        if args.experts != cfg.n_experts:   # smaller expert pool: profiling captures only
            cfg = synth.config("decode1", n_experts=args.experts)
        self.cfg = cfg
        self.stride = (cfg.record_bytes + 4095) // 4096 * 4096
        self.experts = torch.empty(cfg.n_experts * self.stride, dtype=torch.uint8, device=self.dev)
        sd.fill_experts(self.experts, cfg, self.seed, 0, stride=self.stride)
        self.w = synth.layer_weights(cfg, self.seed)
        t = self.t
        self.wr, self.bias = t(self.w["wr"].view(np.int16)), t(self.w["bias"])
        self.sg, self.su, self.sdn = (t(self.w[k].view(np.int16))
                                      for k in ("sh_gate", "sh_up", "sh_down"))
        self.flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=self.dev)
        self.flush_words = self.flush_buf.view(torch.int32)
        self.flush_mode = args.flush
        self.min_seconds = args.min_seconds

    def t(self, a):
        import torch
        return torch.from_numpy(np.ascontiguousarray(a)).to(self.dev)

    def flush(self, s):
        """Evict L2 between timed steps (outside the step's events): a 256 MB write, or a
        256 MB read that leaves no dirty lines behind."""
        if self.flush_mode == "write":
            self.flush_buf.fill_(s & 255)
        else:
            self.flush_words.sum()

    def flush_note(self):
        return ("flushed between timed steps (256 MB %s, outside the step events)" %
                self.flush_mode)


def traced(ctx, step, n, first, flush=None):
    """Per-kernel device times: n steps again with the library's event tracing on (it
    brackets every launch with events and turns off programmatic overlap)."""
    import torch
    k3 = ctx.k3
    k3.k3moe_trace_enable(True)
    for s in range(n):
        if flush:
            flush(first + s)
        step(first + s)
    torch.cuda.synchronize()
    trace = k3.k3moe_trace_read()
    k3.k3moe_trace_enable(False)
    return {k: v for k, v in trace.items() if v[1]}


def e2e_pipelined(ctx, x_host, NX, K, H, layer):
    """Seconds for K steps of `layer(x_dev, y_dev)` with host buffers: step s copies row
    s % NX of x_host (pinned) to the device and its y (H floats) back to pinned host memory.
    Two device x and y buffers alternate; the host-to-device copies run on one stream, the
    device-to-host copies on another, ordered against the layer by events, so that only the
    first input and the last output are not hidden behind a neighbouring step's kernels."""
    import torch
    xh = torch.from_numpy(np.ascontiguousarray(x_host)).pin_memory()
    yh = torch.empty((K, H), dtype=torch.float32).pin_memory()
    xd = [torch.empty((1, H), dtype=xh.dtype, device=ctx.dev) for _ in range(2)]
    yd = [torch.empty((1, H), dtype=torch.float32, device=ctx.dev) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(ctx.dev), torch.cuda.Stream(ctx.dev)
    ev = lambda: [torch.cuda.Event() for _ in range(2)]  # noqa: E731
    in_done, k_done, out_done = ev(), ev(), ev()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def h2d(s):
        b = s % 2
        if s >= 2:
            s_in.wait_event(k_done[b])       # step s-2 has read this buffer
        with torch.cuda.stream(s_in):
            xd[b].copy_(xh[s % NX:s % NX + 1], non_blocking=True)
        in_done[b].record(s_in)

    torch.cuda.synchronize()
    e0.record(ctx.stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    h2d(0)
    for s in range(K):
        b = s % 2
        if s + 1 < K:
            h2d(s + 1)
        ctx.stream.wait_event(in_done[b])
        if s >= 2:
            ctx.stream.wait_event(out_done[b])  # y of step s-2 has left this buffer
        layer(xd[b], yd[b])
        k_done[b].record(ctx.stream)
        s_out.wait_event(k_done[b])
        with torch.cuda.stream(s_out):
            yh[s].copy_(yd[b][0], non_blocking=True)
        out_done[b].record(s_out)
    ctx.stream.wait_event(out_done[(K - 1) % 2])
    e1.record(ctx.stream)
    torch.cuda.synchronize()
    return reduce_max(ctx.dist, e0.elapsed_time(e1) / 1e3, ctx.dev)


def bench_decode1(ctx, args, K):
    """The headline: one decode token per step."""
    import torch
    k3, synth, cfg = ctx.k3, ctx.synth, ctx.cfg
    H, I, E, Kt = cfg.hidden, cfg.inter, cfg.n_experts, cfg.topk
    dims = k3.LayerDims(H, I, E, Kt, cfg.shared_inter)
    NX = 256
    xs_host = synth.activations(cfg, ctx.seed + 1 + ctx.rank, NX)
    xs = ctx.t(xs_host.view(np.int16))
    y = torch.empty((1, H), dtype=torch.float32, device=ctx.dev)
    idx = torch.empty((NX, Kt), dtype=torch.int32, device=ctx.dev)
    wt = torch.empty((NX, Kt), dtype=torch.float32, device=ctx.dev)
    ws = k3.new_workspace(dims, 1, ctx.dev)
    status = k3.new_status(ctx.dev)

    def step(s):
        j = s % NX
        k3.k3moe_layer(dims, xs[j:j + 1], ctx.wr, ctx.bias, ctx.experts, ctx.stride, ctx.sg,
                       ctx.su, ctx.sdn, y, ws, status, idx_out=idx[j:j + 1], w_out=wt[j:j + 1])

    tm = Timer(ctx, "decode1").run(step, K, args.warmup, ctx.flush)
    assert status.item() == 0, k3.status_str(status.item())
    nsteps = tm.blocks * K
    trace = traced(ctx, step, nsteps, args.warmup, ctx.flush)

    # distinct experts actually used per step (for the algorithmic bytes)
    steps_idx = idx.cpu().numpy()
    used = [len(set(steps_idx[(args.warmup + s) % NX].tolist())) for s in range(nsteps)]
    U = statistics.mean(used)
    nb = step_bytes(cfg, U)
    bytes_step = nb["k_decode_fused"]
    launches = sum(v[1] for v in trace.values())
    kernels = {k: {"ms_avg": v[0] / v[1], "launches": v[1]} for k, v in trace.items()}
    # the dominant kernel: most device time among the kernels that stream the weights
    dom = max((k for k in kernels if k in nb),
              key=lambda k: kernels[k]["ms_avg"] * kernels[k]["launches"])
    pk = peaks()
    peak_hbm = pk["hbm_gbs"] if pk else 6800.0
    achieved = nb[dom] / (kernels[dom]["ms_avg"] * 1e-3) / 1e9
    for k in kernels:
        if k in nb:
            kernels[k]["gbs"] = nb[k] / (kernels[k]["ms_avg"] * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak_hbm, "unit": "GB/s",
                "frac": achieved / peak_hbm,
                # the captured bytes are those of the full 896-expert pool
                "traffic": traffic_of(dom) if cfg.n_experts == 896 else None, "kernel": dom,
                "algorithmic_bytes": nb[dom],
                "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if pk else
                               "fallback 6.8 TB/s (of fallback)"}

    # end to end through the C ABI with host buffers: every step copies its token in from
    # pinned host memory and its y back to pinned host memory, as a serving loop would:
    # the copies run on two copy streams with two device buffers each, so the input of
    # step s+1 lands and the output of step s-1 leaves while step s computes
    t_e2e = e2e_pipelined(ctx, xs_host.view(np.int16), NX, K, H, lambda xd, yd: k3.k3moe_layer(
        dims, xd, ctx.wr, ctx.bias, ctx.experts, ctx.stride, ctx.sg, ctx.su, ctx.sdn, yd, ws,
        status))
    assert status.item() == 0, k3.status_str(status.item())

    return {
        "metric": METRIC, "value": job_rate(nsteps, ctx.world, tm.t_dev), "unit": "tokens/s",
        "n_gpus": ctx.world, "steps": K, "warmup": args.warmup,
        "ms_per_step": 1e3 * tm.t_dev / nsteps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOADS["decode1"], "tokens_per_step": 1, "seed": ctx.seed,
                   "l2": ctx.flush_note(), "distinct_experts_per_step": U,
                   "timed_blocks": tm.blocks,
                   "parallelism": "replicas" if ctx.world > 1 else "single"},
        "hbm_gbs_step": bytes_step / (tm.t_dev / nsteps) / 1e9,
        "algorithmic_bytes_per_step": bytes_step,
        "roofline": roofline,
        "kernels": kernels,
        "gpu_launches": launches,
        "clocks": tm.clocks,
        "e2e": {"value": job_rate(K, ctx.world, t_e2e), "unit": "tokens/s",
                "h2d_bytes_per_step": H * 2, "d2h_bytes_per_step": H * 4,
                "copies": "pinned host x in, y out, every step; double-buffered on two copy "
                          "streams beside the layer",
                "l2": "not flushed: each step reads ~360 MB of weights out of a 15.7 GB expert "
                      "pool, above the 129 MB L2"},
        "wall_s": tm.wall,
    }


def useful_flops(cfg, P, T):
    """Multiply-adds x 2 of the expert GEMMs for P (token, slot) pairs and T tokens."""
    H, I, SI = cfg.hidden, cfg.inter, cfg.shared_inter
    return 2.0 * P * 3 * H * I + 2.0 * T * 3 * H * SI


def bench_batch(ctx, name, args, K, tokens=0):
    """decode64_zipf / prefill4096 (one layer, many tokens) or stacked8 (eight layers, one
    token), on the resident pool (the pool is layer 0 of the stack)."""
    import torch
    k3, synth, sd = ctx.k3, ctx.synth, ctx.sd
    cfg = synth.config("decode1" if name == "stacked8" else name,
                       n_experts=ctx.cfg.n_experts)
    L = 8 if name == "stacked8" else 1
    T = 1 if name == "stacked8" else (tokens or cfg.tokens)
    H, I, E, Kt = cfg.hidden, cfg.inter, cfg.n_experts, cfg.topk
    dims = k3.LayerDims(H, I, E, Kt, cfg.shared_inter)
    stride = ctx.stride
    layers = [dict(wr=ctx.wr, bias=ctx.bias, experts=ctx.experts, stride=stride, sh_gate=ctx.sg,
                   sh_up=ctx.su, sh_down=ctx.sdn)]
    if name == "decode64_zipf":   # same weights, the bias that steers popularity
        layers[0]["bias"] = ctx.t(synth.layer_weights(cfg, ctx.seed)["bias"])
    for l in range(1, L):
        ex = torch.empty(E * stride, dtype=torch.uint8, device=ctx.dev)
        sd.fill_experts(ex, cfg, ctx.seed, l, stride=stride)
        w = synth.layer_weights(cfg, ctx.seed, l)
        layers.append(dict(wr=ctx.t(w["wr"].view(np.int16)), bias=ctx.t(w["bias"]), experts=ex,
                           stride=stride, sh_gate=ctx.t(w["sh_gate"].view(np.int16)),
                           sh_up=ctx.t(w["sh_up"].view(np.int16)),
                           sh_down=ctx.t(w["sh_down"].view(np.int16))))
    ws = k3.new_workspace(dims, T, ctx.dev)
    status = k3.new_status(ctx.dev)
    NX = 4
    xs_host = [synth.activations(cfg, ctx.seed + 1 + ctx.rank * NX + j, T) for j in range(NX)]
    xs = [ctx.t(a.view(np.int16)) for a in xs_host]
    y = torch.empty((T, H), dtype=torch.float32, device=ctx.dev)
    idx = torch.empty((L, T, Kt), dtype=torch.int32, device=ctx.dev)
    wts = torch.empty((L, T, Kt), dtype=torch.float32, device=ctx.dev)
    h = ctx.t((xs_host[0].astype(np.uint32) << 16).view(np.float32))
    xsc = torch.empty((T, H), dtype=torch.int16, device=ctx.dev)
    lw = layers[0]

    def step(s):
        if name == "stacked8":
            k3.k3moe_decode_stack(dims, layers, h, xsc, ws, status, eps=cfg.rms_eps,
                                  idx_out=idx, w_out=wts)
        else:
            k3.k3moe_layer(dims, xs[s % NX], lw["wr"], lw["bias"], lw["experts"], stride,
                           lw["sh_gate"], lw["sh_up"], lw["sh_down"], y, ws, status,
                           idx_out=idx[0], w_out=wts[0])

    flush = None if name == "stacked8" else ctx.flush
    tm = Timer(ctx, name).run(step, K, args.warmup, flush)
    assert status.item() == 0, k3.status_str(status.item())
    nsteps = tm.blocks * K
    ntr = min(nsteps, 3)
    trace = traced(ctx, step, ntr, args.warmup, flush)
    kernels = {k: {"ms_avg": v[0] / v[1], "launches_per_step": v[1] / ntr}
               for k, v in trace.items()}
    launches = int(sum(v[1] for v in trace.values()) / ntr * nsteps)
    # distinct experts of the last step, per layer
    ids = idx.cpu().numpy()
    U = [len(set(ids[l].ravel().tolist())) for l in range(L)]
    op = I * H // 2 + I * H // 32
    layer_bytes = [u * 3 * op + E * H * 2 + 3 * cfg.shared_inter * H * 2 + T * H * 6 for u in U]
    step_bytes_v = sum(layer_bytes)
    pk = peaks()
    peak_hbm = pk["hbm_gbs"] if pk else 6800.0
    peak_bf16 = pk["bf16_tflops"] if pk else 1900.0
    sec = tm.t_dev / nsteps
    extra = {}
    if name == "prefill4096":
        P = T * Kt
        gk = kernels.get("k_tc_gemm_gateup", {}).get("ms_avg")
        dk = kernels.get("k_tc_gemm_down", {}).get("ms_avg")
        gfl = 2.0 * P * 2 * H * I
        roofline = {"bound": "tensor", "kernel": "k_tc_gemm_gateup",
                    "achieved": gfl / (gk * 1e-3) / 1e12, "peak": 6 * peak_bf16,
                    "unit": "TFLOP/s", "frac": gfl / (gk * 1e-3) / 1e12 / (6 * peak_bf16),
                    "traffic": None,
                    "peak_source": "MXFP4 dense = measured bf16 x 6 (nominal 13.5 / 2.25)",
                    "useful_flops": gfl,
                    "issued_mma_flops": gfl * k3.k3moe.TC_TERMS_X,
                    "hbm_frac_step": step_bytes_v / sec / 1e9 / peak_hbm}
        extra = {"useful_tflops_step": useful_flops(cfg, P, T) / sec / 1e12,
                 "down_kernel_tflops": 2.0 * P * H * I / (dk * 1e-3) / 1e12 if dk else None}
    else:
        if name.startswith("decode64"):
            dom = "k_tc_gemm_gateup"
            db = sum(u * 2 * op for u in U) / L        # gate/up bytes of the distinct experts
        else:
            # the fused kernel runs up to 16 stacked layers per launch: a launch's bytes are
            # the step's bytes over the launches in a step
            dom = "k_decode_fused"
            db = sum(layer_bytes) / max(kernels.get(dom, {}).get("launches_per_step", L), 1)
        dk = kernels.get(dom, {}).get("ms_avg")
        roofline = {"bound": "hbm", "kernel": dom,
                    "achieved": db / (dk * 1e-3) / 1e9 if dk else None, "peak": peak_hbm,
                    "unit": "GB/s", "frac": db / (dk * 1e-3) / 1e9 / peak_hbm if dk else None,
                    "traffic": None, "algorithmic_bytes": db,
                    "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if pk else
                                   "fallback 6.8 TB/s (of fallback)"}
    lat = sorted(tm.ms)
    line = {
        "metric": METRIC, "value": job_rate(T * nsteps, ctx.world, tm.t_dev),
        "unit": "tokens/s", "n_gpus": ctx.world, "steps": K, "warmup": args.warmup,
        "ms_per_step": 1e3 * sec, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOADS[name], "tokens_per_step": T, "layers": L,
                   "seed": ctx.seed, "distinct_experts_per_layer": U, "timed_blocks": tm.blocks,
                   "l2": ("inputs larger than L2 (2.9 GB of weights per step)" if L > 1 else
                          ctx.flush_note())},
        "hbm_gbs_step": step_bytes_v / sec / 1e9,
        "algorithmic_bytes_per_step": step_bytes_v,
        "latency_ms": {"p50": lat[len(lat) // 2],
                       "p99": lat[min(len(lat) - 1, int(len(lat) * 0.99))]},
        "roofline": roofline, "kernels": kernels, "gpu_launches": launches,
        "clocks": tm.clocks,
    }
    line.update(extra)
    del layers, ws
    torch.cuda.empty_cache()
    return line


def latent_step_bytes(cfg, U):
    """Algorithmic bytes of one LatentMoE decode step with U distinct routed experts, per
    kernel (by trace name): the router, the projection into the latent, the experts'
    gate/up and down, the projection back, the shared experts' gate/up and down."""
    H, L, I, E, SI = cfg.hidden, cfg.latent, cfg.inter, cfg.n_experts, cfg.shared_inter
    op = I * L // 2 + I * L // 32
    return {"k_router_t1": E * H * 2 + H * 2,
            "k_proj_down": L * H * 2,
            "k_proj_up": H * L * 2 + H * 4,
            "k_proj_shared_gateup": 2 * SI * H * 2,
            "k_proj_shared_down": H * SI * 2,
            "k_gateup_t1": U * 2 * op,  # the experts' gate/up: one of the two kernels runs
            "k_gateup_tc1": U * 2 * op,
            "k_down_t1": U * op}


def bench_latent(ctx, args, K):
    """The pages' LatentMoE layer, one decode token per step, on its own expert pool (records
    of the latent layout)."""
    import torch
    k3, synth, sd = ctx.k3, ctx.synth, ctx.sd
    cfg = synth.config("latent_decode1", n_experts=ctx.cfg.n_experts)
    H, L, I, E, Kt, SI = cfg.hidden, cfg.latent, cfg.inter, cfg.n_experts, cfg.topk, cfg.shared_inter
    dims = k3.LatentDims(H, L, I, E, Kt, SI)
    stride = (cfg.record_bytes + 4095) // 4096 * 4096
    ex = torch.empty(E * stride, dtype=torch.uint8, device=ctx.dev)
    sd.fill_experts(ex, cfg, ctx.seed, 0, stride=stride)
    w = synth.layer_weights(cfg, ctx.seed)
    d = {k: ctx.t(w[k].view(np.int16)) for k in ("wr", "w_down", "w_up", "sh_gate", "sh_up",
                                                 "sh_down")}
    d["bias"], d["norm_w"] = ctx.t(w["bias"]), ctx.t(w["norm_w"])
    NX = 64
    xs = ctx.t(synth.activations(cfg, ctx.seed + 1 + ctx.rank, NX).view(np.int16))
    y = torch.empty((1, H), dtype=torch.float32, device=ctx.dev)
    idx = torch.empty((NX, Kt), dtype=torch.int32, device=ctx.dev)
    wt = torch.empty((NX, Kt), dtype=torch.float32, device=ctx.dev)
    ws = k3.new_latent_workspace(dims, 1, ctx.dev)
    status = k3.new_status(ctx.dev)

    def step(s):
        j = s % NX
        k3.k3moe_latent_layer(dims, xs[j:j + 1], d["wr"], d["bias"], d["w_down"], d["w_up"],
                              d["norm_w"], ex, stride, d["sh_gate"], d["sh_up"], d["sh_down"], y,
                              ws, status, idx_out=idx[j:j + 1], w_out=wt[j:j + 1])

    tm = Timer(ctx, "latent_decode1").run(step, K, args.warmup, ctx.flush)
    assert status.item() == 0, k3.status_str(status.item())
    nsteps = tm.blocks * K
    ntr = min(nsteps, 50)
    trace = traced(ctx, step, ntr, args.warmup, ctx.flush)
    ids = idx.cpu().numpy()
    U = statistics.mean(len(set(ids[(args.warmup + s) % NX].tolist())) for s in range(ntr))
    nb = latent_step_bytes(cfg, U)
    kernels = {k: {"ms_avg": v[0] / v[1], "launches_per_step": v[1] / ntr} for k, v in trace.items()}
    for k in kernels:
        if k in nb:
            per_launch = nb[k] / kernels[k]["launches_per_step"]
            kernels[k]["gbs"] = per_launch / (kernels[k]["ms_avg"] * 1e-3) / 1e9
    bytes_step = sum(v for k, v in nb.items() if k != "k_gateup_tc1")  # gate/up counted once
    sec = tm.t_dev / nsteps
    pk = peaks()
    peak_hbm = pk["hbm_gbs"] if pk else 6800.0
    # the step's kernels run on two streams (the shared experts beside the routed chain),
    # so a traced kernel's time includes its neighbours' share of the GPU: the roofline is
    # taken over the whole step (its algorithmic bytes over the timed step)
    achieved = bytes_step / sec / 1e9
    line = {
        "value": job_rate(nsteps, ctx.world, tm.t_dev), "unit": "tokens/s", "steps": K,
        "ms_per_step": 1e3 * sec,
        "config": {"workload": WORKLOADS["latent_decode1"], "tokens_per_step": 1,
                   "seed": ctx.seed, "distinct_experts_per_step": U, "timed_blocks": tm.blocks,
                   "l2": ctx.flush_note()},
        "hbm_gbs_step": bytes_step / sec / 1e9, "algorithmic_bytes_per_step": bytes_step,
        "hbm_frac_step": bytes_step / sec / 1e9 / peak_hbm,
        "roofline": {"bound": "hbm", "kernel": "the whole step (seven launches on two streams)",
                     "achieved": achieved, "peak": peak_hbm,
                     "unit": "GB/s", "frac": achieved / peak_hbm, "traffic": None,
                     "algorithmic_bytes": bytes_step,
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if pk else
                                    "fallback 6.8 TB/s (of fallback)"},
        "kernels": kernels,
        "gpu_launches": int(sum(v[1] for v in trace.values()) / ntr * nsteps),
        "clocks": tm.clocks,
    }
    del ex, ws
    torch.cuda.empty_cache()
    return line


def h2d_gbs(ctx, src_pinned, nbytes):
    """Rate of one large copy from pinned host memory to the device (the link's roof for
    the streamed workload), best of 5."""
    import torch
    dst = torch.empty(nbytes, dtype=torch.uint8, device=ctx.dev)
    best = 0.0
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(ctx.stream)
        dst.copy_(src_pinned[:nbytes], non_blocking=True)
        e1.record(ctx.stream)
        torch.cuda.synchronize()
        best = max(best, nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del dst
    return best


def bench_streamed(ctx, args, K, n_slots=256):
    """One decode token per step with the layer's expert records in pinned host memory and
    n_slots device slots in front of them (k3moe_layer_streamed)."""
    import torch
    k3, synth, cfg = ctx.k3, ctx.synth, ctx.cfg
    H, E, Kt = cfg.hidden, cfg.n_experts, cfg.topk
    dims = k3.LayerDims(H, cfg.inter, E, Kt, cfg.shared_inter)
    host = torch.empty(E * ctx.stride, dtype=torch.uint8, pin_memory=True)
    host.copy_(ctx.experts.view(-1)[:E * ctx.stride])        # the same records as decode1
    n_slots = min(n_slots, E)
    slots = torch.empty(n_slots * ctx.stride, dtype=torch.uint8, device=ctx.dev)
    cache = k3.ExpertCache([host.data_ptr()], E, cfg.record_bytes, ctx.stride, slots.data_ptr(),
                           n_slots, ctx.stride)
    link = h2d_gbs(ctx, host, 1 << 30)
    NX = 4096
    xs = ctx.t(synth.activations(cfg, ctx.seed + 2 + ctx.rank, NX).view(np.int16))
    y = torch.empty((1, H), dtype=torch.float32, device=ctx.dev)
    ws = k3.new_streamed_workspace(dims, 1, ctx.dev)
    status = k3.new_status(ctx.dev)

    def step(s):
        j = s % NX
        k3.k3moe_layer_streamed(dims, cache, 0, xs[j:j + 1], ctx.wr, ctx.bias, ctx.sg, ctx.su,
                                ctx.sdn, y, ws, status)

    for s in range(4 * n_slots // Kt):      # fill the slots before the warm-up proper
        step(s)
    first = cache.stats()
    tm = Timer(ctx, "streamed_decode1").run(step, K, args.warmup, ctx.flush)
    assert status.item() == 0, k3.status_str(status.item())
    nsteps = tm.blocks * K
    last = cache.stats()
    # the timed steps' hits and misses (the warm-up's are in between `first` and the region;
    # the rate over all calls since `first` is used)
    calls = nsteps + args.warmup
    misses = (last["misses"] - first["misses"]) / calls
    hits = (last["hits"] - first["hits"]) / calls
    sec = tm.t_dev / nsteps
    copy_bytes = misses * cfg.record_bytes
    line = {
        "value": job_rate(nsteps, ctx.world, tm.t_dev), "unit": "tokens/s", "steps": K,
        "ms_per_step": 1e3 * sec,
        "config": {"workload": WORKLOADS["streamed_decode1"], "tokens_per_step": 1,
                   "seed": ctx.seed, "slots": n_slots, "slot_bytes": ctx.stride,
                   "timed_blocks": tm.blocks, "l2": ctx.flush_note()},
        "cache": {"hit_rate": hits / max(hits + misses, 1e-9), "misses_per_step": misses,
                  "h2d_bytes_per_step": copy_bytes},
        "roofline": {"bound": "host link", "achieved": copy_bytes / sec / 1e9, "peak": link,
                     "unit": "GB/s", "frac": copy_bytes / sec / 1e9 / link, "traffic": None,
                     "peak_source": "one 1 GiB copy from pinned host memory, measured here"},
        "gpu_launches": None,
        "clocks": tm.clocks,
    }
    cache.close()
    del host, slots, ws
    torch.cuda.empty_cache()
    return line


def run_ours(args):
    import torch
    ctx = Ctx(args)
    steps = lambda name: args.steps or DEFAULT_STEPS[name]
    if args.workload in ("all", "decode1"):
        line = bench_decode1(ctx, args, steps("decode1"))
        # the other workloads ride along at one GPU only: a scaling run times the headline
        # (and N ranks would each hold their own 126 GB stack and pinned host pool)
        if args.workload == "all" and ctx.world == 1:
            line["workloads"] = {}
            for name in ("decode64_zipf", "decode64_uniform", "prefill4096", "stacked8",
                         "latent_decode1", "streamed_decode1"):
                if name == "latent_decode1":
                    sub = bench_latent(ctx, args, steps(name))
                elif name == "streamed_decode1":
                    sub = bench_streamed(ctx, args, steps(name))
                else:
                    sub = bench_batch(ctx, name, args, steps(name))
                for k in ("metric", "n_gpus", "higher_is_better", "scaling", "vs_baseline",
                          "data", "dtype", "warmup"):
                    sub.pop(k, None)
                line["workloads"][name] = sub
            line["gpu_launches"] += sum(v["gpu_launches"] or 0 for v in line["workloads"].values())
        line["cpu_baseline"] = None
        if ctx.rank == 0 and ctx.world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(ctx.cfg, ctx.seed, 2)
    elif args.workload in ("latent_decode1", "streamed_decode1"):
        line = (bench_latent if args.workload == "latent_decode1" else bench_streamed)(
            ctx, args, steps(args.workload))
        line.update({"metric": METRIC, "n_gpus": ctx.world, "warmup": args.warmup,
                     "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                     "dtype": "f32", "data": "synthetic", "cpu_baseline": None})
    else:
        line = bench_batch(ctx, args.workload, args, steps(args.workload), args.tokens)
        line["cpu_baseline"] = None
    if ctx.rank == 0:
        print(json.dumps(line), flush=True)
    if ctx.dist:
        ctx.dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0,
                    help="timed steps per block (0 = each workload's default)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="all",
                    choices=["all", "decode1", "decode64_zipf", "decode64_uniform",
                             "prefill4096", "stacked8", "latent_decode1", "streamed_decode1"])
    ap.add_argument("--min-seconds", type=float, default=MIN_TIMED_SECONDS,
                    help="least timed work per workload, in blocks of --steps (0: one block, "
                         "for profiler captures)")
    ap.add_argument("--flush", default="write", choices=["write", "read"],
                    help="how L2 is evicted between timed steps")
    ap.add_argument("--tokens", type=int, default=0,
                    help="tokens per step of a batch workload (0 = the workload's own; "
                         "other values only for small profiler captures)")
    ap.add_argument("--experts", type=int, default=896,
                    help="routed experts resident (896 = the workload; fewer only to keep "
                         "profiler captures small)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        if args.steps <= 0:
            args.steps = 3
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
