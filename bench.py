"""Benchmark of the MoE layer step on GB300.

Workload (one step = one pass of the whole layer step over one batch):
  decode1: one decode token through one full-shape layer -- hidden 7168, expert
  intermediate 1536, 896 routed MXFP4 experts resident in HBM (15.7 GB), top-16, one bf16
  shared expert 7168x1536.  Synthetic seeded inputs (synth/), distinct tokens per step so
  every step routes to its own experts; L2 is flushed (a 256 MB write) between timed steps.

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead (the reference
arm of this comparison), on the same workload, metric and unit.

N > 1 (torchrun): the layer step does not shard without an exchange step, so every rank
runs an independent replica; value = tokens processed by all ranks / max rank time.
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
sys.path.insert(0, ROOT)

METRIC = "MoE-layer decode tokens/s & HBM GB/s vs ~8 TB/s; prefill tcgen05 % peak"
WORKLOAD = ("decode1: 1 token/step through one full-shape MoE layer (hidden 7168, inter 1536, "
            "896 MXFP4 experts top-16, 1 bf16 shared expert 7168x1536)")


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu
# capture of each decode kernel, keyed to a hash of the sources the kernels are built
# from: a changed kernel reports null until it is captured again.
TRAFFIC_SOURCES = ["mxfp4_routed_expert_02_gb300/csrc/k3moe_decode_fused.cu",
                   "mxfp4_routed_expert_02_gb300/csrc/k3moe_decode.cu",
                   "mxfp4_routed_expert_02_gb300/csrc/k3moe_router.cu",
                   "mxfp4_routed_expert_02_gb300/csrc/k3moe_device.cuh",
                   "mxfp4_routed_expert_02_gb300/csrc/k3moe_topk.cuh",
                   "mxfp4_routed_expert_02_gb300/csrc/k3moe_kernels.cuh"]
# k_decode_fused: captured with a 64-expert pool (351,598,080 B per launch), plus the
# router rows the full 896-expert pool adds ((896 - 64) x 7168 x 2 B): every other byte
# the kernel reads is the same at both pool sizes (16 selected experts, the shared expert).
TRAFFIC_CAPTURED = {"sources": "dacd8f370a02f450",
                    "bytes": {"k_decode_fused": 351598080 + (896 - 64) * 7168 * 2}}


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
        "k_down_combine": down, "k_down_tma": down,
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


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import synth
    import synth.device as sd
    import mxfp4_routed_expert_02_gb300 as k3

    cfg = synth.config("decode1")
    if args.experts != cfg.n_experts:   # smaller expert pool: profiling captures only
        cfg = synth.config("decode1", n_experts=args.experts)
    seed = 0
    dev = torch.device("cuda", local)
    H, I, E, K = cfg.hidden, cfg.inter, cfg.n_experts, cfg.topk
    dims = k3.LayerDims(H, I, E, K, cfg.shared_inter)
    stride = (cfg.record_bytes + 4095) // 4096 * 4096
    experts = torch.empty(E * stride, dtype=torch.uint8, device=dev)
    sd.fill_experts(experts, cfg, seed, 0, stride=stride)
    w = synth.layer_weights(cfg, seed)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    wr, bias = t(w["wr"].view(np.int16)), t(w["bias"])
    sg, su, sdn = (t(w[k].view(np.int16)) for k in ("sh_gate", "sh_up", "sh_down"))
    NX = 256
    xs_host = synth.activations(cfg, seed + 1 + rank, NX)
    xs = t(xs_host.view(np.int16))
    y = torch.empty((1, H), dtype=torch.float32, device=dev)
    idx = torch.empty((NX, K), dtype=torch.int32, device=dev)
    wt = torch.empty((NX, K), dtype=torch.float32, device=dev)
    ws = k3.new_workspace(dims, 1, dev)
    status = k3.new_status(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(s):
        j = s % NX
        k3.k3moe_layer(dims, xs[j:j + 1], wr, bias, experts, stride, sg, su, sdn, y, ws, status,
                       idx_out=idx[j:j + 1], w_out=wt[j:j + 1])

    for s in range(args.warmup):
        flush.fill_(s & 255)
        step(s)
    torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = Clocks("/tmp/k3moe_bench_clocks_%d_%d.csv" % (os.getpid(), rank))
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with clocks:
        t_wall = time.perf_counter()
        for s in range(args.steps):
            flush.fill_((s + 7) & 255)
            ev[s][0].record(stream)
            step(args.warmup + s)
            ev[s][1].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    assert status.item() == 0, k3.status_str(status.item())
    ms = [a.elapsed_time(b) for a, b in ev]
    t_dev = reduce_max(dist, sum(ms) / 1e3, dev)

    # per-kernel device time: the same steps again with the library's event tracing on
    # (tracing brackets every launch with events, so it also turns off the programmatic
    # overlap of consecutive kernels; the step time above is taken without it)
    k3.k3moe_trace_enable(True)
    for s in range(args.steps):
        flush.fill_((s + 7) & 255)
        step(args.warmup + s)
    torch.cuda.synchronize()
    trace = k3.k3moe_trace_read()
    k3.k3moe_trace_enable(False)

    # distinct experts actually used per step (for the algorithmic bytes)
    steps_idx = idx.cpu().numpy()
    used = [len(set(steps_idx[(args.warmup + s) % NX].tolist())) for s in range(args.steps)]
    U = statistics.mean(used)
    nb = step_bytes(cfg, U)
    bytes_step = nb["k_decode_fused"]
    launches = sum(v[1] for v in trace.values())
    kernels = {k: {"ms_avg": v[0] / v[1], "launches": v[1]} for k, v in trace.items() if v[1]}
    # the dominant kernel: most device time among the kernels that stream the weights
    dom = max((k for k in kernels if k in nb),
              key=lambda k: kernels[k]["ms_avg"] * kernels[k]["launches"])
    pk = peaks()
    peak_hbm = pk["hbm_gbs"] if pk else 6800.0
    dom_ms = kernels[dom]["ms_avg"]
    achieved = nb[dom] / (dom_ms * 1e-3) / 1e9
    for k in kernels:
        if k in nb:
            kernels[k]["gbs"] = nb[k] / (kernels[k]["ms_avg"] * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak_hbm, "unit": "GB/s",
                "frac": achieved / peak_hbm, "traffic": traffic_of(dom), "kernel": dom,
                "algorithmic_bytes": nb[dom],
                "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if pk else
                               "fallback 6.8 TB/s (of fallback)"}

    # end to end through the C ABI with host buffers: x in from pinned host memory,
    # y back to pinned host memory, every step
    xh = torch.from_numpy(xs_host.view(np.int16).copy()).pin_memory()
    yh = torch.empty((1, H), dtype=torch.float32).pin_memory()
    xd = torch.empty((1, H), dtype=torch.int16, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for s in range(args.steps):
        j = s % NX
        xd.copy_(xh[j:j + 1], non_blocking=True)
        k3.k3moe_layer(dims, xd, wr, bias, experts, stride, sg, su, sdn, y, ws, status)
        yh.copy_(y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    t_e2e = reduce_max(dist, e0.elapsed_time(e1) / 1e3, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, seed, 2)
    if rank == 0:
        line = {
            "metric": METRIC, "value": job_rate(args.steps, world, t_dev), "unit": "tokens/s",
            "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_dev / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "tokens_per_step": 1, "seed": seed,
                       "l2": "flushed between timed steps (256 MB write, outside the step "
                             "events)", "distinct_experts_per_step": U,
                       "parallelism": "replicas" if world > 1 else "single"},
            "hbm_gbs_step": bytes_step / (t_dev / args.steps) / 1e9,
            "algorithmic_bytes_per_step": bytes_step,
            "roofline": roofline,
            "kernels": kernels,
            "gpu_launches": launches,
            "clocks": clocks.summary(local),
            "e2e": {"value": job_rate(args.steps, world, t_e2e), "unit": "tokens/s",
                    "h2d_bytes_per_step": H * 2,
                    "d2h_bytes_per_step": H * 4},
            "cpu_baseline": cpu,
            "wall_s": t_wall,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


BATCH_WORKLOADS = {
    "decode64_zipf": "decode64_zipf: 64 tokens/step through one full-shape MoE layer, expert "
                     "popularity Zipf(1.1) through the correction bias",
    "prefill4096": "prefill4096: 4096 tokens/step through one full-shape MoE layer, uniform "
                   "routing (grouped MXFP4 GEMM on tcgen05)",
    "stacked8": "stacked8: 1 token/step through 8 stacked full-shape MoE layers (126 GB of "
                "MXFP4 resident) with RMSNorm and the residual stream between them",
}


def useful_flops(cfg, P, T):
    """Multiply-adds x 2 of the expert GEMMs for P (token, slot) pairs and T tokens."""
    H, I, SI = cfg.hidden, cfg.inter, cfg.shared_inter
    return 2.0 * P * 3 * H * I + 2.0 * T * 3 * H * SI


def run_batch(args):
    """The multi-token and stacked workloads (one JSON line each, same contract)."""
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import synth
    import synth.device as sd
    import mxfp4_routed_expert_02_gb300 as k3

    name = args.workload
    cfg = synth.config("decode1" if name == "stacked8" else name)
    if args.experts != cfg.n_experts:   # smaller expert pool: profiling captures only
        cfg = synth.config(cfg.name, n_experts=args.experts)
    L = 8 if name == "stacked8" else 1
    T = 1 if name == "stacked8" else (args.tokens or cfg.tokens)
    seed = 0
    dev = torch.device("cuda", local)
    H, I, E, K = cfg.hidden, cfg.inter, cfg.n_experts, cfg.topk
    dims = k3.LayerDims(H, I, E, K, cfg.shared_inter)
    stride = (cfg.record_bytes + 4095) // 4096 * 4096
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    layers = []
    for l in range(L):
        ex = torch.empty(E * stride, dtype=torch.uint8, device=dev)
        sd.fill_experts(ex, cfg, seed, l, stride=stride)
        w = synth.layer_weights(cfg, seed, l)
        layers.append(dict(wr=t(w["wr"].view(np.int16)), bias=t(w["bias"]), experts=ex,
                           stride=stride, sh_gate=t(w["sh_gate"].view(np.int16)),
                           sh_up=t(w["sh_up"].view(np.int16)),
                           sh_down=t(w["sh_down"].view(np.int16))))
    ws = k3.new_workspace(dims, T, dev)
    status = k3.new_status(dev)
    NX = 4
    xs_host = [synth.activations(cfg, seed + 1 + rank * NX + j, T) for j in range(NX)]
    xs = [t(a.view(np.int16)) for a in xs_host]
    y = torch.empty((T, H), dtype=torch.float32, device=dev)
    idx = torch.empty((L, T, K), dtype=torch.int32, device=dev)
    wts = torch.empty((L, T, K), dtype=torch.float32, device=dev)
    h = torch.empty((T, H), dtype=torch.float32, device=dev)
    h.copy_(torch.from_numpy((xs_host[0].astype(np.uint32) << 16).view(np.float32)).to(dev))
    xsc = torch.empty((T, H), dtype=torch.int16, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    lw = layers[0]

    def step(s):
        if name == "stacked8":
            k3.k3moe_decode_stack(dims, layers, h, xsc, ws, status, eps=cfg.rms_eps,
                                  idx_out=idx, w_out=wts)
        else:
            k3.k3moe_layer(dims, xs[s % NX], lw["wr"], lw["bias"], lw["experts"], stride,
                           lw["sh_gate"], lw["sh_up"], lw["sh_down"], y, ws, status,
                           idx_out=idx[0], w_out=wts[0])

    for s in range(args.warmup):
        if name != "stacked8":
            flush.fill_(s & 255)
        step(s)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = Clocks("/tmp/k3moe_bench_clocks_%d_%d.csv" % (os.getpid(), rank))
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with clocks:
        for s in range(args.steps):
            if name != "stacked8":
                flush.fill_((s + 7) & 255)
            ev[s][0].record(stream)
            step(args.warmup + s)
            ev[s][1].record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    assert status.item() == 0, k3.status_str(status.item())
    ms = [a.elapsed_time(b) for a, b in ev]
    t_dev = reduce_max(dist, sum(ms) / 1e3, torch.device("cuda", local))
    # per-kernel device time from a traced pass
    k3.k3moe_trace_enable(True)
    for s in range(min(args.steps, 3)):
        step(args.warmup + s)
    torch.cuda.synchronize()
    trace = k3.k3moe_trace_read()
    k3.k3moe_trace_enable(False)
    nsteps_tr = min(args.steps, 3)
    kernels = {k: {"ms_avg": v[0] / v[1], "launches_per_step": v[1] / nsteps_tr}
               for k, v in trace.items() if v[1]}
    launches = int(sum(v[1] for v in trace.values()) / nsteps_tr * args.steps)
    # distinct experts of the last step, per layer
    ids = idx.cpu().numpy()
    U = [len(set(ids[l].ravel().tolist())) for l in range(L)]
    op = I * H // 2 + I * H // 32
    layer_bytes = [u * 3 * op + E * H * 2 + 3 * cfg.shared_inter * H * 2 + T * H * 6 for u in U]
    step_bytes_v = sum(layer_bytes)
    pk = peaks()
    peak_hbm = pk["hbm_gbs"] if pk else 6800.0
    peak_bf16 = pk["bf16_tflops"] if pk else 1900.0
    sec = t_dev / args.steps
    if name == "prefill4096":
        P = T * K
        fl = useful_flops(cfg, P, T)
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
        extra = {"useful_tflops_step": fl / sec / 1e12,
                 "down_kernel_tflops": 2.0 * P * H * I / (dk * 1e-3) / 1e12 if dk else None}
    else:
        if name == "decode64_zipf":
            dom = "k_tc_gemm_gateup"
            db = sum(u * 2 * op for u in U) / L        # gate/up bytes of the distinct experts
        else:
            dom = "k_decode_fused"                      # one kernel per layer: all its bytes
            db = sum(layer_bytes) / L
        dk = kernels.get(dom, {}).get("ms_avg")
        roofline = {"bound": "hbm", "kernel": dom,
                    "achieved": db / (dk * 1e-3) / 1e9 if dk else None, "peak": peak_hbm,
                    "unit": "GB/s", "frac": db / (dk * 1e-3) / 1e9 / peak_hbm if dk else None,
                    "traffic": None, "algorithmic_bytes": db,
                    "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if pk else
                                   "fallback 6.8 TB/s (of fallback)"}
        extra = {}
    lat = sorted(ms)
    line = {
        "metric": METRIC, "value": job_rate(T * args.steps, world, t_dev), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sec, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": BATCH_WORKLOADS[name], "tokens_per_step": T, "layers": L,
                   "seed": seed, "distinct_experts_per_layer": U,
                   "l2": ("inputs larger than L2 (2.9 GB of weights per step)" if L > 1 else
                          "flushed between timed steps (256 MB write)")},
        "hbm_gbs_step": step_bytes_v / sec / 1e9,
        "algorithmic_bytes_per_step": step_bytes_v,
        "latency_ms": {"p50": lat[len(lat) // 2], "p99": lat[min(len(lat) - 1, int(len(lat) * 0.99))]},
        "roofline": roofline, "kernels": kernels, "gpu_launches": launches,
        "clocks": clocks.summary(local), "cpu_baseline": None,
    }
    line.update(extra)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0,
                    help="timed steps (0 = the workload's default: long enough for the "
                         "200 ms clock sampler to see the timed region)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="decode1",
                    choices=["decode1", "decode64_zipf", "prefill4096", "stacked8"])
    ap.add_argument("--tokens", type=int, default=0,
                    help="tokens per step of a batch workload (0 = the workload's own; "
                         "other values only for small profiler captures)")
    ap.add_argument("--experts", type=int, default=896,
                    help="routed experts resident (896 = the workload; fewer only to keep "
                         "profiler captures small)")
    args = ap.parse_args()
    if args.steps <= 0:
        args.steps = {"decode1": 3000, "decode64_zipf": 200, "prefill4096": 40,
                      "stacked8": 256}[args.workload]
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload != "decode1":
        run_batch(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
