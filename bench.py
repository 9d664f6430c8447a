#!/usr/bin/env python
"""Benchmark of one MoE layer (DeepSeek-V3 shape) on GB300.

One step = the whole hot path over one batch: router GEMM, top-k, dispatch
(histogram, scan, permute), routed gate/up and down grouped GEMMs, shared
expert, combine -- one ``moe_layer`` call of the C library.  Inputs are
seeded synthetic tensors of the workload's shapes, resident in HBM.

  python bench.py [--gpus N --steps K --warmup W] [--config dsv3_prefill]
  python bench.py --impl reference ...   # the CPU oracle on host cores

With N > 1 (launched by torchrun) every rank runs an independent replica of
the layer on its own GPU (the path has no exchange step on one GPU); the
reported time is the maximum over ranks and the value counts all ranks'
tokens.  Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (DeepSeek-V3 shape)"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 512 << 20


def launches_per_step(cfg, two_streams: bool, fused: bool = False, presplit: bool = False,
                      split: bool = False) -> int:
    """Our kernels per moe_layer call."""
    n = 4  # top-k, count+scan, permute, router GEMM
    if split and cfg.E >= 2:
        n += 2  # the permute and the routed gate/up in two expert halves
    if not fused:
        n += 1  # combine
    if cfg.dtype == "bf16" and not presplit:
        n += 1  # router weight split (unless made once beforehand)
    n += 2  # gate/up and down grouped GEMMs (routed)
    if cfg.shared_I:
        if cfg.dtype == "bf16" and cfg.shared_I == cfg.I and (not two_streams or fused):
            # its tiles ride in the routed launches (fused: its gate/up on the
            # second stream)
            n += 1 if two_streams else 0
        else:
            n += 2  # its own two launches
    return n

# nominal GB300 peaks, quoted beside the measured ones for context
NOMINAL_HBM_GBS = 7900.0
NOMINAL_BF16_TFLOPS = 2250.0

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the routed
# gate/up GEMM per launch, from ncu captures of this kernel source.  Reported
# as null once the kernel source no longer matches the captured one.
TRAFFIC = {"source_sha256": "ef65fc98dbc776913c77b9a236bf365276ff464d7be7536a60a55f25aa034be4",
           # routed gate/up launch on tile-major weights (the shared expert
           # runs on the second stream): dsv3_prefill_e32 from an ncu capture
           # of the 32-expert case (dram__bytes_read.sum 1.951280e9 +
           # dram__bytes_write.sum 0.018274e9); dsv3_prefill is that capture
           # scaled by the units processed (8x the experts at the same rows
           # per expert, 8x the tokens), the workload being too large for a
           # multi-metric capture
           "bytes_per_launch_at_workload": {"dsv3_prefill_e32": 1.969554e9,
                                            "dsv3_prefill": 8 * 1.969554e9}}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return dict(hbm_gbs=j["hbm_gbs"], bf16=j["bf16_tflops"],
                    bf16_sustained=j.get("bf16_tflops_sustained", j["bf16_tflops"]),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


def max_over_ranks(x: float, device="cuda") -> float:
    """The largest x over all ranks (x itself without a process group)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(tokens_per_step: int, steps: int, world: int, seconds: float) -> float:
    """Tokens/s of the whole job: every rank's tokens over the slowest rank's time."""
    return tokens_per_step * steps * world / seconds


def env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index: int):
        self.proc = None
        self.dev = dev_index
        self.lines = []

    def __enter__(self):
        try:
            import torch
            sel = str(self.dev)
            try:
                bus = torch.cuda.get_device_properties(self.dev).pci_bus_id
                if bus:
                    sel = bus
            except Exception:
                pass
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={sel}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is None:
            return False
        time.sleep(0.12)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- oracle leg

def oracle_sample(cfg, inp, n_tok, seed=0):
    """Run the CPU oracle on n_tok sampled tokens; returns (seconds, tokens)."""
    import numpy as np
    import torch

    import oracle
    from combine_router_gemm_gb300 import inputs

    npy = inputs.to_numpy
    g = torch.Generator()
    g.manual_seed(seed)
    tok = torch.randperm(cfg.T, generator=g)[:n_tok].sort().values
    x = npy(inp["x"][tok.to(inp["x"].device)])
    fn = oracle.SIGMOID if cfg.score_fn == "sigmoid" else oracle.SOFTMAX
    w = inp["_host"]
    t0 = time.perf_counter()
    oracle.moe_tokens(x, E=cfg.E, k=cfg.k, w13=w["w13"], w2=w["w2"], w_router=w["w_router"],
                      bias=w["bias"], n_group=cfg.n_group, topk_group=cfg.topk_group,
                      score_fn=fn, routed_scale=cfg.routed_scale, w13_sh=w["w13_sh"],
                      w2_sh=w["w2_sh"], round_h=cfg.dtype == "bf16")
    return time.perf_counter() - t0, n_tok


def host_weights(inp):
    from combine_router_gemm_gb300 import inputs
    npy = inputs.to_numpy
    return {k: npy(inp[k]) for k in ("w13", "w2", "w_router", "bias", "w13_sh", "w2_sh")}


def eager_layer(cfg, inp):
    """The same layer as plain PyTorch GPU ops (a comparator, timed only):
    fp32 router, torch.topk selection, one matmul chain per active expert,
    index_add_ combine."""
    import torch
    import torch.nn.functional as F
    x, T, E, k, I = inp["x"], cfg.T, cfg.E, cfg.k, cfg.I
    logits = x.float() @ inp["w_router"].t()
    if cfg.score_fn == "sigmoid":
        s = torch.sigmoid(logits)
        key = s + inp["bias"] if inp["bias"] is not None else s
    else:
        s = logits
        key = logits
    if cfg.n_group > 1:
        gs = key.view(T, cfg.n_group, E // cfg.n_group).topk(2, dim=-1).values.sum(-1)
        keep = torch.zeros_like(gs, dtype=torch.bool)
        keep.scatter_(1, gs.topk(cfg.topk_group, dim=-1).indices, True)
        key = key.masked_fill(~keep.repeat_interleave(E // cfg.n_group, dim=1), float("-inf"))
    idx = key.topk(k, dim=-1).indices
    if cfg.score_fn == "sigmoid":
        w = s.gather(1, idx)
    else:
        w = torch.softmax(logits, dim=-1).gather(1, idx)
    w = w / w.sum(-1, keepdim=True) * cfg.routed_scale
    flat = idx.reshape(-1)
    order = torch.argsort(flat, stable=True)
    counts = torch.bincount(flat, minlength=E).tolist()
    tok = order // k
    wsel = w.reshape(-1)[order]
    out = torch.zeros((T, cfg.d), dtype=torch.float32, device=x.device)
    start = 0
    for e, n in enumerate(counts):
        if n == 0:
            continue
        rows = tok[start:start + n]
        xe = x[rows]
        gu = xe @ inp["w13"][e].t()
        h = (F.silu(gu[:, :I].float()) * gu[:, I:].float()).to(x.dtype)
        y = (h @ inp["w2"][e].t()).float()
        out.index_add_(0, rows, y * wsel[start:start + n, None])
        start += n
    if inp["w13_sh"] is not None:
        gu = x @ inp["w13_sh"].t()
        Is = cfg.shared_I
        h = (F.silu(gu[:, :Is].float()) * gu[:, Is:].float()).to(x.dtype)
        out += (h @ inp["w2_sh"].t()).float()
    return out


def dispatch_alone_ms(cfg, x, layer, flush, steps=20):
    """moe_dispatch (histogram, scan, permute) timed on its own, on the
    routing of the layer's input (L2 flushed before each call)."""
    import torch
    from combine_router_gemm_gb300 import binding as B
    S = cfg.S
    idx = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device="cuda")
    layer.forward(x, topk_idx_out=idx)
    counts = torch.empty(cfg.E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(cfg.E + 1, dtype=torch.int32, device="cuda")
    s2r = torch.empty(S, dtype=torch.int32, device="cuda")
    r2t = torch.empty(S, dtype=torch.int32, device="cuda")
    xp = torch.empty((S, cfg.d), dtype=x.dtype, device="cuda")
    ws = torch.empty(B.moe_dispatch_workspace_size(cfg.T, cfg.k, cfg.E), dtype=torch.uint8,
                     device="cuda")
    return time_cuda(lambda: B.moe_dispatch(idx, x, cfg.E, counts, offsets, s2r, r2t, xp, ws),
                     steps, flush)


def time_cuda(fn, steps, flush):
    import torch
    fn()
    torch.cuda.synchronize()
    ms = []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    return statistics.median(ms)


def comparators(cfg, inp, ours_out, flush, steps=3):
    """PyTorch comparator on the same inputs: the eager layer.  Reports what
    it measured, or why it could not run.  (A library grouped GEMM,
    torch._grouped_mm of torch 2.9.1, failed with an unspecified launch
    failure on GB300 and is not run.)"""
    import torch
    res = {}
    if cfg.dtype != "bf16":
        return res
    try:
        ms = time_cuda(lambda: eager_layer(cfg, inp), steps, flush)
        ref = eager_layer(cfg, inp)
        rel = float(torch.linalg.norm(ref - ours_out) / torch.linalg.norm(ref))
        res["torch_eager_layer"] = {"ms": round(ms, 3), "tokens_per_s": round(cfg.T / ms * 1e3, 1),
                                    "rel_fro_vs_ours": rel}
    except Exception as exc:  # a comparator that cannot run is reported, not fatal
        res["torch_eager_layer"] = {"unavailable": f"{type(exc).__name__}: {exc}"[:200]}
    return res


def cpu_baseline(cfg, inp, target_s=15.0):
    import oracle
    inp["_host"] = inp.get("_host") or host_weights(inp)
    probe = 16
    dt, _ = oracle_sample(cfg, inp, probe, seed=1)
    n = int(max(probe, min(cfg.T, probe * target_s / max(dt, 1e-3))))
    dt, n = oracle_sample(cfg, inp, n, seed=2)
    return {"value": n / dt, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} of {cfg.T} tokens of {cfg.name}, whole layer per token "
                      f"(router, top-{cfg.k}, experts, shared expert), {dt:.1f} s"}


def run_reference(args, cfg):
    rank, local_rank, world = env_rank()
    if rank != 0:
        return 0
    import torch

    import oracle
    from combine_router_gemm_gb300 import inputs
    oracle.build()
    dev = f"cuda:{local_rank}" if torch.cuda.is_available() else "cpu"
    inp = inputs.make_inputs(cfg, seed=0, device=dev)
    inp["_host"] = host_weights(inp)
    # size one step's token sample so the whole run stays within a few minutes
    dt, _ = oracle_sample(cfg, inp, 8, seed=99)
    per_tok = dt / 8
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = max(1, min(cfg.T, int(budget / max(per_tok, 1e-6))))
    for w in range(args.warmup):
        oracle_sample(cfg, inp, n, seed=1000 + w)
    total = 0.0
    for s in range(args.steps):
        dt, _ = oracle_sample(cfg, inp, n, seed=s)
        total += dt
    value = n * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(cfg, flushed=False),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"{n} of {cfg.T} tokens per step of {cfg.name}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm

def config_dict(cfg, flushed=True):
    return {"workload": cfg.name, "T": cfg.T, "d": cfg.d, "E": cfg.E, "k": cfg.k, "I": cfg.I,
            "shared_I": cfg.shared_I, "routing": f"{cfg.score_fn}, {cfg.n_group} groups keep "
            f"{cfg.topk_group}, scale {cfg.routed_scale}, bias {cfg.bias}",
            "global_batch": cfg.T,
            "l2": ("flushed between steps (512 MB write)" if flushed else "n/a (host)"),
            "parallelism": "replicas (one independent layer per GPU)"}


def kernel_source_sha():
    p = os.path.join(ROOT, "combine_router_gemm_gb300", "csrc", "grouped_gemm_tc.cu")
    return hashlib.sha256(open(p, "rb").read()).hexdigest()


def stage_metrics(cfg, stage_ms, offs, merged, merged_gu, pk):
    """Per-stage algorithmic bytes and flops, rates and roofline fractions,
    and the roofline object of the dominant kernel (the routed gate/up)."""
    o = offs.cpu().numpy()
    active = int((o[1:] - o[:-1] > 0).sum())
    S, d, I, T = cfg.S, cfg.d, cfg.I, cfg.T
    es = 2 if cfg.dtype == "bf16" else 4
    gu_bytes = active * 2 * I * d * es + S * d * es + S * I * es
    gu_flops = 2.0 * S * d * 2 * I
    dn_bytes = active * d * I * es + S * I * es + S * d * 4
    dn_flops = 2.0 * S * I * d
    Is = cfg.shared_I
    if merged_gu:
        gu_bytes += 2 * Is * d * es + T * d * es + T * Is * es
        gu_flops += 2.0 * T * d * 2 * Is
    if merged:
        dn_bytes += d * Is * es + T * Is * es + T * d * 4
        dn_flops += 2.0 * T * Is * d
    perm_bytes = T * d * es + S * d * es + S * 4 * 3 + S * 4
    # stage 1 covers the router GEMM and top-k (top-k sums the router's
    # partial logits), stage 2 is empty
    names = ["route", "route_", "dispatch", "gate_up_gemm", "down_gemm", "combine"]
    stages = {n: {"ms": round(m, 4)} for n, m in zip(names, stage_ms) if n != "route_"}

    def bw(b, ms):
        return b / (ms * 1e-3) / 1e9

    def tf(f, ms):
        return f / (ms * 1e-3) / 1e12

    stages["dispatch"].update(GBps=round(bw(perm_bytes, stage_ms[2]), 1),
                              frac_hbm=round(bw(perm_bytes, stage_ms[2]) / pk["hbm_gbs"], 4),
                              note="count + permute, beside the shared expert's GEMMs")
    for key, b, f, ms in (("gate_up_gemm", gu_bytes, gu_flops, stage_ms[3]),
                          ("down_gemm", dn_bytes, dn_flops, stage_ms[4])):
        stages[key].update(GBps=round(bw(b, ms), 1), TFLOPs=round(tf(f, ms), 1),
                           frac_hbm=round(bw(b, ms) / pk["hbm_gbs"], 4),
                           frac_bf16=round(tf(f, ms) / pk["bf16_sustained"], 4))
    ridge = pk["bf16_sustained"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    ai = gu_flops / gu_bytes
    ms = stage_ms[3]
    traffic = None
    if TRAFFIC["source_sha256"] == kernel_source_sha():
        traffic = TRAFFIC["bytes_per_launch_at_workload"].get(cfg.name)
    if ai < ridge:
        roof = {"bound": "hbm", "achieved": round(bw(gu_bytes, ms), 1), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(bw(gu_bytes, ms) / pk["hbm_gbs"], 4)}
    else:
        roof = {"bound": "tensor", "achieved": round(tf(gu_flops, ms), 1),
                "peak": pk["bf16_sustained"], "unit": "TFLOP/s",
                "frac": round(tf(gu_flops, ms) / pk["bf16_sustained"], 4)}
    roof.update(traffic=traffic,
                kernel="grouped_gemm_tc gate/up+SwiGLU (routed" + (" + shared)" if merged_gu else ")"),
                algorithmic_bytes=gu_bytes, algorithmic_flops=gu_flops,
                arithmetic_intensity=round(ai, 1), peak_source=pk["source"],
                launch_ms=round(ms, 4))
    # context: the same achieved figure against the nominal GB300 peaks
    # (HBM3e 7.9 TB/s, dense bf16 2.25 PFLOP/s)
    nominal = NOMINAL_HBM_GBS if roof["bound"] == "hbm" else NOMINAL_BF16_TFLOPS
    roof.update(nominal_peak=nominal, frac_of_nominal=round(roof["achieved"] / nominal, 4))
    return stages, roof, active, perm_bytes


def measure_layer(cfg, args, layer, x, flush, pk, K, warm, clk_dev, world, graph_too):
    """Warm-up, then K stream-launched layer calls (L2 flushed before each,
    stage events recorded, clocks sampled), optionally K graph replays of the
    same call in the same clock-sampled region.  Returns the measured figures."""
    import torch
    import torch.distributed as dist
    from combine_router_gemm_gb300 import binding as B

    out = torch.empty((cfg.T, cfg.d), dtype=torch.float32, device="cuda")
    offs = torch.empty(cfg.E + 1, dtype=torch.int32, device="cuda")
    for _ in range(warm):
        layer.forward(x, out=out, offsets_out=offs)
    rc, detail = B.moe_check_error(layer.ws)
    if rc != B.OK:
        raise RuntimeError(f"device error word {detail:#x} during warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(B.LAYER_EVENTS)] for _ in range(K)]
    graph = None
    if graph_too:
        graph, gout = layer.capture(x, offsets_out=offs)
        for _ in range(warm):
            graph.replay()
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    with ClockSampler(clk_dev) as clk:
        # pass 1 (the reported value): stream-launched calls with stage events
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        for s in range(K):
            flush.zero_()
            layer.forward(x, out=out, offsets_out=offs, stage_events=evs[s])
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        if world > 1:
            dist.barrier()
        # pass 2: graph replays of the same call (inputs resident, L2 flushed
        # between steps)
        if graph is not None:
            torch.cuda.synchronize()
            for s in range(K):
                flush.zero_()
                gev[s][0].record()
                graph.replay()
                gev[s][1].record()
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
    rc, detail = B.moe_check_error(layer.ws)
    if rc != B.OK:
        raise RuntimeError(f"device error word {detail:#x} during the timed steps")
    step_ms = [e[0].elapsed_time(e[-1]) for e in evs]
    stage_ms = [statistics.fmean(e[i].elapsed_time(e[i + 1]) for e in evs)
                for i in range(B.LAYER_EVENTS - 1)]
    total_s = max_over_ranks(sum(step_ms) / 1e3)
    res = {"value": whole_job_value(cfg.T, K, world, total_s), "ms_per_step": 1e3 * total_s / K,
           "steps": K, "warmup": warm, "clocks": clk.summary(), "wall_s_timed": round(t_wall, 3)}
    if graph is not None:
        g_s = max_over_ranks(sum(a.elapsed_time(b) for a, b in gev) / 1e3)
        res["graph_replay"] = {"value": whole_job_value(cfg.T, K, world, g_s), "unit": UNIT,
                               "ms_per_step": 1e3 * g_s / K}
        del graph, gout
    # bf16, I_sh == I: with a second stream the shared expert runs there in
    # launches of its own (with the fused combine, only its gate/up; its down
    # tiles ride in the routed down launch); without one, both halves ride
    # in the routed launches
    two_streams = layer.stream2 is not None
    merged = (bool(cfg.shared_I) and cfg.dtype == "bf16" and cfg.shared_I == cfg.I
              and (not two_streams or args.fused_combine))
    stages, roof, active, perm_bytes = stage_metrics(cfg, stage_ms, offs, merged,
                                                     merged and not two_streams, pk)
    # the dispatch (count + permute) alone, on this step's routing
    d_ms = dispatch_alone_ms(cfg, x, layer, flush, steps=min(K, 20))
    gbs = perm_bytes / (d_ms * 1e-3) / 1e9
    stages["dispatch_alone"] = {"ms": round(d_ms, 4), "GBps": round(gbs, 1),
                                "frac_hbm": round(gbs / pk["hbm_gbs"], 4)}
    res.update(stages=stages, roofline=roof, active_experts=active, two_streams=two_streams)
    return res


def make_layer(cfg, args, inp):
    from combine_router_gemm_gb300 import binding as B
    return B.MoELayer(inp["w_router"], inp["bias"], inp["w13"], inp["w2"], inp["w13_sh"],
                      inp["w2_sh"], B.cfg_from(cfg), cfg.T, overlap=not args.no_overlap,
                      fused_combine=args.fused_combine, pack_weights=not args.row_major_weights,
                      split_dispatch=getattr(args, "split_dispatch", False))


# the other workloads timed beside the headline one (N = 1), each with the
# same protocol but fewer steps and without the host-side legs
EXTRA_WORKLOADS = ("mixtral_bf16", "dsv3_decode", "dsv3_zipf")


def extra_workloads(args, pk, flush, names):
    """Each named workload built, timed and freed in turn."""
    import gc

    import torch
    from combine_router_gemm_gb300 import inputs
    res = {}
    for name in names:
        cfg = inputs.CONFIGS[name]
        inp = inputs.make_inputs(cfg, seed=0, device="cuda")
        layer = make_layer(cfg, args, inp)
        x = inp["x"]
        for k in ("w13", "w2", "w13_sh", "w2_sh"):  # the layer holds its own copies
            if layer.packed:
                inp[k] = None
        m = measure_layer(cfg, args, layer, x, flush, pk, min(args.steps, 30), 3, 0, 1, False)
        m["config"] = config_dict(cfg)
        m["dtype"] = cfg.dtype
        res[name] = m
        del layer, inp, x
        gc.collect()
        torch.cuda.empty_cache()
    return res


def run_ours(args, cfg):
    import gc

    import torch
    import torch.distributed as dist

    rank, local_rank, world = env_rank()
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    from combine_router_gemm_gb300 import binding as B
    from combine_router_gemm_gb300 import build as build_mod
    from combine_router_gemm_gb300 import inputs
    build_mod.build()

    pk = peaks()
    inp = inputs.make_inputs(cfg, seed=0, device="cuda")
    layer = make_layer(cfg, args, inp)
    x = inp["x"]
    host_legs = rank == 0 and world == 1 and not (args.no_cpu_baseline and args.no_comparators)
    if layer.packed and not host_legs:
        # the layer holds the packed copies; the row-major originals are only
        # needed by the comparator and the CPU oracle legs
        for k in ("w13", "w2", "w13_sh", "w2_sh"):
            inp[k] = None
        gc.collect()
        torch.cuda.empty_cache()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    K = args.steps
    warm = max(3, args.warmup)
    m = measure_layer(cfg, args, layer, x, flush, pk, K, warm, local_rank, world,
                      graph_too=not args.no_graph)
    presplit = layer.w_router_split is not None
    T, d = cfg.T, cfg.d

    # ---- end to end through the public API with host buffers: every step
    # copies its input from pinned host memory and its output back; copies of
    # neighbouring steps overlap the compute (MoELayer.forward_host)
    e2e = None
    if not args.no_e2e:
        ne = args.e2e_steps
        xh = [torch.empty((T, d), dtype=x.dtype, pin_memory=True) for _ in range(2)]
        for h in xh:
            h.copy_(x)
        oh = [torch.empty((T, d), dtype=torch.float32, pin_memory=True) for _ in range(2)]
        ins = [xh[i % 2] for i in range(ne)]
        outs = [oh[i % 2] for i in range(ne)]
        layer.forward_host(ins[:3], outs[:3])  # warm-up
        torch.cuda.synchronize()
        ev0, ev1 = layer.forward_host(ins, outs)
        torch.cuda.synchronize()
        e_s = max_over_ranks(ev0.elapsed_time(ev1) / 1e3)
        e2e = {"value": whole_job_value(T, ne, world, e_s), "unit": UNIT,
               "h2d_bytes_per_step": T * d * x.element_size(),
               "d2h_bytes_per_step": T * d * 4, "steps": ne,
               "pipelined": "H2D of step i+1 and D2H of step i-1 overlap step i"}

    comp = None
    if rank == 0 and world == 1 and not args.no_comparators:
        out = layer.forward(x)
        torch.cuda.synchronize()
        comp = comparators(cfg, inp, out, flush)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, inp)

    extras = None
    if world == 1 and not args.no_workloads:
        names = [n for n in EXTRA_WORKLOADS if n != cfg.name]
        del layer, inp, x
        gc.collect()
        torch.cuda.empty_cache()
        extras = extra_workloads(args, pk, flush, names)

    if rank == 0:
        launches = launches_per_step(cfg, m["two_streams"], args.fused_combine, presplit,
                                     args.split_dispatch) * K
        line = {
            "metric": METRIC, "value": m["value"], "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": warm, "ms_per_step": m["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
            "config": config_dict(cfg),
            "expert_weights": ("tile-major, packed once at layer construction"
                               if not args.row_major_weights else "row-major"),
            "dispatch": ("permute of the upper expert half on a second stream beside the "
                         "lower half's gate/up" if args.split_dispatch else "one pass"),
            "roofline": m["roofline"], "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches, "clocks": m["clocks"], "stages": m["stages"],
            "active_experts": m["active_experts"], "wall_s_timed": m["wall_s_timed"],
        }
        if "graph_replay" in m:
            line["graph_replay"] = m["graph_replay"]
        if comp:
            line["comparators"] = comp
        if extras:
            line["workloads"] = extras
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="dsv3_prefill")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timing")
    ap.add_argument("--no-comparators", action="store_true",
                    help="skip the PyTorch comparator (the eager layer)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip timing the other workloads beside the headline one (N = 1)")
    ap.add_argument("--no-overlap", action="store_true", help="shared expert on the main stream")
    ap.add_argument("--row-major-weights", action="store_true",
                    help="keep the expert weights row-major (no tile-major packing)")
    ap.add_argument("--fused-combine", action="store_true",
                    help="add the down projection's results straight into the output (atomics)")
    ap.add_argument("--split-dispatch", action="store_true",
                    help="permute the upper half of the experts on a second stream beside the "
                         "lower half's gate/up")
    args = ap.parse_args()
    from combine_router_gemm_gb300 import inputs
    cfg = inputs.CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
