#!/usr/bin/env python
"""Throughput of the fused NVFP4 MoE layer on GB300.

Workload (default "decode"): H=2048, E=128 experts, top-8, I=768, SwiGLU, x ~ N(0,1) BF16, router
logits ~ N(0,1) ("uniform routing"), weights ~ N(0,0.02) NVFP4-quantised; the layer is run at
T in {1, 8, 32, 64} tokens.  One step = one layer call (moe_run) at T = (1, 8, 32, 64)[step % 4];
the L2 cache is flushed (a write of 2x its size) before every call, outside the timed events, so
each call reads its weights from HBM as a layer of a real model does.  Inputs are resident in
HBM before the timed region.  Metric: tokens/s (+ effective TFLOPS and %% of HBM bandwidth).

Multi-GPU (torchrun): the layer does not shard across GPUs here, so each rank runs an
independent replica on its own GPU (weak scaling); timing is the max over ranks.

--impl reference times the CPU oracle (the plain single-threaded C++ implementation the tests
check against) on the host cores, on a bounded token sample of every step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "NVFP4 MoE tokens/s & eff. TFLOPS; % of HBM BW (decode) / FP4 peak (prefill)"
UNIT = "tokens/s"
FP4_PER_BF16 = 6.0     # nominal dense FP4 / BF16 tensor rate of the part (13.5 / 2.25 PFLOP/s)
# Layer variants: "base" = softmax router + SwiGLU; "sqrtsoftplus_clamp" = sqrt(softplus) router
# with a seeded per-expert selection bias (N(0, 0.3)) + SwiGLU clamped at L = 10.
VARIANTS = {"base": dict(router="softmax", swiglu_limit=None),
            "sqrtsoftplus_clamp": dict(router="sqrtsoftplus", swiglu_limit=10.0)}


def sharing_level(args):
    if not args.routing:
        return None
    if not args.routing.startswith("shared_") or not args.routing[7:].isdigit():
        raise SystemExit(f"--routing wants shared_<percent>, got {args.routing!r}")
    return int(args.routing[7:])


def gen_router_logits(args, cs, T, i, dev):
    import synth
    share = sharing_level(args)
    if share is None:
        return synth.gen_logits(cs, T, device=dev, row0=1000 * i)
    return synth.gen_sharing_logits(cs, T, share, device=dev)


def variant_bias(cs, variant):
    import numpy as np
    if VARIANTS[variant]["router"] != "sqrtsoftplus":
        return None
    return (np.random.default_rng(1000 + cs.config_id).standard_normal(cs.experts) * 0.3
            ).astype(np.float32)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "tiny", "prefill", "large", "skewed"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", default=None,
                    help="comma-separated batch sizes replacing the workload's own list")
    ap.add_argument("--variant", default="base", choices=list(VARIANTS),
                    help="router / activation variant of the layer")
    ap.add_argument("--producer", action="store_true",
                    help="time the RMSNorm + NVFP4 producer of the layer's input instead of the layer")
    ap.add_argument("--routing", default=None,
                    help="shared_<p> (p in 0..100): the expert-sharing decode workload, whose "
                         "batches reuse p%% of their token/expert assignments")
    ap.add_argument("--ref-budget-s", type=float, default=150.0,
                    help="wall-time budget of the reference arm's timed + warm-up steps")
    ap.add_argument("--workloads", default="tiny,prefill,large,skewed",
                    help="comma-separated configurations measured after the headline workload "
                         "(each one its own sub-record); 'none' skips them")
    return ap.parse_args()


# ----------------------------------------------------------------------------------------- peaks
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


def measured_traffic(key):
    """DRAM bytes per launch from the committed ncu summary, only while the kernel sources
    still hash to what was profiled (null once the kernel has changed)."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        entry = json.load(f).get(key)
    if not entry:
        return None
    for rel, sha in entry["sources"].items():
        with open(os.path.join(ROOT, rel), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != sha:
                return None
    return entry["dram_bytes_per_launch"]


# ----------------------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks / throttle reasons, sampled while the GPU is under load."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0=None, t1=None):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if t0 is not None and not (t0 <= ts <= t1):
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_activity(index: int):
    """Utilisation, memory in use and compute processes of the GPU (nvidia-smi), to show that
    nothing else ran on it around the measurement."""
    out = {}
    try:
        q = subprocess.run(["nvidia-smi", f"--id={index}",
                            "--query-gpu=utilization.gpu,memory.used,clocks.sm",
                            "--format=csv,noheader,nounits"], capture_output=True, text=True,
                           timeout=20)
        u, m, c = [v.strip() for v in q.stdout.strip().split(",")[:3]]
        out = {"util_pct": float(u), "mem_used_mib": float(m), "sm_mhz": float(c)}
        q = subprocess.run(["nvidia-smi", f"--id={index}", "--query-compute-apps=pid",
                            "--format=csv,noheader"], capture_output=True, text=True, timeout=20)
        pids = [int(v) for v in q.stdout.split() if v.strip().isdigit()]
        out["other_processes"] = len([p for p in pids if p != os.getpid()])
    except (OSError, ValueError, subprocess.TimeoutExpired):
        pass
    return out


# ----------------------------------------------------------------------------------------- helpers
def workload(name, tokens=None):
    import synth
    cs = synth.CONFIGS[name]
    Ts = [int(t) for t in tokens.split(",")] if tokens else list(cs.tokens)
    return cs, Ts


def expert_bytes(cs):
    """NVFP4 bytes of one expert: codes (1/2 byte) + E4M3 scales (1/16 byte) per weight."""
    per_matrix = cs.inter * cs.hidden
    return 3 * per_matrix * 9 // 16


def layer_counters(cs, T, touched, has_shared, decode=False):
    """Algorithmic bytes / FLOPs of one call (touched experts' weights counted once).  Decode-sized
    batches run both grouped GEMMs as one launch ("grouped_gemms") whose down projection stores
    one FP32 row per assignment instead of reducing into the token rows."""
    H, I, k = cs.hidden, cs.inter, cs.top_k
    R = T * k
    rows = R + (T if has_shared else 0)
    n_exp = touched + (1 if has_shared else 0)
    w13 = n_exp * 2 * I * H * 9 // 16
    w2 = n_exp * H * I * 9 // 16
    act_in = T * H * 2 + T * cs.experts * 4
    out = T * H * 2
    g1 = w13 + rows * H * 9 // 16 + rows * I * 9 // 16
    g2 = w2 + rows * I * 9 // 16 + (rows * H * 4 if decode else T * H * 4)
    return dict(
        flops=rows * 6 * H * I,
        grouped_gemms_flops=rows * 6 * H * I,
        grouped_gemms=g1 + g2,
        gemm1_swiglu_flops=rows * 4 * H * I,
        gemm2_combine_flops=rows * 2 * H * I,
        layer_bytes=w13 + w2 + act_in + out,
        # GEMM1: gate/up weights + gathered activation codes/scales + requantised h out
        gemm1_swiglu=g1,
        # GEMM2: down weights + h codes/scales in + the FP32 token accumulator (or, decode, the
        # stored FP32 rows) written
        gemm2_combine=g2,
        act_quant=2 * T * H * 2 + T * H * 9 // 16 + T * H * 4,
        router_plan=T * cs.experts * 4 + R * 16,
        bf16_out=T * H * 4 + T * H * 2,
    )


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(tokens_per_rank: float, seconds_per_rank: float, world: int):
    """Whole-job throughput: all ranks' tokens over the slowest rank's time."""
    tmax = max_over_ranks(seconds_per_rank, world)
    return tokens_per_rank * world / tmax, tmax


# ----------------------------------------------------------------------------------------- oracle
def oracle_inputs(cs, wg, wu, wd, sh, need):
    import numpy as np
    import oracle
    experts = [None] * cs.experts
    for e in sorted(set(int(i) for i in need)):
        experts[e] = oracle.QuantExpert.from_bf16(wg[e].cpu(), wu[e].cpu(), wd[e].cpu())
    sho = oracle.QuantExpert.from_bf16(*[s.cpu() for s in sh]) if sh is not None else None
    return experts, sho


def oracle_call(cs, x_cpu, lg_np, experts, sho, variant="base"):
    import oracle
    xq, xsf, ts, st = oracle.quantize_bf16(x_cpu)
    v = VARIANTS[variant]
    return oracle.moe_forward(xq, xsf, ts, lg_np, experts, cs.top_k, shared=sho,
                              router_mode=v["router"], router_bias=variant_bias(cs, variant),
                              swiglu_limit=v["swiglu_limit"])


# ----------------------------------------------------------------------------------------- configs
def time_graph(graph, flush, stream, reps):
    """Device time of each replay of a captured layer call (L2 flushed before each, outside the
    events), in ms."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        graph.replay()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def roofline_of(counters, stage_ms, key, hbm_peak, fp4_peak, peak_src):
    """Roofline entry of one kernel: its algorithmic bytes and FLOPs per launch over its measured
    duration, against whichever of the two roofs bounds it (the larger time at 100%%)."""
    sec = stage_ms / 1e3
    nbytes = counters.get(key, 0)
    flops = counters.get(key + "_flops", 0)
    t_hbm = nbytes / (hbm_peak * 1e9)
    t_fp4 = flops / (fp4_peak * 1e12)
    r = {"kernel": key, "avg_launch_us": round(sec * 1e6, 2),
         "algorithmic_bytes_per_launch": nbytes, "algorithmic_flops_per_launch": flops,
         "hbm_frac": round(nbytes / sec / 1e9 / hbm_peak, 4),
         "fp4_frac": round(flops / sec / 1e12 / fp4_peak, 4)}
    if t_fp4 > t_hbm:
        r.update(bound="tensor", achieved=round(flops / sec / 1e12, 1), peak=round(fp4_peak, 1),
                 unit="TFLOP/s", frac=r["fp4_frac"],
                 peak_source=f"{peak_src} bf16 x {FP4_PER_BF16} nominal FP4/BF16 ratio")
    else:
        r.update(bound="hbm", achieved=round(nbytes / sec / 1e9, 1), peak=hbm_peak, unit="GB/s",
                 frac=r["hbm_frac"], peak_source=f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)")
    return r


def oracle_baselines(cs, x_cpu, lg_np, experts, sho, ntok, variant="base"):
    """The oracle on the first ntok tokens of a call: single-threaded, then on every host core
    (its OpenMP build).  Returns the two cpu_baseline records."""
    import oracle
    out = []
    for threads in (1, None):
        used = oracle.use_threads(threads)
        t0 = time.perf_counter()
        oracle_call(cs, x_cpu[:ntok], lg_np[:ntok], experts, sho, variant)
        dt = time.perf_counter() - t0
        out.append({"value": round(ntok / dt, 4), "unit": UNIT, "cores": used, "kind": "oracle",
                    "sample": f"the first {ntok} token(s) of the call (router, plan, both GEMMs, "
                              f"combine; activation quantisation included, weight quantisation "
                              f"untimed)"})
    oracle.use_threads(1)
    return out


def measure_config(args, name, dev, hbm_peak, fp4_peak, peak_src, beta=None, cpu_tokens=0):
    """One layer configuration at its own token count: CUDA-graph replays (L2 flushed before
    each), per-stage times from a replay that records the stage events, the dominant kernel's
    roofline and the oracle on a token sample.  beta replaces the Zipf strength of the routing."""
    import numpy as np
    import oracle
    import synth
    import nvfp4_mixture_experts_softmax_gb300 as moe
    cs = synth.CONFIGS[name]
    T = cs.tokens[0]
    cfg = moe.make_config(cs.experts, cs.hidden, cs.inter, cs.top_k,
                          shared_inter=cs.shared_inter, max_tokens=T)
    wg, wu, wd = synth.gen_all_experts(cs, device=dev)
    sh = synth.gen_shared(cs, device=dev) if cs.has_shared else None
    wbuf = moe.quantize_weights(cfg, wg, wu, wd, shared=sh)
    x = synth.gen_x(cs, T, device=dev)
    lg = synth.gen_logits(cs, T, device=dev, beta=beta)
    ids = moe.plan(lg, cs.top_k)["topk_ids"].cpu().numpy()
    loads = np.bincount(ids.reshape(-1), minlength=cs.experts)
    # the oracle's inputs for the CPU sample: only the experts its tokens use, before the BF16
    # weights are released
    cpu = []
    if cpu_tokens:
        need = set(ids[:cpu_tokens].reshape(-1).tolist())
        oracle.use_threads(None)
        experts, sho = oracle_inputs(cs, wg, wu, wd, sh, need)
        oracle.use_threads(1)
        x_cpu, lg_np = x[:cpu_tokens].cpu(), lg[:cpu_tokens].cpu().numpy()
    del wg, wu, wd, sh
    torch.cuda.empty_cache()
    ws = torch.empty(moe.workspace_size(cfg, T), dtype=torch.uint8, device=dev)
    y = torch.empty(T, cs.hidden, dtype=torch.bfloat16, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(args.warmup, 3)):
        moe.run(cfg, wbuf, x, lg, y=y, workspace=ws)
    torch.cuda.synchronize()
    assert moe.last_device_status(ws) == 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.run(cfg, wbuf, x, lg, y=y, workspace=ws)
    timer = moe.StageTimer()
    gs = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gs):
        moe.run(cfg, wbuf, x, lg, y=y, workspace=ws, timer=timer)
    reps = max(5, min(args.steps, 20))
    time_graph(g, flush, stream, 3)
    ms = time_graph(g, flush, stream, reps)
    stages = []
    for _ in range(reps):
        flush.zero_()
        gs.replay()
        torch.cuda.synchronize()
        stages.append(timer.stage_ms())
    assert moe.last_device_status(ws) == 0
    stage_ms = {n: statistics.median(s_[n] for s_ in stages) for n in stages[0]}
    touched = int((loads > 0).sum())
    fused = moe.run_kernel_count(cfg, T) == 3     # decode path: both GEMMs in one launch
    counters = layer_counters(cs, T, touched, cs.has_shared, fused)
    per = statistics.median(ms) / 1e3
    if fused:
        stage_ms["grouped_gemms"] = stage_ms.pop("gemm1_swiglu") + stage_ms.pop("gemm2_combine")
        dom = "grouped_gemms"
    else:
        dom = max(("gemm1_swiglu", "gemm2_combine"), key=lambda n: stage_ms[n])
    rec = {
        "workload": f"{name}: {cs.description}" + (f" (Zipf beta {beta})" if beta else ""),
        "tokens": T, "per_call_us": round(per * 1e6, 2),
        "samples_us": [round(v * 1e3, 2) for v in ms],
        "tokens_per_s": round(T / per, 1),
        "eff_tflops": round(counters["flops"] / per / 1e12, 2),
        "layer_hbm_frac": round(counters["layer_bytes"] / per / 1e9 / hbm_peak, 4),
        "fp4_peak_frac": round(counters["flops"] / per / 1e12 / fp4_peak, 4),
        "stage_us": {n: round(v * 1e3, 2) for n, v in stage_ms.items()},
        "roofline": roofline_of(counters, stage_ms[dom], dom, hbm_peak, fp4_peak, peak_src),
        "gpu_launches_per_call": moe.run_kernel_count(cfg, T),
        "touched_experts": touched,
        "expert_loads": {"min": int(loads.min()), "max": int(loads.max()),
                         "empty": int((loads == 0).sum())},
    }
    rec["roofline"]["traffic"] = measured_traffic(f"{dom}@{name}_T{T}")
    if cpu_tokens:
        cpu = oracle_baselines(cs, x_cpu, lg_np, experts, sho, cpu_tokens)
        rec["cpu_baseline"] = cpu[1]
        rec["cpu_baseline_1core"] = cpu[0]
    del wbuf, ws, flush, g, gs
    torch.cuda.empty_cache()
    return rec


def steady_state_decode(args, dev, hbm_peak):
    """Decode without an L2 flush, as consecutive layers of a model run: the call cycles through
    enough distinct weight sets (each its own buffer) that their total is at least 4x the L2, so
    no call finds its weights cached by the previous one."""
    import synth
    import nvfp4_mixture_experts_softmax_gb300 as moe
    cs = synth.CONFIGS["decode"]
    Ts = list(cs.tokens)
    cfg = moe.make_config(cs.experts, cs.hidden, cs.inter, cs.top_k, max_tokens=max(Ts))
    wg, wu, wd = synth.gen_all_experts(cs, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    w0 = moe.quantize_weights(cfg, wg, wu, wd)
    del wg, wu, wd
    nsets = max(2, -(-4 * l2 // w0.numel()))
    sets = [w0] + [w0.clone() for _ in range(nsets - 1)]
    ws = torch.empty(moe.workspace_size(cfg, max(Ts)), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    out = {}
    for i, T in enumerate(Ts):
        x = synth.gen_x(cs, T, device=dev, row0=1000 * i)
        lg = synth.gen_logits(cs, T, device=dev, row0=1000 * i)
        y = torch.empty(T, cs.hidden, dtype=torch.bfloat16, device=dev)
        graphs = []
        for w in sets:
            g = torch.cuda.CUDAGraph()
            moe.run(cfg, w, x, lg, y=y, workspace=ws)
            torch.cuda.synchronize()
            with torch.cuda.graph(g):
                moe.run(cfg, w, x, lg, y=y, workspace=ws)
            graphs.append(g)
        reps = 8 * nsets
        for j in range(2 * nsets):
            graphs[j % nsets].replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for j in range(reps):
            graphs[j % nsets].replay()
        e1.record(stream)
        torch.cuda.synchronize()
        out[str(T)] = round(e0.elapsed_time(e1) * 1e3 / reps, 2)
        del graphs
    assert moe.last_device_status(ws) == 0
    return {"per_T_us": out, "weight_sets": nsets,
            "weight_set_bytes": int(w0.numel()),
            "note": "back-to-back calls, no flush; each call reads a different weight set"}


# Layer variants and precisions measured beside the base layer (the further rows of the layer's
# scope: activations, the variant router, expert sharing, the fused RMSNorm producer feeding the
# quantised-input entry, W4A16 and W4A8): the decode batch sizes, the W4A16 / W4A8 layers also at
# the prefill size; CUDA-graph replays with the L2 flushed before each, as for the headline.
VARIANT_RECORDS = (
    ("relu2", "decode", dict(activation="relu2"), None, False),
    ("swiglu_oai", "decode", dict(activation="swiglu_oai", swiglu_limit=7.0), None, False),
    ("sqrtsoftplus_clamp", "decode", dict(router="sqrtsoftplus", swiglu_limit=10.0), None, False),
    ("sharing_80pct", "decode", {}, "shared_80", False),
    ("rmsnorm_producer_into_layer", "decode", {}, None, True),
    ("w4a16", "decode", dict(precision="w4a16"), None, False),
    ("w4a8", "decode", dict(precision="w4a8"), None, False),
    ("w4a16_prefill", "prefill", dict(precision="w4a16"), None, False),
    ("w4a8_prefill", "prefill", dict(precision="w4a8"), None, False),
)


def measure_variants(args, dev, hbm_peak):
    """One record per entry of VARIANT_RECORDS: per-call time at each batch size, tokens/s, the
    touched experts and their weight bytes over the call time as a fraction of HBM bandwidth."""
    import types
    import numpy as np
    import oracle
    import synth
    import nvfp4_mixture_experts_softmax_gb300 as moe
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    out = {}
    for name, wl, kw, routing, producer in VARIANT_RECORDS:
        cs, Ts = workload(wl)
        if routing:            # the sharing workloads are defined for small batches
            Ts = [8]
        Tmax = max(Ts)
        gated = kw.get("activation") != "relu2"
        cfg = moe.make_config(cs.experts, cs.hidden, cs.inter, cs.top_k,
                              shared_inter=cs.shared_inter, max_tokens=Tmax, **kw)
        wg, wu, wd = synth.gen_all_experts(cs, device=dev)
        sh = synth.gen_shared(cs, device=dev) if cs.has_shared else None
        wbuf = moe.quantize_weights(
            cfg, wg if gated else None, wu, wd,
            shared=None if sh is None else (sh[0] if gated else None, sh[1], sh[2]))
        del wg, wu, wd, sh
        torch.cuda.empty_cache()
        bias = None
        if kw.get("router") == "sqrtsoftplus":
            bias = variant_bias(cs, "sqrtsoftplus_clamp")
            moe.set_router_bias(cfg, wbuf, torch.from_numpy(bias))
        ws = torch.empty(moe.workspace_size(cfg, Tmax), dtype=torch.uint8, device=dev)
        gamma = torch.from_numpy(np.random.default_rng(7).normal(1.0, 0.1, cs.hidden)
                                 .astype(np.float32)).to(torch.bfloat16).to(dev)
        pws = torch.empty(max(int(moe.lib().moe_rmsnorm_workspace_size(Tmax)), 256),
                          dtype=torch.uint8, device=dev)
        # weight bytes per element: NVFP4 (also the W4A16 layer's weights) 1/2 + 1/16, MXFP4 1/2 + 1/32
        per_elem = (1 / 2 + 1 / 32) if kw.get("precision") == "w4a8" else (1 / 2 + 1 / 16)
        exp_bytes = (3 if gated else 2) * cs.inter * cs.hidden * per_elem
        rec = {"workload": f"{wl}: {cs.description}", "variant": {**kw, "routing": routing,
               "producer": producer}, "per_T_us": {}, "touched_experts": {},
               "weight_hbm_frac": {}, "gpu_launches_per_call": {}}
        tot_tok, tot_s = 0, 0.0
        for i, T in enumerate(Ts):
            x = synth.gen_x(cs, T, device=dev, row0=1000 * i)
            lg = gen_router_logits(types.SimpleNamespace(routing=routing), cs, T, i, dev)
            y = torch.empty(T, cs.hidden, dtype=torch.bfloat16, device=dev)

            def call():
                if producer:
                    q = moe.rmsnorm_quantize_act(x, gamma, 1e-6, workspace=pws)
                    moe.run(cfg, wbuf, None, lg, y=y, workspace=ws, quantized=q)
                else:
                    moe.run(cfg, wbuf, x, lg, y=y, workspace=ws)
            for _ in range(3):
                flush.zero_()
                call()
            torch.cuda.synchronize()
            assert moe.last_device_status(ws) == 0, name
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                call()
            ms = statistics.median(time_graph(g, flush, stream, max(5, min(args.steps, 20))))
            del g
            if kw.get("router") == "sqrtsoftplus":
                ids, _ = oracle.router(lg.cpu().numpy(), cs.top_k, "sqrtsoftplus", bias)
            else:
                ids = moe.plan(lg, cs.top_k)["topk_ids"].cpu().numpy()
            touched = len(np.unique(ids)) + (1 if cs.has_shared else 0)
            rec["per_T_us"][str(T)] = round(ms * 1e3, 2)
            rec["touched_experts"][str(T)] = touched
            rec["weight_hbm_frac"][str(T)] = round(touched * exp_bytes / (ms / 1e3) / 1e9 / hbm_peak,
                                                   4)
            rec["gpu_launches_per_call"][str(T)] = moe.run_kernel_count(cfg, T) + (2 if producer
                                                                                 else 0)
            tot_tok += T
            tot_s += ms / 1e3
        rec["tokens_per_s"] = round(tot_tok / tot_s, 1)
        out[name] = rec
        del wbuf, ws
        torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------------------- ours
def run_ours(args, world, rank, local):
    import numpy as np
    import synth
    import nvfp4_mixture_experts_softmax_gb300 as moe
    from nvfp4_mixture_experts_softmax_gb300 import _build

    _build.build()
    dev = torch.device("cuda", local)
    cs, Ts = workload(args.workload, args.tokens)
    has_shared = cs.has_shared
    Tmax = max(Ts)
    cfg = moe.make_config(cs.experts, cs.hidden, cs.inter, cs.top_k, shared_inter=cs.shared_inter,
                          max_tokens=Tmax, **VARIANTS[args.variant])
    wg, wu, wd = synth.gen_all_experts(cs, device=dev)
    sh = synth.gen_shared(cs, device=dev) if has_shared else None
    wbuf = moe.quantize_weights(cfg, wg, wu, wd, shared=sh)
    if variant_bias(cs, args.variant) is not None:
        moe.set_router_bias(cfg, wbuf, torch.from_numpy(variant_bias(cs, args.variant)))
    xs = {T: synth.gen_x(cs, T, device=dev, row0=1000 * i) for i, T in enumerate(Ts)}
    lgs = {T: gen_router_logits(args, cs, T, i, dev) for i, T in enumerate(Ts)}
    ws = torch.empty(moe.workspace_size(cfg, Tmax), dtype=torch.uint8, device=dev)
    ys = {T: torch.empty(T, cs.hidden, dtype=torch.bfloat16, device=dev) for T in Ts}

    # touched experts per call (read once before timing: the device plan for the base router, the
    # oracle's router for the variant, whose selection moe_plan does not implement)
    def route_ids(T):
        if VARIANTS[args.variant]["router"] == "softmax":
            return moe.plan(lgs[T], cs.top_k)["topk_ids"].cpu().numpy()
        import oracle
        ids, _ = oracle.router(lgs[T].cpu().numpy(), cs.top_k, VARIANTS[args.variant]["router"],
                               variant_bias(cs, args.variant))
        return ids

    touched = {T: len(np.unique(route_ids(T))) for T in Ts}
    rows_per_expert = {T: sorted(np.unique(route_ids(T), return_counts=True)[1].tolist(),
                                 reverse=True) for T in Ts}
    launches = {T: moe.run_kernel_count(cfg, T) for T in Ts}
    fused = {T: launches[T] == 3 for T in Ts}   # decode path: both GEMMs in one launch
    counters = {T: layer_counters(cs, T, touched[T], has_shared, fused[T]) for T in Ts}

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call(i, timer=None):
        T = Ts[i % len(Ts)]
        moe.run(cfg, wbuf, xs[T], lgs[T], y=ys[T], workspace=ws, timer=timer)
        return T

    for i in range(args.warmup):
        flush.zero_()
        call(i)
    torch.cuda.synchronize()
    assert moe.last_device_status(ws) == 0, "device status after warm-up"

    # one CUDA graph per batch size (the layer reads nothing back and allocates nothing, so a
    # whole call is capturable).  The timed graphs hold only the layer's kernels, so consecutive
    # kernels can overlap through programmatic dependent launch; a second set of graphs also
    # records the library's stage events (event nodes between kernels break that overlap) and is
    # replayed separately for the per-stage breakdown.
    graphs, staged = {}, {}
    try:
        for T in Ts:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                moe.run(cfg, wbuf, xs[T], lgs[T], y=ys[T], workspace=ws)
            graphs[T] = g
            timer = moe.StageTimer()
            gs = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gs):
                moe.run(cfg, wbuf, xs[T], lgs[T], y=ys[T], workspace=ws, timer=timer)
            staged[T] = (gs, timer)
        for i in range(len(Ts)):
            flush.zero_()
            graphs[Ts[i]].replay()
            staged[Ts[i]][0].replay()
        torch.cuda.synchronize()
    except RuntimeError:
        graphs, staged = {}, {}

    idle_before = gpu_activity(local)
    sampler = ClockSampler(local)
    sampler.start()
    t_settle = time.time()
    while time.time() - t_settle < 0.4:      # hold the GPU busy so sampled clocks are under load
        flush.zero_()
        torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    w0 = time.time()
    tokens = 0
    Tseq = []
    for i in range(args.steps):
        T = Ts[i % len(Ts)]
        flush.zero_()
        ev[i][0].record(stream)
        if graphs:
            graphs[T].replay()
        else:
            moe.run(cfg, wbuf, xs[T], lgs[T], y=ys[T], workspace=ws)
        ev[i][1].record(stream)
        tokens += T
        Tseq.append(T)
    torch.cuda.synchronize()
    barrier(world)
    w1 = time.time()
    time.sleep(0.1)
    sampler.stop()
    st = moe.last_device_status(ws)
    assert st == 0, f"device status {st}"
    call_ms = [a.elapsed_time(b) for a, b in ev]

    # per-stage breakdown: the same steps replayed with the stage events recorded
    stage_records = []
    for i in range(args.steps):
        T = Ts[i % len(Ts)]
        flush.zero_()
        if staged:
            g, timer = staged[T]
            g.replay()
        else:
            timer = moe.StageTimer()
            moe.run(cfg, wbuf, xs[T], lgs[T], y=ys[T], workspace=ws, timer=timer)
        torch.cuda.synchronize()
        stage_records.append(timer.stage_ms())

    # the decode path's one GEMM launch is recorded under GEMM1's stage and leaves GEMM2's empty
    stage_names = list(moe.STAGES)
    if all(fused.values()):
        stage_names = [n for n in stage_names if n != "gemm2_combine"]
        stage_names[stage_names.index("gemm1_swiglu")] = "grouped_gemms"

    def stage_name(n):
        return "grouped_gemms" if n == "gemm1_swiglu" and all(fused.values()) else n

    stage_ms = {n: 0.0 for n in stage_names}
    stage_ms_T = {T: {n: [] for n in stage_names} for T in Ts}
    per_T_ms = {T: [] for T in Ts}
    for T, s_, c in zip(Tseq, stage_records, call_ms):
        for n0, v in s_.items():
            n = stage_name(n0)
            if n not in stage_ms:
                continue
            stage_ms[n] += v
            stage_ms_T[T][n].append(v)
        per_T_ms[T].append(c)
    dev_s = sum(call_ms) / 1e3
    value, tmax = aggregate(tokens, dev_s, world)

    hbm_peak, bf16_peak, peak_src = measured_peaks()
    tot = {key: sum(counters[T][key] for T in Tseq) for key in counters[Ts[0]]}
    dominant = max(stage_ms, key=stage_ms.get)
    # roofline of the dominant kernel on the launches of the largest batch of the workload: the
    # weight-streaming decode batches against HBM bandwidth, the large batches' GEMMs against the
    # dense FP4 tensor peak (measured BF16 peak x the nominal FP4/BF16 ratio)
    Tr = max(Ts)
    dom_launch_s = statistics.mean(stage_ms_T[Tr][dominant]) / 1e3
    tensor_bound = Tr > 64 and dominant in ("gemm1_swiglu", "gemm2_combine", "grouped_gemms")
    if tensor_bound:
        fp4_peak = bf16_peak * FP4_PER_BF16
        achieved = counters[Tr][dominant + "_flops"] / dom_launch_s / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(fp4_peak, 1),
                "unit": "TFLOP/s", "frac": round(achieved / fp4_peak, 4),
                "algorithmic_flops_per_launch": counters[Tr][dominant + "_flops"],
                "peak_source": (f"{peak_src} bf16 {bf16_peak} TFLOP/s x {FP4_PER_BF16} nominal "
                                f"FP4/BF16 ratio")}
    else:
        achieved = counters[Tr][dominant] / dom_launch_s / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4),
                "algorithmic_bytes_per_launch": counters[Tr][dominant],
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                else "fallback"}
    traffic = measured_traffic(f"{dominant}@{args.workload}_T{Tr}")
    eff_tflops = tot["flops"] / dev_s / 1e12
    layer_gbs = tot["layer_bytes"] / dev_s / 1e9

    # ---- end to end through the C ABI with host buffers (pinned), copies inside the timed region
    hx = {T: xs[T].cpu().pin_memory() for T in Ts}
    hl = {T: lgs[T].cpu().pin_memory() for T in Ts}
    hy = {T: torch.empty(T, cs.hidden, dtype=torch.bfloat16).pin_memory() for T in Ts}
    dx = {T: torch.empty_like(xs[T]) for T in Ts}
    dl = {T: torch.empty_like(lgs[T]) for T in Ts}
    e_ms, h2d, d2h = [], 0, 0
    for i in range(args.warmup + args.steps):
        T = Ts[i % len(Ts)]
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dx[T].copy_(hx[T], non_blocking=True)
        dl[T].copy_(hl[T], non_blocking=True)
        moe.run(cfg, wbuf, dx[T], dl[T], y=ys[T], workspace=ws)
        hy[T].copy_(ys[T], non_blocking=True)
        e1.record(stream)
        if i >= args.warmup:
            e_ms.append((e0, e1, T))
    torch.cuda.synchronize()
    e2e_s = sum(a.elapsed_time(b) for a, b, _ in e_ms) / 1e3
    e2e_tokens = sum(T for _, _, T in e_ms)
    for _, _, T in e_ms:
        h2d += T * cs.hidden * 2 + T * cs.experts * 4
        d2h += T * cs.hidden * 2
    e2e_value, _ = aggregate(e2e_tokens, e2e_s, world)

    idle_after = gpu_activity(local)

    # ---- CPU baseline: the oracle, one pass over the workload's token counts, on one core and
    # on every host core (its OpenMP build)
    cpu = cpu1 = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        need = set()
        for T in Ts:
            need.update(route_ids(T).reshape(-1).tolist())
        experts, sho = oracle_inputs(cs, wg, wu, wd, sh, need)
        recs = []
        for threads in (1, None):
            used = oracle.use_threads(threads)
            c_tok, c_s = 0, 0.0
            for T in Ts:
                xc, lc = xs[T].cpu(), lgs[T].cpu().numpy()
                t0 = time.perf_counter()
                oracle_call(cs, xc, lc, experts, sho, args.variant)
                c_s += time.perf_counter() - t0
                c_tok += T
            recs.append({"value": c_tok / c_s, "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": f"one layer call at each T in {Ts} ({c_tok} tokens), C++ oracle "
                                   f"on {used} thread(s) incl. activation quantisation; weight "
                                   f"quantisation untimed"})
        oracle.use_threads(1)
        cpu1, cpu = recs

    # ---- every other configuration, each at its own token count (one sub-record each)
    workloads = {}
    if world == 1 and args.workloads != "none" and not args.tokens and args.variant == "base" \
            and not args.routing and args.workload == "decode":
        del wg, wu, wd
        torch.cuda.empty_cache()
        fp4_peak = bf16_peak * FP4_PER_BF16
        cpu_tok = {"tiny": 16, "prefill": 4, "large": 1, "skewed": 2}
        for name in [w for w in args.workloads.split(",") if w]:
            workloads[name] = measure_config(
                args, name, dev, hbm_peak, fp4_peak, peak_src,
                cpu_tokens=0 if args.no_cpu_baseline else cpu_tok.get(name, 1))
            if name == "skewed":
                # the same layer with a much stronger Zipf bias: a few experts take nearly all
                # tokens and most get a handful or none
                workloads["skewed_beta1"] = measure_config(args, name, dev, hbm_peak, fp4_peak,
                                                           peak_src, beta=1.0)
        workloads["decode_steady_state"] = steady_state_decode(args, dev, hbm_peak)
        workloads["variants"] = measure_variants(args, dev, hbm_peak)

    clocks = sampler.summary(t_settle, w1 + 0.05)
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tmax * 1e3 / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4(e2m1+e4m3) mma, f32 acc",
        "data": "synthetic (seeded SplitMix64/Box-Muller), random-init weights",
        "config": {"workload": f"{args.workload}: {cs.description}", "tokens_per_step": Ts,
                   "variant": {"name": args.variant, **VARIANTS[args.variant]},
                   "routing": args.routing or "iid",
                   "step": f"one moe_run call at T = tokens_per_step[step mod {len(Ts)}]",
                   "l2": "flushed (2x L2 write) before every call, outside the timed events",
                   "launch": ("CUDA graph replay of one moe_run per T (programmatic dependent "
                              "launch between its kernels); stage shares and the roofline kernel's "
                              "duration from a second replay of graphs that also record stage "
                              "events") if graphs else "eager moe_run",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "eff_tflops": round(eff_tflops, 3),
        "layer_hbm_gbs": round(layer_gbs, 1),
        "layer_hbm_frac": round(layer_gbs / hbm_peak, 4),
        "per_T_us": {str(T): round(statistics.median(v) * 1e3, 2) for T, v in per_T_ms.items()},
        "touched_experts": {str(T): touched[T] for T in Ts},
        "routing": {"workload": args.routing or "iid N(0,1) logits",
                    "rows_per_expert": {str(T): rows_per_expert[T] for T in Ts},
                    "useful_weight_bytes": {str(T): touched[T] * expert_bytes(cs) for T in Ts}},
        "stage_share": {n: round(v / sum(stage_ms.values()), 4) for n, v in stage_ms.items()},
        "stage_us_per_T": {str(T): {n: round(statistics.median(v) * 1e3, 2) for n, v in d.items() if v}
                           for T, d in stage_ms_T.items()},
        "fp4_peak_frac": round(eff_tflops / (bf16_peak * FP4_PER_BF16), 4),
        "roofline": dict(kernel=f"{dominant} (T={Tr} launches)", **roof,
                         avg_launch_us=round(dom_launch_s * 1e6, 2), traffic=traffic),
        "cpu_baseline": cpu,
        "cpu_baseline_1core": cpu1,
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d // max(len(e_ms), 1),
                "d2h_bytes_per_step": d2h // max(len(e_ms), 1)},
        "gpu_launches": sum(launches[T] for T in Tseq),
        "clocks": clocks,
        "gpu_idle": {"before": idle_before, "after": idle_after},
        "samples_us": [round(v * 1e3, 2) for v in call_ms],
        "wall_s_timed_region": round(w1 - w0, 4),
        "workloads": workloads,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------- producer
def run_producer(args, world, rank, local):
    """RMSNorm + NVFP4 quantisation of the workload's activations [T, H] (two kernels per step)."""
    import numpy as np
    import synth
    import oracle
    import nvfp4_mixture_experts_softmax_gb300 as moe
    from nvfp4_mixture_experts_softmax_gb300 import _build

    _build.build()
    dev = torch.device("cuda", local)
    cs, Ts = workload(args.workload, args.tokens)
    T, H = max(Ts), cs.hidden
    x = synth.gen_x(cs, T, device=dev)
    gamma = torch.from_numpy(np.random.default_rng(7).normal(1.0, 0.1, H).astype(np.float32))
    gamma = gamma.to(torch.bfloat16).to(dev)
    ws = torch.empty(moe.lib().moe_rmsnorm_workspace_size(T), dtype=torch.uint8, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        flush.zero_()
        moe.rmsnorm_quantize_act(x, gamma, 1e-6, workspace=ws)
    torch.cuda.synchronize()
    assert moe.last_device_status(ws) == 0
    sampler = ClockSampler(local)
    sampler.start()
    t_settle = time.time()
    while time.time() - t_settle < 0.4:
        flush.zero_()
        torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    w0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        moe.rmsnorm_quantize_act(x, gamma, 1e-6, workspace=ws)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    w1 = time.time()
    time.sleep(0.1)
    sampler.stop()
    ms = [a.elapsed_time(b) for a, b in ev]
    value, tmax = aggregate(T * args.steps, sum(ms) / 1e3, world)
    hbm_peak, _, peak_src = measured_peaks()
    nbytes = 2 * T * H * 2 + H * 2 + T * H * 9 // 16 + T * 4     # x twice, gamma, codes + scales
    per = statistics.mean(ms) / 1e3
    achieved = nbytes / per / 1e9
    # end to end: host x in, host codes/scales out, copies inside the timed region
    hx = x.cpu().pin_memory()
    dx = torch.empty_like(x)
    hc = torch.empty(T, H // 2, dtype=torch.uint8).pin_memory()
    hs = torch.empty(T, H // 16, dtype=torch.uint8).pin_memory()
    e_ms = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dx.copy_(hx, non_blocking=True)
        codes, sf, _ = moe.rmsnorm_quantize_act(dx, gamma, 1e-6, workspace=ws)
        hc.copy_(codes, non_blocking=True)
        hs.copy_(sf, non_blocking=True)
        e1.record(stream)
        if i >= args.warmup:
            e_ms.append((e0, e1))
    torch.cuda.synchronize()
    e2e_value, _ = aggregate(T * len(e_ms), sum(a.elapsed_time(b) for a, b in e_ms) / 1e3, world)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n = min(T, 1024)
        xc, gc = x[:n].cpu(), gamma.cpu()
        t0 = time.perf_counter()
        oracle.rmsnorm_quantize(xc, gc, 1e-6)
        dt = time.perf_counter() - t0
        cpu = {"value": n / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"the first {n} rows, single-threaded C++ oracle"}
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tmax * 1e3 / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in, f32 norm (f64 sum of squares), nvfp4 out",
        "data": "synthetic (seeded SplitMix64/Box-Muller)",
        "config": {"workload": f"RMSNorm + NVFP4 producer of the {args.workload} input: T={T}, H={H}",
                   "l2": "flushed (2x L2 write) before every call, outside the timed events",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"kernel": "rmsnorm_amax_kernel + rmsnorm_encode_kernel", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "algorithmic_bytes_per_launch": nbytes,
                     "avg_launch_us": round(per * 1e6, 2),
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)", "traffic": None},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": T * H * 2,
                "d2h_bytes_per_step": T * H * 9 // 16},
        "gpu_launches": 2 * args.steps,
        "clocks": sampler.summary(t_settle, w1 + 0.05),
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------- reference
def run_reference(args, world, rank, local):
    if rank != 0:
        return
    import numpy as np
    import synth
    cs, Ts = workload(args.workload, args.tokens)
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    wg, wu, wd = synth.gen_all_experts(cs, device=dev)
    sh = synth.gen_shared(cs, device=dev) if cs.has_shared else None
    xs = {T: synth.gen_x(cs, T, device=dev, row0=1000 * i).cpu() for i, T in enumerate(Ts)}
    lgs = {T: gen_router_logits(args, cs, T, i, dev).cpu().numpy() for i, T in enumerate(Ts)}
    import oracle
    need = set()
    for T in Ts:
        ids, _ = oracle.router(lgs[T], cs.top_k, VARIANTS[args.variant]["router"],
                               variant_bias(cs, args.variant))
        need.update(ids.reshape(-1).tolist())
    experts, sho = oracle_inputs(cs, wg, wu, wd, sh, need)
    del wg, wu, wd
    # per-step token sample: one token per call costs about one expert-set decode; size the
    # sample so that warm-up + timed steps fit the budget
    t0 = time.perf_counter()
    oracle_call(cs, xs[Ts[0]][:1], lgs[Ts[0]][:1], experts, sho, args.variant)
    one = max(time.perf_counter() - t0, 1e-3)
    nsteps = args.warmup + args.steps
    per_step = args.ref_budget_s / max(nsteps, 1)
    cap = max(1, int(per_step / one))
    tok, secs = 0, 0.0
    for i in range(nsteps):
        T = Ts[i % len(Ts)]
        n = min(T, cap)
        t0 = time.perf_counter()
        oracle_call(cs, xs[T][:n], lgs[T][:n], experts, sho, args.variant)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            tok += n
            secs += dt
    value = tok / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32 (host oracle)",
        "data": "synthetic (seeded SplitMix64/Box-Muller), random-init weights",
        "config": {"workload": f"{args.workload}: {cs.description}", "tokens_per_step": Ts,
                   "variant": {"name": args.variant, **VARIANTS[args.variant]},
                   "token_sample_cap": cap},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"per step the first min(T, {cap}) tokens of that step's call"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank, local)
        elif args.producer:
            run_producer(args, world, rank, local)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
