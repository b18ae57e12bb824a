"""Benchmark of the folded multi-branch verification pass.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config 1.5b] [--delta 0.1]

One step = one verification pass (every layer: gate, compaction, source
resolution, QKV, attention, O, FFN, residual) over one denoising block of
R * (B+1) * L branch-position rows.  Prints one JSON line.  Under torchrun
every rank runs its own independent requests (replicas; no data-path
collective) and rank 0 prints the whole-job numbers (max time over ranks).
"""
from __future__ import annotations

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

METRIC = "verify passes/s and branch-tokens/s (folded vs dense), % of roofline"
UNIT = "branch-tokens/s"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p["bf16_tflops_sustained"], "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def workload_desc(cfg):
    return (f"{cfg.name}-shaped: {cfg.n_layers} layers, d={cfg.d_model}, {cfg.n_q_heads}q/{cfg.n_kv_heads}kv "
            f"heads x {cfg.head_dim}, SwiGLU {cfg.d_ffn}, {cfg.dtype}; R={cfg.n_requests}, main + B={cfg.n_drafts} "
            f"drafts ({cfg.tree} tree), L={cfg.block_len}, prefix {cfg.prefix_len}")


# ------------------------------------------------------------------ algorithmic work model

def layer_work(cfg, t_rc):
    """Algorithmic FLOPs and bytes of one folded layer with t_rc recompute rows.
    Weights are counted once per layer (each weight tile streamed once for all
    rows), the prefix K/V once per request, activations once per read/write."""
    d, nq, nkv, hd, F = cfg.d_model, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.d_ffn
    T, R, P, L = cfg.rows, cfg.n_requests, cfg.prefix_len, cfg.block_len
    wb = 2 if cfg.dtype == "bf16" else 4
    p_qkv, p_o, p_ffn = d * (nq + 2 * nkv) * hd, nq * hd * d, 3 * d * F
    fam = {}
    fam["gemm_qkv"] = dict(flops=2.0 * t_rc * p_qkv, bytes=p_qkv * wb + t_rc * d * wb + t_rc * (nq + 2 * nkv) * hd * wb)
    fam["gemm_o"] = dict(flops=2.0 * T * p_o, bytes=p_o * wb + T * nq * hd * wb + 2 * T * d * 4)
    fam["gemm_gateup"] = dict(flops=2.0 * t_rc * 2 * d * F, bytes=2 * d * F * wb + t_rc * d * wb + t_rc * F * wb)
    fam["gemm_down"] = dict(flops=2.0 * t_rc * d * F, bytes=d * F * wb + t_rc * F * wb + t_rc * d * 4)
    fam["attn_prefix"] = dict(flops=4.0 * t_rc * nq * hd * P, bytes=R * 2 * P * nkv * hd * wb + t_rc * nq * hd * wb)
    fam["attn_block"] = dict(flops=4.0 * T * nq * hd * L, bytes=t_rc * (nq + 2 * nkv) * hd * wb + T * nq * hd * wb)
    # gate: h and the recompute rows of f read, H written, the attention
    # RMSNorm of the recompute rows written; norm: the FFN RMSNorm
    fam["gate"] = dict(flops=10.0 * T * d, bytes=(2 * T + t_rc) * d * 4 + t_rc * d * wb)
    fam["norm"] = dict(flops=4.0 * t_rc * d, bytes=t_rc * d * (4 + wb))
    return fam


def weight_bytes(cfg):
    wb = 2 if cfg.dtype == "bf16" else 4
    d, nq, nkv, hd, F = cfg.d_model, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.d_ffn
    return cfg.n_layers * wb * (d * (nq + 2 * nkv) * hd + nq * hd * d + 3 * d * F)


def pass_work(cfg, rc_counts):
    tot = {"flops": 0.0, "bytes": 0.0}
    for t_rc in rc_counts:
        for v in layer_work(cfg, int(t_rc)).values():
            tot["flops"] += v["flops"]
            tot["bytes"] += v["bytes"]
    return tot


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch,
# from the committed ncu capture of the current kernels (the 1.5B GEMM
# summary under profiles/).  A kernel changed since its capture has no entry
# (traffic is then reported as null).
NCU_TRAFFIC = {
    ("1.5b", "gemm_gateup"): 55.29e6,
    ("1.5b", "gemm_down"): 28.70e6,
    ("1.5b", "gemm_o"): 7.57e6,
    ("1.5b", "gemm_qkv"): 6.55e6,
}


# ------------------------------------------------------------------ multi-GPU replicas

def replica_seed(rank: int) -> int:
    """Every rank verifies its own independent requests (weak scaling)."""
    return rank


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The job's time is the slowest rank's time (no data-path collective)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, rows_per_pass: int, passes: int, seconds: float) -> float:
    """Branch-tokens per second over all ranks: each rank ran `passes` passes
    of `rows_per_pass` rows; the job took the slowest rank's `seconds`."""
    return world * rows_per_pass * passes / seconds


# ------------------------------------------------------------------ clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.6)   # nvidia-smi is sampling before the timed region starts
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle baseline

def oracle_sample(cfg, wl, delta, budget_s=12.0):
    """Time the oracle (float64, as it stands) on the first layers of the same
    workload until ~budget_s of CPU work; extrapolate to a whole pass."""
    import oracle
    H = wl.hidden.double().cpu().numpy()
    t0 = time.perf_counter()
    layers = 0
    t_layers = 0.0
    while layers < cfg.n_layers:
        W = oracle.layer_weights_f64(wl.weights[layers])
        pk = wl.prefix_k[layers].double().cpu().numpy()
        pv = wl.prefix_v[layers].double().cpu().numpy()
        t1 = time.perf_counter()
        out = np.empty_like(H)
        for r in range(cfg.n_requests):
            out[r] = oracle.folded_layer_resolved(H[r], wl.parents[r], delta, W, pk[r], pv[r], cfg)[0]
        t_layers += time.perf_counter() - t1
        H = out
        layers += 1
        if time.perf_counter() - t0 > budget_s:
            break
    per_pass = t_layers / layers * cfg.n_layers
    return {"value": cfg.rows / per_pass, "unit": UNIT, "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"float64 oracle on layers 0..{layers - 1} of {cfg.n_layers} of the same workload, "
                      f"time per layer x {cfg.n_layers}", "passes_per_s": 1.0 / per_pass}


# ------------------------------------------------------------------ config sweep

def sweep(args, dev):
    """Folded vs dense throughput for every workload config on this GPU."""
    import torch
    import synth
    import sparse_reuse_gb300 as sf
    pk = peaks()
    runs = [("tiny", None, [synth.CONFIGS["tiny"].delta]), ("1.5b", None, [0.1]), ("7b", None, [0.1]),
            ("8b", None, list(synth.DELTA_SWEEP_8B))] + [("14b", b, [0.1]) for b in synth.DRAFT_SWEEP_14B]
    for name, drafts, deltas in runs:
        cfg = synth.CONFIGS[name] if drafts is None else synth.CONFIGS[name].with_(n_drafts=drafts)
        wl = synth.make_workload(cfg, seed=0, device=dev)
        ctx = sf.from_config(cfg, wl.weights)
        stream = torch.cuda.Stream(device=dev)
        nl = cfg.n_layers
        out = torch.empty_like(wl.hidden)
        fold = torch.empty((nl, cfg.n_requests, cfg.n_branches, cfg.block_len), dtype=torch.uint8, device=dev)
        rcc = torch.empty((nl,), dtype=torch.int32, device=dev)
        pk_ = wl.prefix_k if cfg.prefix_len else None
        pv_ = wl.prefix_v if cfg.prefix_len else None

        def timed(dl):
            for _ in range(args.warmup):
                ctx.verify(wl.hidden, wl.parents, pk_, pv_, dl, out=out, fold=fold, rc_count=rcc, stream=stream)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                ctx.verify(wl.hidden, wl.parents, pk_, pv_, dl, out=out, fold=fold, rc_count=rcc, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / args.steps

        dense_ms = timed(0.0)
        dense_rc = rcc.cpu().numpy().tolist()
        for dl in deltas:
            ms = timed(dl)
            rc = rcc.cpu().numpy().tolist()
            pw = pass_work(cfg, rc)
            t_roof = max(pw["flops"] / (pk["bf16_tflops"] * 1e12), pw["bytes"] / (pk["hbm_gbs"] * 1e9))
            pwd = pass_work(cfg, dense_rc)
            t_roof_d = max(pwd["flops"] / (pk["bf16_tflops"] * 1e12), pwd["bytes"] / (pk["hbm_gbs"] * 1e9))
            line = {"metric": METRIC, "config": workload_desc(cfg), "delta": dl, "dtype": cfg.dtype,
                    "ms_per_pass": ms, "passes_per_s": 1e3 / ms, "branch_tokens_per_s": cfg.rows * 1e3 / ms,
                    "fold_fraction": float(fold[:, :, 1:].float().mean().item()) if cfg.n_drafts else 0.0,
                    "rc_rows_mean": sum(rc) / len(rc), "pass_roofline_frac": t_roof * 1e3 / ms,
                    "roofline_bound": "tensor" if pw["flops"] / (pk["bf16_tflops"] * 1e12) >
                                      pw["bytes"] / (pk["hbm_gbs"] * 1e9) else "hbm",
                    "dense_ms_per_pass": dense_ms, "dense_branch_tokens_per_s": cfg.rows * 1e3 / dense_ms,
                    "dense_pass_roofline_frac": t_roof_d * 1e3 / dense_ms, "speedup_vs_dense": dense_ms / ms}
            print(json.dumps(line), flush=True)
        ctx.close()
        del wl, ctx
        torch.cuda.empty_cache()


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="1.5b")
    ap.add_argument("--delta", type=float, default=None)
    ap.add_argument("--drafts", type=int, default=None)
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--layers", type=int, default=None,
                    help="profiling only: run the first N layers of the config")
    ap.add_argument("--profile-only", action="store_true",
                    help="profiling only: warm-up and timed passes, nothing else, no JSON line")
    ap.add_argument("--sweep", action="store_true",
                    help="every workload config (8B delta sweep, 14B draft sweep): one JSON line each")
    args = ap.parse_args()

    import torch
    import synth

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    cfg = synth.CONFIGS[args.config]
    if args.drafts is not None:
        cfg = cfg.with_(n_drafts=args.drafts)
    if args.layers is not None:
        cfg = cfg.with_(n_layers=args.layers)
    delta = cfg.delta if args.delta is None else args.delta
    config = {"workload": workload_desc(cfg), "R": cfg.n_requests, "B": cfg.n_drafts, "L": cfg.block_len,
              "P": cfg.prefix_len, "layers": cfg.n_layers, "d_model": cfg.d_model, "delta": delta,
              "parallelism": f"replicas x{args.gpus}" if args.gpus > 1 else "single GPU"}

    if args.impl == "reference":
        if rank != 0:
            return
        wl = synth.make_workload(cfg, seed=0, device="cpu")
        times = []
        samp = None
        for _ in range(args.warmup + args.steps):
            samp = oracle_sample(cfg, wl, delta, budget_s=0.0)   # one layer per step
            times.append(1.0 / samp["passes_per_s"])
        t = times[args.warmup:]
        per_pass = sum(t) / len(t)
        v = cfg.rows / per_pass
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_pass * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": v, "unit": UNIT, "cores": samp["cores"], "kind": "oracle",
                                 "sample": "float64 oracle, one layer per step, time x n_layers"},
                "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import sparse_reuse_gb300 as sf

    if args.sweep:
        sweep(args, dev)
        return

    wl = synth.make_workload(cfg, seed=replica_seed(rank), device=dev)
    ctx = sf.from_config(cfg, wl.weights)
    stream = torch.cuda.Stream(device=dev)
    nl, T, d = cfg.n_layers, cfg.rows, cfg.d_model
    out = torch.empty_like(wl.hidden)
    fold = torch.empty((nl, cfg.n_requests, cfg.n_branches, cfg.block_len), dtype=torch.uint8, device=dev)
    src = torch.empty(fold.shape, dtype=torch.int32, device=dev)
    rcc = torch.empty((nl,), dtype=torch.int32, device=dev)

    def step(dl):
        ctx.verify(wl.hidden, wl.parents, wl.prefix_k, wl.prefix_v, dl, out=out, fold=fold, src=src,
                   rc_count=rcc, stream=stream)

    def barrier():
        if dist is not None:
            dist.barrier()

    def timed(dl, k, w):
        for _ in range(w):
            step(dl)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        s0 = stats0 = ctx.stats()["kernel_launches"]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k):
            step(dl)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
        return ms, ctx.stats()["kernel_launches"] - s0

    if args.profile_only:
        timed(delta, args.steps, args.warmup)
        ctx.close()
        return
    with ClockSampler(local) as clk:
        ms, launches = timed(delta, args.steps, args.warmup)
    rc_fold = rcc.cpu().numpy().tolist()
    fold_frac = float(fold[:, :, 1:].float().mean().item()) if cfg.n_drafts else 0.0
    ms_step = ms / args.steps
    value = whole_job_rate(world, T, args.steps, ms / 1e3)

    dense = None
    if not args.no_dense:
        dms, _ = timed(0.0, args.steps, args.warmup)
        dense = {"delta": 0.0, "value": whole_job_rate(world, T, args.steps, dms / 1e3), "unit": UNIT,
                 "ms_per_step": dms / args.steps, "passes_per_s": world * args.steps / (dms / 1e3),
                 "rc_count": rcc.cpu().numpy().tolist()}

    # per-family kernel timing (direct launches bracketed by events on the same stream)
    sf.sf_timing_begin(ctx.ctx, sf.FAMILIES)
    for _ in range(args.steps):
        step(delta)
    fam_t = sf.sf_timing_read(ctx.ctx)
    sf.sf_timing_begin(ctx.ctx, [])
    pk = peaks()
    work = {}
    for t_rc in rc_fold:
        for f, v in layer_work(cfg, int(t_rc)).items():
            w = work.setdefault(f, {"flops": 0.0, "bytes": 0.0})
            w["flops"] += v["flops"]
            w["bytes"] += v["bytes"]
    total_fam_ms = sum(v[0] for v in fam_t.values())
    dom = max((f for f in fam_t if f in work), key=lambda f: fam_t[f][0])
    dom_ms, dom_n = fam_t[dom]
    per_launch_s = dom_ms / dom_n / 1e3
    launches_per_pass = dom_n / args.steps
    flops_l = work[dom]["flops"] / launches_per_pass
    bytes_l = work[dom]["bytes"] / launches_per_pass
    t_tensor = flops_l / (pk["bf16_tflops"] * 1e12)
    t_hbm = bytes_l / (pk["hbm_gbs"] * 1e9)
    if t_tensor > t_hbm:
        roof = {"bound": "tensor", "achieved": flops_l / per_launch_s / 1e12, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": bytes_l / per_launch_s / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = NCU_TRAFFIC.get((cfg.name, dom))
    roof["traffic_unit"] = "bytes per launch"
    roof["kernel"] = dom
    roof["peak_source"] = pk["source"]
    roof["share_of_pass"] = dom_ms / total_fam_ms if total_fam_ms else None
    pw = pass_work(cfg, rc_fold)
    t_roof = max(pw["flops"] / (pk["bf16_tflops"] * 1e12), pw["bytes"] / (pk["hbm_gbs"] * 1e9))

    # end to end through the C ABI with host buffers: H2D of the block's hidden
    # states, the pass, D2H of the output hidden states and fold masks
    h_host = wl.hidden.cpu().pin_memory()
    o_host = torch.empty_like(h_host).pin_memory()
    f_host = torch.empty(fold.shape, dtype=torch.uint8).pin_memory()
    h_dev = torch.empty_like(wl.hidden)

    def e2e_step():
        with torch.cuda.stream(stream):
            h_dev.copy_(h_host, non_blocking=True)
        ctx.verify(h_dev, wl.parents, wl.prefix_k, wl.prefix_v, delta, out=out, fold=fold, src=src,
                   rc_count=rcc, stream=stream)
        with torch.cuda.stream(stream):
            o_host.copy_(out, non_blocking=True)
            f_host.copy_(fold, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    stream.synchronize()
    e2e_s = time.perf_counter() - t0
    barrier()
    e2e_s = max_over_ranks(e2e_s, dist, dev)
    e2e = {"value": whole_job_rate(world, T, args.steps, e2e_s), "unit": UNIT,
           "h2d_bytes_per_step": h_host.numel() * h_host.element_size(),
           "d2h_bytes_per_step": o_host.numel() * o_host.element_size() + f_host.numel()}

    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = oracle_sample(cfg, wl, delta)
        cpu.pop("passes_per_s", None)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic (random-init N(0,0.02) weights)",
                "config": dict(config, l2="weights streamed per pass %.2f GB > 129 MB L2" % (weight_bytes(cfg) / 1e9)),
                "passes_per_s": world * args.steps / (ms / 1e3),
                "fold_fraction": fold_frac, "rc_count_per_layer": rc_fold,
                "dense": dense,
                "speedup_vs_dense": (value / dense["value"]) if dense else None,
                "pass_roofline": {"t_roofline_ms": t_roof * 1e3, "frac": t_roof * 1e3 / ms_step,
                                  "flops": pw["flops"], "bytes": pw["bytes"]},
                "roofline": roof,
                "kernel_ms_per_pass": {f: v[0] / args.steps for f, v in fam_t.items()},
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
                "clocks": clk.summary()}
        print(json.dumps(line))
    ctx.close()
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
