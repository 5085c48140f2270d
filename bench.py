#!/usr/bin/env python3
"""Throughput of the routed-expert MoE layer on GB300 (one JSON line).

Workload (default, --config decode): the Qwen4Exp decode verifier block, one
MoE layer call per step: T=16 tokens, hidden 2560, 512 experts, top-10,
SwiGLU intermediate 640, bf16, Zipf(s=1) router bias.  Each step runs the
whole path (route -> permute+gather -> gate/up -> down -> combine) through the
C ABI on inputs already in HBM.  Steps rotate over NL distinct seeded layer
weight sets (8 x 5.03 GB) and as many token batches, so the working set is far
larger than L2 and every step streams its experts' weights from HBM.

--config prefill runs the T=4096 uniform-router layer instead.
--config offload keeps the decode layer's expert records in pinned host
memory behind an HBM slot cache and reports tokens/s, hit rate, bytes fetched
per token and the hidden fraction of the fetch for several wave widths.
--config trace records synthetic decode routes and replays them through the
cache plan for each replacement policy and slot count, and times merged
multi-request calls against one call per request.
--config crossover measures, for token blocks of 16 to 4,096, the time to
bring the routed records from host memory (selected records) against the
whole layer, finds the crossover in the unique-record fraction, and times
macro prefill through the two-layer ring.
--config sidecar times the route-sidecar forward pass (trunk 2560 -> 256,
48 layer embeddings, 512 expert heads, 16 ranked candidates per layer).
--impl reference times the CPU oracle (the reference arm) on the same workload.

Multi-GPU: one process per GPU under torchrun; every rank runs independent
replicas of the layer (token data-parallelism does not shard the expert
bytes, so there is no data-path collective); value = all ranks' tokens / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s at 2560h/512e/top-10; % of HBM / tensor-core roofline"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="decode",
                    choices=["decode", "prefill", "stack48", "sweep", "offload", "trace", "crossover", "sidecar"])
    ap.add_argument("--policy", default="fifo", choices=["fifo", "lru", "score"],
                    help="offload: replacement policy of the expert cache")
    ap.add_argument("--decay", type=float, default=0.9, help="offload/trace: the score policy's use-rate factor")
    ap.add_argument("--slots", default="160,192,256", help="offload: HBM expert slot counts")
    ap.add_argument("--waves", default="1,2,4,0", help="offload: wave widths to time (0 = all misses)")
    ap.add_argument("--int4", action="store_true",
                    help="offload: int4 g64 expert records (quantised from the same weights), copy-first fetch")
    ap.add_argument("--layers", type=int, default=0, help="distinct layer weight sets rotated (0 = auto)")
    ap.add_argument("--experts", type=int, default=0, help="override the expert count (small profiling case)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the tokens per call of decode/prefill (e.g. 32768: the compute-bound regime)")
    ap.add_argument("--plain", action="store_true",
                    help="stream bf16 weights from the plain record layout through TMA tensor maps "
                         "instead of the tile-packed records")
    ap.add_argument("--no-extra", action="store_true",
                    help="decode: leave out the other workloads' short runs (other_configs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's x (the slowest rank's time); x itself on
    one rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, seconds_max: float, world: int) -> float:
    """Units all ranks processed (each rank the same share: weak scaling)
    over the slowest rank's time."""
    return units_per_rank * world / seconds_max


# nominal GB300 figures, reported beside the measured ones: HBM3e ~7.9 TB/s
# (the layer's target is quoted against ~8 TB/s) and dense bf16 2.25 PF/s
NOMINAL_HBM_GBS = 7900.0
NOMINAL_BF16_TFLOPS = 2250.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# kernels each boundary call launches (the grouping calls also launch the
# row gather unless their x_perm argument is null)
PER_CALL = {"moe_route": 2, "moe_route_permute": 1, "moe_permute": 2, "moe_permute_ws": 4, "moe_permute_gather": 2,
            "moe_expert_swiglu_fused": 1, "moe_expert_gateup": 1, "moe_expert_down": 1,
            "moe_combine": 1, "moe_expert_swiglu_fused_weighted": 1, "moe_combine_weighted": 1, "moe_rmsnorm": 1}


def call_launches(call) -> int:
    name, _, a = call
    if name == "moe_permute":
        return 1 if a[10] is None else 2
    if name == "moe_permute_ws":
        return 3 if a[10] is None else 4
    return PER_CALL[name]


# the files whose text a recorded DRAM-traffic figure depends on
KERNEL_SOURCES = {
    "fused": ["fused.cu", "gemm_common.cuh", "ptx.cuh", "common.cuh"],
    "gateup": ["gemm.cu", "gemm_common.cuh", "ptx.cuh", "common.cuh"],
}


def kernel_source_sha(kernel: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(ROOT, "sparse_moe_routed_gb300", "csrc", name), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, units: float):
    """DRAM bytes per launch from a committed ncu summary (per distinct expert,
    scaled by the launch's units), if the kernel's sources are unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        ent = d.get(kernel, {}).get(workload)
        if ent and ent.get("src_sha") == kernel_source_sha(kernel):
            return ent["dram_bytes_per_unit"] * units
    except Exception:
        return None
    return None


class ClockSampler:
    """nvidia-smi clock/throttle samples (every 100 ms) while the GPU works."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        win = [p for (t, p) in self.samples if t0 <= t <= t1] or [p for (_, p) in self.samples]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [num(p[0]) for p in win if num(p[0]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(win[0][1]), "reasons": reasons, "samples": len(win),
                "power_w_max": max((num(p[2]) or 0.0) for p in win)}


def gpu_uuid(dev):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev)


# ------------------------------------------------------------------ oracle
def oracle_tokens_per_s(cfg, host_w, xs_bits, seconds, max_threads=0):
    """Time the CPU oracle on whole decode blocks until `seconds` have passed."""
    import oracle
    threads = oracle.threads(max_threads)
    done = 0
    t0 = time.perf_counter()
    i = 0
    while True:
        xb = xs_bits[i % len(xs_bits)]
        ids, w, gap, _ = oracle.route(xb, host_w["wr"], host_w["bias"], cfg.k)
        oracle.experts_combine(oracle.bits_to_f32(xb), ids, w, cfg.H, cfg.I, wgu_bits=host_w["wgu"],
                               wd_bits=host_w["wd"])
        done += xb.shape[0]
        i += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return done / el, threads, done, el


def host_weights(d):
    import oracle
    return {"wr": oracle.bf16_bits(d["w_router"]), "bias": None if d["bias"] is None else d["bias"].cpu().numpy(),
            "wgu": oracle.bf16_bits(d["w_gateup"]), "wd": oracle.bf16_bits(d["w_down"])}


def workload_name(cfg):
    return f"{cfg.name}_T{cfg.T}_H{cfg.H}_E{cfg.E}_k{cfg.k}_I{cfg.I}" + ("_zipf" if cfg.bias == "zipf" else "")


def layer_config(cfg, NL, world, plain=False):
    """The `config` object of a single-layer workload's line (both arms)."""
    rec = cfg.E * 3 * cfg.H * cfg.I * 2 + cfg.E * cfg.H * 2
    return {"workload": workload_name(cfg), "T": cfg.T, "H": cfg.H, "E": cfg.E, "k": cfg.k, "I": cfg.I,
            "router_bias": cfg.bias or "none", "layer_weight_sets": NL,
            "weights": "plain bf16 records (TMA tensor maps)" if plain else
                       "tile-packed bf16 records (one bulk copy per stage)",
            "l2": f"inputs larger than L2: {NL} distinct layer weight sets rotated ({NL * rec / 1e9:.1f} GB)",
            "parallelism": f"replicas x{world}"}


def run_reference(args):
    """Reference arm: the CPU oracle as it stands, on the host cores."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import torch
    import workloads as wl
    import oracle
    cfg = wl.CONFIGS[args.config]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    d = wl.layer_inputs(cfg, dev, with_x=False)
    hw = host_weights(d)
    del d
    # the decode block whole (16 tokens); larger workloads in 16-token samples
    sample_T = min(cfg.T, 16)
    xs = [oracle.bf16_bits(wl.token_batch(cfg, "cpu", index=i, T=sample_T)) for i in range(4)]
    threads = oracle.threads(0)
    for i in range(args.warmup):
        oracle_step(cfg, hw, xs[i % len(xs)])
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_step(cfg, hw, xs[i % len(xs)])
    el = time.perf_counter() - t0
    value = sample_T * args.steps / el
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": layer_config(cfg, args.layers or (8 if args.config == "decode" else 1), world),
            "tokens_per_step": sample_T,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"{sample_T} tokens of the {cfg.name} workload per step "
                                       f"(route + 10 experts + combine, fp64 C, OpenMP)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def oracle_step(cfg, hw, xb):
    import oracle
    ids, w, gap, _ = oracle.route(xb, hw["wr"], hw["bias"], cfg.k)
    oracle.experts_combine(oracle.bits_to_f32(xb), ids, w, cfg.H, cfg.I, wgu_bits=hw["wgu"], wd_bits=hw["wd"])


# ------------------------------------------------------------------ GPU arm
def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    import numpy as np
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    from sparse_moe_routed_gb300 import MoELayer, _lib, build as gbuild, pack_layer_experts
    if rank == 0:
        gbuild.build()
    if world > 1:
        dist.barrier()
    import workloads as wl

    if args.config in ("stack48", "sweep"):
        return run_stack(args, rank, world, local, dev)
    if args.config == "offload":
        return run_offload(args, rank, world, local, dev)
    if args.config == "trace":
        return run_trace(args, rank, world, local, dev)
    if args.config == "crossover":
        return run_crossover(args, rank, world, local, dev)
    if args.config == "sidecar":
        return run_sidecar(args, rank, world, local, dev)
    line = run_layer(args, rank, world, local, dev)
    if args.config == "decode" and world == 1 and not args.no_extra:
        line["other_configs"] = other_configs(args, rank, world, local, dev)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def sub_args(args, **over):
    """A copy of the command line for one of the other workloads' runs."""
    import copy
    sub = copy.copy(args)
    sub.layers, sub.experts, sub.tokens, sub.plain = 0, 0, 0, False
    sub.no_cpu_baseline, sub.no_e2e, sub.no_extra = True, True, True
    for k, v in over.items():
        setattr(sub, k, v)
    return sub


def other_configs(args, rank, world, local, dev):
    """Short runs of the prefill layer (T = 4,096 and the compute-bound point
    T = 32,768), the int4 48-layer stack and the route sweep, so that the
    default line carries a measurement of every workload: the same code
    paths and timing as their own --config runs, with fewer steps."""
    import torch
    out = {}
    runs = [("prefill", lambda: run_layer(sub_args(args, config="prefill", steps=10, warmup=3), rank, world, local,
                                          dev)),
            ("prefill_T32768", lambda: run_layer(sub_args(args, config="prefill", tokens=32768, steps=5, warmup=3),
                                                 rank, world, local, dev)),
            ("stack48_and_sweep", lambda: run_stack(sub_args(args, config="stack48", steps=5, warmup=3), rank, world,
                                                    local, dev, emit=False, with_sweep=True))]
    keep = ("metric", "value", "unit", "steps", "warmup", "ms_per_step", "config", "roofline", "roofline_other",
            "layer_roofline", "clocks", "gpu_launches", "sweep", "device_status", "dtype")
    for name, fn in runs:
        try:
            res = fn()
        except Exception as e:  # report the failure of one extra run, keep the line
            out[name] = {"error": f"{type(e).__name__}: {e}"[:300]}
            continue
        for key, line in (res.items() if name == "stack48_and_sweep" else [(name, res)]):
            out[key] = {k: line[k] for k in keep if k in line}
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def run_layer(args, rank, world, local, dev):
    """One layer workload (decode or prefill) through the C ABI; returns the
    JSON line."""
    import numpy as np
    import torch
    import torch.distributed as dist
    import workloads as wl
    from sparse_moe_routed_gb300 import MoELayer, _lib, pack_layer_experts

    cfg = wl.CONFIGS[args.config]
    if args.experts:
        from dataclasses import replace
        cfg = replace(cfg, E=args.experts)
    if args.tokens:
        cfg = wl.with_tokens(cfg, args.tokens)
    NL = args.layers or (8 if args.config == "decode" else 1)
    layers, xs, host_w = [], [], None
    for l in range(NL):
        d = wl.layer_inputs(cfg, dev, layer=l, x_seed_offset=l)
        if args.plain:
            layers.append(MoELayer(d["w_router"], d["bias"], d["w_gateup"], d["w_down"], cfg.k, cfg.T))
        else:
            gu, dn = pack_layer_experts(d["w_gateup"], d["w_down"], _lib.MOE_W_BF16, cfg.E, cfg.H, cfg.I)
            layers.append(MoELayer(d["w_router"], d["bias"], gu, dn, cfg.k, cfg.T, fmt=_lib.MOE_W_BF16_TILED,
                                   I=cfg.I))
        xs.append(d["x"])
        if l == 0 and rank == 0 and world == 1 and not args.no_cpu_baseline:
            host_w = host_weights(d)
        if not args.plain:
            del d["w_gateup"], d["w_down"]
        torch.cuda.synchronize()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()

    # per-layer unique experts (deterministic: fixed x per layer) for the byte
    # accounting; this first pass over every layer also checks its status
    U = []
    for l, L in enumerate(layers):
        L.forward(xs[l])
        torch.cuda.synchronize()
        assert L.read_status() == 0, f"device status {L.read_status():#x}"
        U.append(int((L.counts > 0).sum().item()))
    R = cfg.T * cfg.k
    H, I, E = cfg.H, cfg.I, cfg.E
    gu_w_bytes = 2 * I * H * 2          # gate + up rows of one expert, bf16
    dn_w_bytes = H * I * 2
    router_bytes = E * H * 2

    def gateup_bytes(u):
        return u * gu_w_bytes + R * H * 2 + R * I * 2

    def fused_bytes(u):
        # both components of the distinct experts + token rows + h out and back
        # + y out (fp32, or bf16 rows already weighted) (+ the row gather's
        # token reads and row writes when the launch gathers)
        b = u * (gu_w_bytes + dn_w_bytes) + R * H * 2 + 2 * R * I * 2 + R * H * (2 if weighted else 4)
        return b + (cfg.T * H * 2 + R * H * 2 if gather_in_fused else 0)

    def layer_bytes(u):
        # distinct experts' weights + router + x in + out + route labels
        return u * (gu_w_bytes + dn_w_bytes) + router_bytes + 2 * cfg.T * H * 2 + R * 8

    K = args.steps
    # the host-side argument lists of every layer's calls, built before the
    # timed region
    bound = [layers[l].bound_calls(xs[l], cfg.T, stream=st) for l in range(NL)]
    names = [c[0] for c in bound[0]]
    weighted = "moe_expert_swiglu_fused_weighted" in names
    fused = "moe_expert_swiglu_fused" in names or weighted
    # kernels each boundary call launches in this configuration
    launches_per_step = sum(call_launches(c) for c in bound[0])
    gather_in_fused = fused and R <= MoELayer.GATHER_IN_FUSED_MAX_ROWS
    # the dominant kernel(s): the fused contraction, or gate/up then down
    i_main = names.index("moe_expert_swiglu_fused_weighted" if weighted else
                         "moe_expert_swiglu_fused" if fused else "moe_expert_gateup")
    issue = MoELayer.issue
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_uuid(local))
    time.sleep(0.3)
    # the W warm-up steps, right before the timed ones (after the sampler's
    # start, so that the clocks are up when the timed region begins)
    for i in range(max(args.warmup, 3)):
        for c in bound[i % NL]:
            issue(c)
    torch.cuda.synchronize()

    # Headline: K whole steps with nothing between the kernels (an event
    # between two kernels would end the overlap that programmatic dependent
    # launch gives the next one), bracketed by two events.
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    t_issue0 = time.perf_counter()
    e_start.record(st)
    for i in range(K):
        for c in bound[i % NL]:
            issue(c)
    e_end.record(st)
    t_issue1 = time.perf_counter()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    sampler.stop()

    # Instrumented pass, after the headline region: the same steps with
    # events around the dominant launch(es) of every step, to time that
    # kernel alone.  Its prologue then no longer overlaps the previous
    # kernel, so this launch time is an upper bound of the one inside the
    # headline steps.
    KE = min(max(K, 64), 2000)
    ev_g0 = [torch.cuda.Event(enable_timing=True) for _ in range(KE)]
    ev_g1 = [torch.cuda.Event(enable_timing=True) for _ in range(KE)]
    ev_d1 = [torch.cuda.Event(enable_timing=True) for _ in range(KE)]
    EV_EVERY = 1
    for j in range(KE):
        calls = bound[j % NL]
        for c in calls[:i_main]:
            issue(c)
        ev_g0[j].record(st)
        issue(calls[i_main])
        ev_g1[j].record(st)
        if not fused:
            issue(calls[i_main + 1])
        ev_d1[j].record(st)
        for c in calls[i_main + (1 if fused else 2):]:
            issue(c)
    torch.cuda.synchronize()

    total_ms = max_over_ranks(e_start.elapsed_time(e_end), world, dev)
    gu_ms = [ev_g0[j].elapsed_time(ev_g1[j]) for j in range(KE)]
    dn_ms = [ev_g1[j].elapsed_time(ev_d1[j]) for j in range(KE)]
    gu_avg = sum(gu_ms) / KE
    dn_avg = sum(dn_ms) / KE
    for L in layers:
        assert L.read_status() == 0, f"device status {L.read_status():#x}"

    value = whole_job_rate(cfg.T * K, total_ms / 1e3, world)
    pk = peaks()
    U_steps = [U[i % NL] for i in range(K)]
    main_bytes = fused_bytes if fused else gateup_bytes
    gu_bytes_avg = sum(main_bytes(U[(j * EV_EVERY) % NL]) for j in range(KE)) / KE
    layer_bytes_avg = sum(layer_bytes(u) for u in U_steps) / K
    achieved = gu_bytes_avg / (gu_avg / 1e3) / 1e9
    # the dominant launch's dense FLOPs (padding rows excluded): gate/up, and
    # down when the launch is fused
    main_flops = 2 * R * 2 * I * H + (2 * R * H * I if fused else 0)
    main_tflops = main_flops / (gu_avg / 1e3) / 1e12
    step_ms = total_ms / K
    flops_step = 2 * R * 3 * H * I + 2 * cfg.T * H * E

    clocks = sampler.summary(t_wall0, t_wall1)

    # e2e: host buffers in, host result out, through the public layer call
    e2e = None
    if not args.no_e2e:
        x_host = [xs[l].cpu().pin_memory() for l in range(NL)]
        out_host = [torch.empty((cfg.T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        Ke = max(10, min(K, 2000))
        for i in range(max(3, NL)):
            for o in out_host:
                layers[i % NL].forward_host_graph(x_host[i % NL], o)
        torch.cuda.synchronize()
        # synchronous calls: each returns once its result is in host memory
        t0 = time.perf_counter()
        for i in range(Ke):
            layers[i % NL].forward_host_graph(x_host[i % NL], out_host[0])
        el_sync = max_over_ranks(time.perf_counter() - t0, world, dev)
        # two calls in flight: step i is queued before the wait for step i - 1,
        # whose result (in its own pinned buffer) is then in host memory
        def in_flight(submit):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            prev = None
            for i in range(Ke):
                done = submit(layers[i % NL], x_host[i % NL], out_host[i % 2])
                if prev is not None:
                    MoELayer.wait(prev)
                prev = done
            MoELayer.wait(prev)
            return max_over_ranks(time.perf_counter() - t0, world, dev)

        el_graph = in_flight(lambda L, xh, oh: L.forward_host_submit(xh, oh))
        for i in range(max(3, 2 * NL)):  # the pipelined path's graphs are captured on first use
            MoELayer.wait(layers[i % NL].forward_host_pipelined(x_host[i % NL], out_host[i % 2]))
        el = in_flight(lambda L, xh, oh: L.forward_host_pipelined(xh, oh))
        e2e_val = whole_job_rate(cfg.T * Ke, el, world)
        e2e = {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": cfg.T * H * 2,
               "d2h_bytes_per_step": cfg.T * H * 2, "steps": Ke,
               "value_one_call_at_a_time": whole_job_rate(cfg.T * Ke, el_sync, world),
               "value_copies_in_the_graph": whole_job_rate(cfg.T * Ke, el_graph, world),
               "path": "MoELayer.forward_host_pipelined / MoELayer.wait: pinned x in, result out; the input copy "
                       "on a copy stream, the layer's launches as one CUDA graph, the result copy on a second "
                       "copy stream; two calls in flight, each step's result waited for in host memory"}

    cpu = None
    if host_w is not None:
        xs_bits = [np.ascontiguousarray(xs[0].cpu().view(torch.int16).numpy().view(np.uint16))]
        v, threads, ntok, el = oracle_tokens_per_s(cfg, host_w, xs_bits, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{ntok} tokens ({ntok // cfg.T} repeats of one {cfg.T}-token block of layer 0) in "
                         f"{el:.1f} s; fp64 C oracle, OpenMP"}

    wl_name = workload_name(cfg)
    U_ev = sum(U[(j * EV_EVERY) % NL] for j in range(KE)) / KE
    traffic = recorded_traffic("fused" if fused else "gateup", wl_name, U_ev)
    main_kernel = ("grouped_swiglu_fused_kernel (" +
                   ("moe_expert_swiglu_fused_weighted: " if weighted else "moe_expert_swiglu_fused: ") +
                   ("row gather, " if gather_in_fused else "") + "gate/up + SwiGLU, down" +
                   (", route-weighted bf16 outputs)" if weighted else ")")
                   if fused else "grouped_gemm_kernel (moe_expert_gateup)")
    roof_hbm = {"bound": "hbm", "kernel": main_kernel,
                "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                "traffic": traffic, "peak_source": pk["source"] + " hbm_gbs",
                "bytes_per_launch": gu_bytes_avg, "avg_launch_us": gu_avg * 1e3, "timed_launches": KE}
    # a launch of several ms inside the step: the sustained bf16 figure
    roof_tensor = {"bound": "tensor", "kernel": main_kernel,
                   "achieved": main_tflops, "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s",
                   "frac": main_tflops / pk["bf16_tflops_sustained"],
                   "frac_of_nominal": main_tflops / NOMINAL_BF16_TFLOPS, "traffic": traffic,
                   "peak_source": pk["source"] + " bf16_tflops_sustained",
                   "flops_per_launch": main_flops, "avg_launch_us": gu_avg * 1e3, "timed_launches": KE}
    # the bound is whichever the launch's arithmetic intensity puts it under
    intensity = main_flops / gu_bytes_avg
    ridge = pk["bf16_tflops_sustained"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    roof_main, roof_other = (roof_tensor, roof_hbm) if intensity > ridge else (roof_hbm, roof_tensor)
    roof_main["flop_per_byte"] = intensity
    roof_main["ridge_flop_per_byte"] = ridge
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded; x~N(0,1), weights~N(0,0.02) bf16)",
        "config": layer_config(cfg, NL, world, args.plain),
        "unique_experts_per_step": U,
        "roofline": roof_main, "roofline_other": roof_other,
        "layer_roofline": {"bytes_per_step": layer_bytes_avg,
                           "achieved_gbs": layer_bytes_avg / (step_ms / 1e3) / 1e9,
                           "frac_hbm": layer_bytes_avg / (step_ms / 1e3) / 1e9 / pk["hbm_gbs"],
                           "frac_hbm_of_nominal": layer_bytes_avg / (step_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                           "tflops": flops_step / (step_ms / 1e3) / 1e12,
                           "frac_tensor": flops_step / (step_ms / 1e3) / 1e12 / pk["bf16_tflops_sustained"],
                           "frac_tensor_of_nominal": flops_step / (step_ms / 1e3) / 1e12 / NOMINAL_BF16_TFLOPS,
                           **({} if fused else {"down_avg_us": dn_avg * 1e3})},
        "host_issue_us_per_step": 1e6 * (t_issue1 - t_issue0) / K,
        "dominant_kernel_timing": f"separate pass of {KE} steps after the headline region, events around "
                                  f"the dominant launch of every step; the headline steps carry no events",
        "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        # route: logits + selection; permute (+ row gather unless the fused
        # launch gathers); experts (fused: one launch; else gate/up, down, combine)
        "gpu_launches": launches_per_step * K,
    }
    return line


def run_stack(args, rank, world, local, dev, emit=True, with_sweep=False):
    """48-layer int4 g64 residual stack over 32 decode blocks of 16 tokens
    (stack48), or the route-prediction / dedup sweep over it (sweep)."""
    import torch
    import torch.distributed as dist
    import workloads as wl
    from sparse_moe_routed_gb300 import MoELayer, MoEStack, _lib, pack_layer_experts
    from sparse_moe_routed_gb300.sweep import route_sweep

    cfg = wl.STACK48
    L = args.layers or wl.STACK_LAYERS
    NB = wl.STACK_BLOCKS
    sweep_too = args.config == "sweep" or with_sweep
    T = NB * cfg.T if sweep_too else cfg.T  # layers sized for the sweep's 512 tokens serve 16-token blocks too
    mls = []
    for l in range(L):
        w = wl.stack_layer_weights(l, dev)
        gu, dn = pack_layer_experts(w["w_gateup_q"], w["w_down_q"], _lib.MOE_W_INT4_G64, cfg.E, cfg.H, cfg.I,
                                    s_gateup=w["s_gateup"], s_down=w["s_down"])
        mls.append(MoELayer(w["w_router"], None, gu, dn, cfg.k, T, fmt=_lib.MOE_W_INT4_G64_TILED, I=cfg.I))
        del w
    stack = MoEStack(mls, T)
    torch.cuda.synchronize()
    pk = peaks()
    st = torch.cuda.current_stream()
    rec_bytes = 2 * cfg.I * cfg.H // 2 + cfg.H * cfg.I // 2 + (2 * cfg.I * cfg.H // 64 + cfg.H * cfg.I // 64) * 2
    router_bytes = cfg.E * cfg.H * 2

    T_sweep = T

    def sweep_line():
        T = T_sweep
        preds = [wl.predictor_weights(cfg.H, cfg.E, l, dev) for l in range(L)]
        x0 = torch.cat([wl.token_batch(cfg, dev, index=b, T=cfg.T) for b in range(NB)]).float()
        for _ in range(max(args.warmup, 1)):
            route_sweep(stack, x0, preds)
        torch.cuda.synchronize()
        reps = max(1, min(args.steps, 5))
        t0 = time.perf_counter()
        for _ in range(reps):
            res = route_sweep(stack, x0, preds)
        el = (time.perf_counter() - t0) / reps
        line = {"metric": METRIC, "value": T / el, "unit": UNIT, "n_gpus": world, "steps": reps,
                "warmup": args.warmup, "ms_per_step": 1e3 * el, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "int4 g64 experts, bf16 router", "data": "synthetic",
                "config": {"workload": f"route_sweep_L{L}_T{T}_blocks1-4-16-64", "layers": L, "tokens": T},
                "sweep": res["summary"], "device_status": res["status"]}
        return line

    if args.config == "sweep":
        line = sweep_line()
        if rank == 0 and emit:
            print(json.dumps(line), flush=True)
        return 0 if emit else {"sweep": line}

    T = cfg.T  # stack48: blocks of 16 tokens
    xs = [wl.token_batch(cfg, dev, index=b, T=T).float() for b in range(NB)]
    xw = torch.empty_like(xs[0])
    # unique experts per layer of one block (for the byte accounting)
    xw.copy_(xs[0])
    Ul = []
    for l in range(L):
        for call in stack.layer_calls(xw, l):
            MoELayer.issue(call)
        torch.cuda.synchronize()
        Ul.append(int((stack.layers[l].counts > 0).sum().item()))
    bytes_block = sum(u * rec_bytes for u in Ul) + L * router_bytes
    K = args.steps
    # every layer's calls on the fixed stream buffer, built before the timed region
    lcalls = [stack.layer_calls(xw, l, stream=st) for l in range(L)]
    launches_per_block = sum(call_launches(c) for l in range(L) for c in lcalls[l])
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_uuid(local))
    time.sleep(0.3)
    # the W warm-up blocks, right before the timed ones
    for i in range(max(args.warmup, 3)):
        xw.copy_(xs[i % NB])
        for l in range(L):
            for c in lcalls[l]:
                MoELayer.issue(c)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    tw0 = time.time()
    # headline: K blocks through all L layers, no events between the kernels
    e0.record(st)
    for i in range(K):
        xw.copy_(xs[i % NB])
        for l in range(L):
            for c in lcalls[l]:
                MoELayer.issue(c)
    e1.record(st)
    torch.cuda.synchronize()
    tw1 = time.time()
    sampler.stop()
    total_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    for ml in stack.layers:
        assert ml.read_status() == 0, f"device status {ml.read_status():#x}"
    # instrumented pass after the headline region: events around one layer's
    # gate/up launch per block, the layer rotating over the stack
    KE = min(max(K, 2 * L), 4 * L)
    EV = 1
    g0 = [torch.cuda.Event(enable_timing=True) for _ in range(KE)]
    g1 = [torch.cuda.Event(enable_timing=True) for _ in range(KE)]
    for i in range(KE):
        xw.copy_(xs[i % NB])
        lt = i % L
        for l in range(L):
            calls = lcalls[l]
            if l == lt:
                for c in calls[:3]:
                    MoELayer.issue(c)
                g0[i].record(st)
                MoELayer.issue(calls[3])
                g1[i].record(st)
                for c in calls[4:]:
                    MoELayer.issue(c)
            else:
                for c in calls:
                    MoELayer.issue(c)
    torch.cuda.synchronize()
    gu = [g0[j].elapsed_time(g1[j]) for j in range(KE)]
    gu_avg = sum(gu) / KE
    R = T * cfg.k
    # decode-sized blocks (routes <= 320, K <= 2560) run on the CUDA-core int4 kernel
    cuda_core_int4 = R <= 320 and cfg.H <= 2560
    gu_bytes = sum((Ul[(j * EV) % L] * (2 * cfg.I * cfg.H // 2 + 2 * cfg.I * cfg.H // 64 * 2) + R * cfg.H * 2 +
                    R * cfg.I * 2) for j in range(KE)) / KE
    step_ms = total_ms / K
    line = {"metric": METRIC, "value": whole_job_rate(T * K, total_ms / 1e3, world), "unit": UNIT, "n_gpus": world,
            "steps": K,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": ("int4 g64 experts (codes expanded to bf16 pairs in registers, warp-level bf16 MMA, fp32 "
                      "accumulation), bf16 router, fp32 residual" if cuda_core_int4 else
                      "int4 g64 experts (bf16 tensor-core operands), bf16 router, fp32 residual"),
            "data": "synthetic (seeded)",
            "config": {"workload": f"stack48_int4g64_L{L}_T{T}_blocks{NB}", "layers": L, "T": T, "blocks": NB,
                       "unique_experts_per_layer_block0": Ul,
                       "l2": f"inputs larger than L2: {L} layers of int4 experts "
                             f"({L * (cfg.E * rec_bytes + router_bytes) / 1e9:.1f} GB) streamed per block"},
            "roofline": {"bound": "hbm",
                         "kernel": "gemv_q4_kernel (moe_expert_gateup, warp-level MMA)" if cuda_core_int4 else
                                   "grouped_gemm_q4_kernel (moe_expert_gateup, tcgen05)",
                         "achieved": gu_bytes / (gu_avg / 1e3) / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gu_bytes / (gu_avg / 1e3) / 1e9 / pk["hbm_gbs"],
                         "frac_of_nominal": gu_bytes / (gu_avg / 1e3) / 1e9 / NOMINAL_HBM_GBS, "traffic": None,
                         "bytes_per_launch": gu_bytes, "avg_launch_us": gu_avg * 1e3},
            "layer_roofline": {"bytes_per_block": bytes_block,
                               "achieved_gbs": bytes_block / (step_ms / 1e3) / 1e9,
                               "frac_hbm": bytes_block / (step_ms / 1e3) / 1e9 / pk["hbm_gbs"],
                               "frac_hbm_of_nominal": bytes_block / (step_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS},
            # per layer: RMSNorm 1, route 2 (logits, selection), grouping 2
            # (grouping, row gather), gate/up 1, down 1, combine 1
            "clocks": sampler.summary(tw0, tw1), "gpu_launches": launches_per_block * K}
    if emit:
        if rank == 0:
            print(json.dumps(line), flush=True)
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0
    out = {"stack48": line}
    if with_sweep:
        out["sweep"] = sweep_line()
    return out


def run_offload(args, rank, world, local, dev):
    """Decode blocks with the expert records in host memory behind S HBM slots.

    Every pass runs the same sequence of token blocks from the same cache
    state, so the cached passes see the same hits and misses:
      resident    MoELayer with the records in HBM;
      all-hit     the cached layer with every expert already in a slot (its
                  compute-only time, cache bookkeeping included);
    and for each slot count S, from an empty cache:
      copy-first  moe_cache_fetch timed on its own (the I/O wall time of the
                  misses), then the contraction;
      wave W      the in-launch fetch with wave width W.
    hidden fraction = 1 - (wave step time - all-hit step time) / fetch time:
    the exposed part of the I/O is what the wave path takes beyond compute.
    """
    import torch
    import workloads as wl
    from sparse_moe_routed_gb300 import CachedMoELayer, MoELayer, _lib, pack_layer_experts

    cfg = wl.DECODE
    if args.experts:
        from dataclasses import replace
        cfg = replace(cfg, E=args.experts)
    E, H, I, T = cfg.E, cfg.H, cfg.I, cfg.T
    slots = [int(v) for v in str(args.slots).split(",")]
    d = wl.layer_inputs(cfg, dev, with_x=False)
    q4 = args.int4
    fmt = _lib.MOE_W_INT4_G64_TILED if q4 else _lib.MOE_W_BF16_TILED
    if q4:
        q_gu, s_gu = wl.quantize_int4_g64(d["w_gateup"])
        q_d, s_d = wl.quantize_int4_g64(d["w_down"])
        gu, dn = pack_layer_experts(q_gu, q_d, _lib.MOE_W_INT4_G64, E, H, I, s_gateup=s_gu, s_down=s_d)
        del q_gu, s_gu, q_d, s_d
    else:
        gu, dn = pack_layer_experts(d["w_gateup"], d["w_down"], _lib.MOE_W_BF16, E, H, I)
    del d["w_gateup"], d["w_down"]
    hgu = torch.empty(gu.shape, dtype=torch.uint8, pin_memory=True)
    hdn = torch.empty(dn.shape, dtype=torch.uint8, pin_memory=True)
    hgu.copy_(gu)
    hdn.copy_(dn)
    torch.cuda.synchronize()
    rg, rd = hgu.numel() // E, hdn.numel() // E
    rec = rg + rd
    NB = 64
    xs = [wl.token_batch(cfg, dev, index=b, T=T) for b in range(NB)]
    st = torch.cuda.current_stream()
    K = max(args.steps, 16) if args.steps < 20000 else 256
    W0 = max(args.warmup, 3)
    resident = MoELayer(d["w_router"], d["bias"], gu, dn, cfg.k, T, fmt=fmt, I=I)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    # link bandwidth: a copy-engine copy of 1 GiB pinned -> device, and the
    # fetch kernel copying whole records alone
    nb = min(hgu.numel(), 1 << 30)
    dst = torch.empty((nb,), dtype=torch.uint8, device=dev)
    for _ in range(2):
        dst.copy_(hgu[:nb], non_blocking=True)
    e0.record(st)
    for _ in range(5):
        dst.copy_(hgu[:nb], non_blocking=True)
    e1.record(st)
    torch.cuda.synchronize()
    ce_gbs = 5 * nb / (e0.elapsed_time(e1) / 1e3) / 1e9
    del dst

    # the all-hit layer: S = E slots, every expert in slot e
    full = CachedMoELayer(d["w_router"], d["bias"], hgu, hdn, cfg.k, T, I=I, S=E, fmt=fmt)
    ar = torch.arange(E, dtype=torch.int32, device=dev)
    stt = torch.tensor([0, E, 0, 0], dtype=torch.int32, device=dev)
    _lib.moe_cache_fetch(hgu, hdn, rg, rd, ar, ar, stt, full.pool_gu, full.pool_dn)
    nf = min(E, 96)
    stt[1] = nf
    e0.record(st)
    for _ in range(5):
        _lib.moe_cache_fetch(hgu, hdn, rg, rd, ar, ar, stt, full.pool_gu, full.pool_dn)
    e1.record(st)
    full.slot_of.copy_(ar)
    full.expert_of.copy_(ar)
    torch.cuda.synchronize()
    fetch_gbs = 5 * nf * rec / (e0.elapsed_time(e1) / 1e3) / 1e9

    def timed(layer, fetch_events=False):
        for i in range(W0):
            layer.forward(xs[i % NB])
        torch.cuda.synchronize()
        if isinstance(layer, CachedMoELayer):
            layer.stats[2:].zero_()
        f0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        f1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for i in range(K):
            for c in layer.bound_calls(xs[(W0 + i) % NB], T, stream=st):
                if fetch_events and c[0] == "moe_cache_fetch":
                    f0[i].record(st)
                    MoELayer.issue(c)
                    f1[i].record(st)
                else:
                    MoELayer.issue(c)
        b.record(st)
        torch.cuda.synchronize()
        assert layer.read_status() == 0, f"device status {layer.read_status():#x}"
        io = sum(f0[i].elapsed_time(f1[i]) for i in range(K)) / K if fetch_events else None
        return a.elapsed_time(b) / K, io

    sampler = ClockSampler(gpu_uuid(local))
    time.sleep(0.3)
    tw0 = time.time()
    res_ms, _ = timed(resident)
    hit_ms, _ = timed(full)
    assert int(full.stats[3].item()) == 0
    del full
    by_slots = {}
    for S in slots:
        bar = CachedMoELayer(d["w_router"], d["bias"], hgu, hdn, cfg.k, T, I=I, S=S, fetch="barrier",
                             policy=args.policy, decay=args.decay, fmt=fmt)
        bar_ms, io_ms = timed(bar, fetch_events=True)
        hits, misses = [int(v) for v in bar.stats[2:].cpu().tolist()]
        del bar
        waves = {}
        # int4 records: the gate/up launch fetches every miss (gate/up pieces
        # first, then down): one in-launch variant, width "all"
        for w in ([0] if q4 else [int(v) for v in args.waves.split(",")]):
            lay = CachedMoELayer(d["w_router"], d["bias"], hgu, hdn, cfg.k, T, I=I, S=S,
                                 wave=w if w > 0 else 1 << 20, policy=args.policy, decay=args.decay, fmt=fmt)
            ms_w, _ = timed(lay)
            assert tuple(int(v) for v in lay.stats[2:].cpu().tolist()) == (hits, misses), "passes differ"
            del lay
            waves["all" if w <= 0 else str(w)] = {
                "tokens_per_s": T / (ms_w / 1e3), "ms_per_step": ms_w,
                "hidden_fraction": (1.0 - (ms_w - hit_ms) / io_ms) if io_ms > 0 else None}
        fetched = misses * rec / K
        best = max(waves.values(), key=lambda v: v["tokens_per_s"])
        by_slots[str(S)] = {
            "hit_rate": hits / max(hits + misses, 1), "misses_per_step": misses / K,
            "fetched_bytes_per_token": fetched / T,
            "copy_first": {"ms_per_step": bar_ms, "tokens_per_s": T / (bar_ms / 1e3), "fetch_ms_per_step": io_ms,
                           "fetch_gbs": fetched / (io_ms / 1e3) / 1e9 if io_ms else None},
            "waves": waves, "best_tokens_per_s": best["tokens_per_s"],
            "link_gbs_during_best": fetched / (best["ms_per_step"] / 1e3) / 1e9}
    tw1 = time.time()
    sampler.stop()
    head = by_slots[str(slots[0])]
    line = {
        "metric": METRIC, "value": head["best_tokens_per_s"], "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W0, "ms_per_step": T / head["best_tokens_per_s"] * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int4 g64 experts, bf16 router" if q4 else "bf16",
        "data": "synthetic (seeded; 64 independent token blocks in turn)",
        "config": {"workload": f"offload_{workload_name(cfg)}{'_int4' if q4 else ''}_S{slots[0]}", "slots": slots,
                   "T": T, "E": E,
                   "records": f"tile-packed {'int4 g64' if q4 else 'bf16'} in pinned host memory; HBM slot cache, "
                              f"{args.policy} replacement",
                   "policy": args.policy, "decay": args.decay, "record_bytes": rec},
        "resident": {"ms_per_step": res_ms, "tokens_per_s": T / (res_ms / 1e3)},
        "all_hit": {"ms_per_step": hit_ms, "tokens_per_s": T / (hit_ms / 1e3)},
        "by_slots": by_slots,
        "link": {"copy_engine_h2d_gbs": ce_gbs, "fetch_kernel_gbs": fetch_gbs,
                 "fetch_kernel_sample": f"{nf} experts' records, kernel alone"},
        "roofline": {"bound": "link", "kernel": "moe_cache_fetch (cache_fetch_kernel), alone",
                     "achieved": fetch_gbs, "peak": ce_gbs, "unit": "GB/s", "frac": fetch_gbs / ce_gbs,
                     "traffic": None, "peak_source": "copy-engine host-to-device copy measured in this run"},
        "clocks": sampler.summary(tw0, tw1),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_trace(args, rank, world, local, dev):
    """Route traces through the cache plan, and merged multi-request calls.

    Traces: NB decode blocks (T = 16) of each of 8 seeded layers (their own
    router weights and Zipf bias), routed by moe_route.  Two token-block
    recipes: independent blocks (x ~ N(0,1) each), and a random walk
    x_{b+1} = rho x_b + sqrt(1 - rho^2) z (rho = 0.9) whose neighbouring
    blocks share experts.  Each (recipe, policy, slot count) replays the
    blocks in order through moe_cache_plan, one cache per layer, from empty.
    Merge: R independent requests' blocks grouped into one layer call of
    16 R tokens, against R calls of 16 tokens (records in HBM).
    """
    import torch
    import workloads as wl
    from sparse_moe_routed_gb300 import MoELayer, _lib, pack_layer_experts

    cfg = wl.DECODE
    E, H, I, T, k = cfg.E, cfg.H, cfg.I, cfg.T, cfg.k
    NL, NB = 8, 256
    rec = 3 * H * I * 2
    st = torch.cuda.current_stream()
    routers = []
    for l in range(NL):
        routers.append(wl.router_inputs(cfg, dev, layer=l))
    g = torch.Generator(device=dev)
    g.manual_seed(cfg.seed * 1_000_003 + 77)

    def blocks(rho):
        x = torch.randn((T, H), generator=g, device=dev)
        out = []
        for _ in range(NB):
            out.append(x.to(torch.bfloat16))
            x = rho * x + (1 - rho * rho) ** 0.5 * torch.randn((T, H), generator=g, device=dev)
        return out

    ws = torch.empty((_lib.route_workspace_size(T, E),), dtype=torch.uint8, device=dev)

    def trace(xs):
        cnt = torch.zeros((NL, NB, E), dtype=torch.int32, device=dev)
        ids = torch.empty((T, k), dtype=torch.int32, device=dev)
        w = torch.empty((T, k), dtype=torch.float32, device=dev)
        for l, (wr, b) in enumerate(routers):
            for bi, x in enumerate(xs):
                _lib.moe_route(x, wr, b, k, ids, w, None, ws)
                cnt[l, bi].index_add_(0, ids.flatten().long(), torch.ones(T * k, dtype=torch.int32, device=dev))
        return cnt

    pols = {"fifo": _lib.MOE_CACHE_FIFO, "lru": _lib.MOE_CACHE_LRU, "score": _lib.MOE_CACHE_SCORE}
    slots = [160, 192, 256, 320]
    result = {}
    t0 = time.perf_counter()
    for recipe, rho in (("independent", 0.0), ("walk_rho0.9", 0.9)):
        cnt = trace(blocks(rho))
        routed = (cnt > 0)
        uniq = routed.sum(-1).float()
        overlap = (routed[:, 1:] & routed[:, :-1]).sum(-1).float() / uniq[:, 1:]
        r = {"unique_experts_per_block": float(uniq.mean()), "overlap_with_previous_block": float(overlap.mean())}
        for pol, pid in pols.items():
            for S in slots:
                hits = misses = 0
                for l in range(NL):
                    so = torch.full((E,), -1, dtype=torch.int32, device=dev)
                    eo = torch.full((S,), -1, dtype=torch.int32, device=dev)
                    hand = torch.zeros((2,), dtype=torch.int32, device=dev)
                    sc = torch.zeros((E,), dtype=torch.float32, device=dev)
                    lu = torch.full((S,), -1, dtype=torch.int32, device=dev)
                    ml = torch.empty((S,), dtype=torch.int32, device=dev)
                    msl = torch.empty((S,), dtype=torch.int32, device=dev)
                    stt = torch.zeros((4,), dtype=torch.int32, device=dev)
                    sw = torch.zeros((1,), dtype=torch.int32, device=dev)
                    for bi in range(NB):
                        _lib.moe_cache_plan(cnt[l, bi], so, eo, hand, ml, msl, stt, sw, policy=pid,
                                            decay=args.decay, score=sc, last_use=lu)
                    torch.cuda.synchronize()
                    assert int(sw.item()) == 0
                    hits += int(stt[2].item())
                    misses += int(stt[3].item())
                r[f"{pol}_S{S}"] = {"hit_rate": hits / (hits + misses),
                                    "fetched_bytes_per_token": misses * rec / (NL * NB * T)}
        result[recipe] = r
    sim_s = time.perf_counter() - t0

    # merged multi-request calls vs one call per request (records in HBM)
    d = wl.layer_inputs(cfg, dev, with_x=False)
    gu, dn = pack_layer_experts(d["w_gateup"], d["w_down"], _lib.MOE_W_BF16, E, H, I)
    del d["w_gateup"], d["w_down"]
    xs = [wl.token_batch(cfg, dev, index=b, T=T) for b in range(64)]
    merge = {}
    for R in (1, 2, 4, 8):
        lay = MoELayer(d["w_router"], d["bias"], gu, dn, k, T * R, fmt=_lib.MOE_W_BF16_TILED, I=I)
        xm = [torch.cat(xs[i * R:(i + 1) * R]) for i in range(64 // R)]
        single = MoELayer(d["w_router"], d["bias"], gu, dn, k, T, fmt=_lib.MOE_W_BF16_TILED, I=I)
        K = 64 // R * 4

        def run(fn, n):
            for i in range(3):
                fn(i)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            for i in range(n):
                fn(i)
            b.record(st)
            torch.cuda.synchronize()
            return a.elapsed_time(b) / n

        ms_merged = run(lambda i: lay.forward(xm[i % len(xm)]), K)
        ms_sep = run(lambda i: [single.forward(xs[(i % len(xm)) * R + j]) for j in range(R)], K)
        u = []
        for i in range(len(xm)):
            lay.forward(xm[i])
            torch.cuda.synchronize()
            u.append(int((lay.counts > 0).sum().item()))
        assert lay.read_status() == 0 and single.read_status() == 0
        merge[str(R)] = {"tokens_per_s_merged": T * R / (ms_merged / 1e3),
                         "tokens_per_s_separate": T * R / (ms_sep / 1e3),
                         "unique_experts_per_call": sum(u) / len(u),
                         "record_bytes_per_token_merged": sum(u) / len(u) * rec / (T * R)}
    best = max(merge.values(), key=lambda v: v["tokens_per_s_merged"])
    line = {"metric": METRIC, "value": best["tokens_per_s_merged"], "unit": UNIT, "n_gpus": world,
            "steps": None, "warmup": 3, "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded route traces)",
            "config": {"workload": f"trace_{workload_name(cfg)}_L{NL}_B{NB}", "layers": NL, "blocks": NB,
                       "slots": slots, "decay": args.decay, "record_bytes": rec},
            "cache_simulation": result, "simulation_seconds": sim_s, "merge": merge}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_crossover(args, rank, world, local, dev):
    """Selected records against the whole layer, and the two-layer ring.

    For T in 16 .. 4096 tokens of the uniform-router layer: U = distinct
    routed experts; t_selected = moe_cache_fetch of those U records from
    pinned host memory (SM copy warps); t_layer = moe_layer_stream of all E
    records (copy engines); t_compute = the layer with its records in HBM.
    t_selected is fitted as a + b U; the crossover is where it meets t_layer.
    Macro prefill: L layers (two host record sets in turn) at T = 4096
    through PrefillRing, against the same stack resident in HBM.
    """
    import numpy as np
    import torch
    import workloads as wl
    from sparse_moe_routed_gb300 import MoELayer, MoEStack, PrefillRing, _lib, pack_layer_experts

    cfg = wl.PREFILL
    E, H, I, k = cfg.E, cfg.H, cfg.I, cfg.k
    st = torch.cuda.current_stream()
    sets = []
    for l in range(2):
        d = wl.layer_inputs(cfg, dev, layer=l, with_x=False)
        gu, dn = pack_layer_experts(d["w_gateup"], d["w_down"], _lib.MOE_W_BF16, E, H, I)
        del d["w_gateup"], d["w_down"]
        hgu = torch.empty(gu.shape, dtype=torch.uint8, pin_memory=True)
        hdn = torch.empty(dn.shape, dtype=torch.uint8, pin_memory=True)
        hgu.copy_(gu)
        hdn.copy_(dn)
        torch.cuda.synchronize()
        sets.append({"wr": d["w_router"], "bias": d["bias"], "gu": gu, "dn": dn, "hgu": hgu, "hdn": hdn})
    s0 = sets[0]
    rg, rd = s0["hgu"].numel() // E, s0["hdn"].numel() // E
    rec = rg + rd
    pool_gu = torch.empty_like(s0["gu"])
    pool_dn = torch.empty_like(s0["dn"])
    ring_gu = torch.empty_like(s0["gu"])
    ring_dn = torch.empty_like(s0["dn"])

    def timed(fn, reps=5, warm=2):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(reps):
            fn()
        b.record(st)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps * 1e3  # microseconds

    t_layer = timed(lambda: _lib.moe_layer_stream(s0["hgu"], s0["hdn"], ring_gu, ring_dn))
    points = []
    for T in (16, 64, 256, 1024, 4096):
        lay = MoELayer(s0["wr"], s0["bias"], s0["gu"], s0["dn"], k, T, fmt=_lib.MOE_W_BF16_TILED, I=I)
        x = wl.token_batch(cfg, dev, index=T, T=T)
        t_comp = timed(lambda: lay.forward(x), reps=10)
        assert lay.read_status() == 0
        routed = torch.nonzero(lay.counts > 0).flatten().to(torch.int32)
        U = int(routed.numel())
        ms = torch.arange(U, dtype=torch.int32, device=dev)
        stt = torch.tensor([0, U, 0, 0], dtype=torch.int32, device=dev)
        t_sel = timed(lambda: _lib.moe_cache_fetch(s0["hgu"], s0["hdn"], rg, rd, routed, ms, stt, pool_gu, pool_dn))
        points.append({"T": T, "U": U, "unique_fraction": U / E, "t_selected_us": t_sel, "t_layer_us": t_layer,
                       "t_compute_us": t_comp, "selected_gbs": U * rec / t_sel / 1e3})
        del lay
    Us = np.array([p["U"] for p in points], float)
    ts = np.array([p["t_selected_us"] for p in points], float)
    b, a = np.polyfit(Us, ts, 1)
    u_star = (t_layer - a) / b / E
    sel_gbs = rec / b / 1e3
    layer_gbs = E * rec / t_layer / 1e3
    for p in points:
        p["mode"] = ["selected", "layer"][_lib.stream_mode(p["U"], E, rec, sel_gbs, layer_gbs, max(a, 0.0))[0]]

    # macro prefill through the ring, L layers, T = 4096
    L, T = 8, 4096
    routers = [(sets[l % 2]["wr"], sets[l % 2]["bias"]) for l in range(L)]
    host = [(sets[l % 2]["hgu"], sets[l % 2]["hdn"]) for l in range(L)]
    ring = PrefillRing(routers, host, k, T, I)
    res = MoEStack([MoELayer(sets[l % 2]["wr"], sets[l % 2]["bias"], sets[l % 2]["gu"], sets[l % 2]["dn"], k, T,
                             fmt=_lib.MOE_W_BF16_TILED, I=I) for l in range(L)], T)
    x0 = wl.token_batch(cfg, dev, index=7, T=T).float()
    xr = x0.clone()
    xs_ = x0.clone()
    sampler = ClockSampler(gpu_uuid(local))
    time.sleep(0.3)
    tw0 = time.time()
    t_ring = timed(lambda: ring.forward(xr), reps=3, warm=1)
    t_res = timed(lambda: res.forward(xs_), reps=3, warm=1)
    tw1 = time.time()
    sampler.stop()
    for ml in ring.stack.layers + res.layers:
        assert ml.read_status() == 0
    io = L * t_layer
    line = {"metric": METRIC, "value": T / (t_ring / 1e6), "unit": UNIT, "n_gpus": world, "steps": 3, "warmup": 1,
            "ms_per_step": t_ring / 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded; uniform router)",
            "config": {"workload": f"crossover_{workload_name(cfg)}", "record_bytes": rec,
                       "ring": f"{L} layers x {T} tokens, records in pinned host memory, two-layer HBM ring"},
            "points": points,
            "fit": {"selected_overhead_us": a, "selected_us_per_record": b, "selected_gbs": sel_gbs,
                    "layer_gbs": layer_gbs, "crossover_unique_fraction": u_star},
            "ring": {"layers": L, "T": T, "t_ring_ms": t_ring / 1e3, "t_resident_ms": t_res / 1e3,
                     "t_io_ms": io / 1e3, "hidden_fraction": 1.0 - (t_ring - t_res) / io,
                     "tokens_per_s_ring": T / (t_ring / 1e6), "tokens_per_s_resident": T / (t_res / 1e6)},
            "clocks": sampler.summary(tw0, tw1)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_sidecar(args, rank, world, local, dev):
    """Route-sidecar forward pass: T positions -> 48 layers x N candidates."""
    import torch
    import workloads as wl
    from sparse_moe_routed_gb300 import _lib

    F, r, E, L, N = 2560, 256, 512, 48, 16
    w = wl.sidecar_weights(F, r, E, L, dev)
    hb = torch.empty((L, E), dtype=torch.float32, device=dev)
    _lib.moe_sidecar_prepare(w["w_head"], w["layer_emb"], hb)
    st = torch.cuda.current_stream()
    pk = peaks()
    res = {}
    for T in (1, 16, 64, 256):
        NB = 64
        feats = [wl.token_batch(wl.DECODE, dev, index=b, T=T) for b in range(NB)]
        z = torch.empty((T, r), dtype=torch.float32, device=dev)
        cand = torch.empty((T, L, N), dtype=torch.int32, device=dev)
        cs = torch.empty((T, L, N), dtype=torch.float32, device=dev)
        sw = torch.zeros((1,), dtype=torch.int32, device=dev)
        K = max(args.steps, 16) if args.steps < 20000 else 2000
        for i in range(max(args.warmup, 3)):
            _lib.moe_sidecar_forward(feats[i % NB], w["w_trunk"], w["w_head"], hb, N, z, cand, cs, sw)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for i in range(K):
            _lib.moe_sidecar_forward(feats[i % NB], w["w_trunk"], w["w_head"], hb, N, z, cand, cs, sw)
        b.record(st)
        torch.cuda.synchronize()
        assert int(sw.item()) == 0
        us = a.elapsed_time(b) / K * 1e3
        byts = r * F * 2 + E * r * 2 + L * E * 4 + T * F * 2 + T * L * N * 8
        flops = 2 * T * (r * F + E * r) + T * L * E
        res[str(T)] = {"us_per_call": us, "positions_per_s": T / (us / 1e6),
                       "achieved_gbs": byts / (us / 1e6) / 1e9, "frac_hbm": byts / (us / 1e6) / 1e9 / pk["hbm_gbs"],
                       "tflops": flops / (us / 1e6) / 1e12, "bytes_per_call": byts}
    line = {"metric": METRIC, "value": res["16"]["positions_per_s"], "unit": "positions/s", "n_gpus": world,
            "steps": K, "warmup": max(args.warmup, 3), "ms_per_step": res["16"]["us_per_call"] / 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 weights, fp32",
            "data": "synthetic (seeded random sidecar weights)",
            "config": {"workload": f"sidecar_F{F}_r{r}_E{E}_L{L}_N{N}", "F": F, "r": r, "E": E, "L": L, "N": N},
            "by_positions": res,
            "roofline": {"bound": "hbm", "kernel": "router_logits_mma_kernel (trunk) + sidecar_head_kernel",
                         "achieved": res["16"]["achieved_gbs"], "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": res["16"]["frac_hbm"], "traffic": None,
                         "peak_source": pk["source"] + " hbm_gbs",
                         "note": "1.7 MB of weights per call: launch and round-trip latency bound"},
            "gpu_launches": 2 * K}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
