"""Benchmark of the MoE FFN layer forward on GB300.

One step = one moe_layer_forward over one batch of synthetic tokens: router,
top-k gating, dispatch, grouped SwiGLU GEMMs, combine.  Default workload: the
Qwen3-235B-A22B-shaped layer (H=4096, E=128, top-8, I=1536, softmax-then-top-k
renormalised, Zipf(1.1) routing skew) at T=1024 tokens per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--T T]
    python bench.py --impl reference ...     # the CPU oracle, timed on host cores

Prints one JSON line.  With N > 1 (torchrun) every rank runs an independent
replica on its own batch (weak scaling); ranks exchange only timings.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s at Qwen3-235B layer shape; % of HBM / bf16-TC roofline"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--config", default="qwen3")
    p.add_argument("--T", type=int, default=1024)
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--E", type=int, default=0,
                   help="override the number of experts (reduced cases for profiler captures)")
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-tokens", type=int, default=0,
                   help="tokens of the oracle's timed sample (0: sized from a short probe "
                        "to about 15 s of CPU work for the cpu_baseline, about 90 s over all "
                        "steps of --impl reference)")
    p.add_argument("--op", default="layer", choices=["layer", "reshard"],
                   help="layer: the MoE layer forward (default); reshard: the EP<->TP "
                        "expert-weight permute of one rank's experts")
    p.add_argument("--tp", type=int, default=8, help="--op reshard: ranks P of the switch")
    p.add_argument("--sweep", action="store_true",
                   help="time every layer configuration at each of its batch sizes, one JSON "
                        "line each (appended to --sweep-out)")
    p.add_argument("--sweep-out", default="",
                   help="--sweep: file the lines are appended to")
    p.add_argument("--sweep-configs", default="",
                   help="--sweep: comma-separated layer names to keep (default: all)")
    p.add_argument("--sweep-max-T", type=int, default=0,
                   help="--sweep: keep batch sizes up to this many tokens (default: all)")
    p.add_argument("--weights", default="bf16", choices=["bf16", "fp8"],
                   help="expert weight format: bf16, or E4M3 codes with a power-of-two scale "
                        "per 128x128 block (moe_layer_forward_fp8)")
    p.add_argument("--capacity-factor", type=float, default=0.0,
                   help="time moe_layer_forward_capacity with C = ceil(cf * T * k / E) "
                        "(0: the dropless layer)")
    p.add_argument("--path", default="auto", choices=["auto", "chain", "persistent", "chain1sm"],
                   help="execution path of the layer forward: automatic choice (default), "
                        "the kernel chain, the persistent single-kernel layer (T <= 16), or "
                        "the kernel chain with one-SM GEMM tiles only (no CTA-pair tiles for "
                        "prefill batches)")
    p.add_argument("--l2-flush", action="store_true",
                   help="write a 256 MB buffer before every timed step (each step then "
                        "timed alone); for layers whose working set fits in L2")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        return {"hbm_gbs": m["hbm_gbs"], "bf16_tflops": m["bf16_tflops"],
                "bf16_tflops_sustained": m.get("bf16_tflops_sustained", m["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def layer_config(args):
    import dataclasses

    import synth
    cfg = synth.CONFIGS[args.config]
    if args.E:
        cfg = dataclasses.replace(cfg, name=f"{cfg.name}_E{args.E}", E=args.E, k=min(cfg.k, args.E))
    return cfg


L2_BYTES = 129 << 20


def workload_config(cfg, T, l2_flush=False):
    weights = (cfg.E + (1 if cfg.shared else 0)) * 3 * cfg.H * cfg.I * 2
    if l2_flush:
        l2 = "L2 flushed before every step (256 MB write), each step timed alone"
    elif weights > L2_BYTES:
        l2 = ("inputs larger than L2 (the step streams the touched experts' weights, "
              f"{weights / 1e9:.2f} GB for all experts)")
    else:
        l2 = f"inputs smaller than L2 ({weights / 1e6:.1f} MB of weights), warm, no flush"
    return {"workload": f"{cfg.name} layer, T={T} tokens/step", "layer": cfg.name,
            "H": cfg.H, "E": cfg.E, "k": cfg.k, "I": cfg.I, "T": T,
            "gating": ["topk_softmax", "softmax_topk", "softmax_topk_renorm",
                       "sigmoid_bias_renorm"][cfg.gating],
            "shared_expert": cfg.shared, "routing_skew": str(cfg.skew), "l2": l2}


# ------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi samples (every 100 ms) taken while the timed region runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = [r for t, r in self.rows if t0 <= t <= t1 + 0.15]
        used = inside if inside else [r for _, r in self.rows]
        sm = [float(r[1]) for r in used if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in used if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in used for n, v in zip(names, r[5:9]) if v == "Active"})
        pw = [float(r[3]) for r in used if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w_max": max(pw) if pw else None,
                "samples": len(inside), "window": "timed region" if inside else "whole run"}


# ------------------------------------------------------ roofline model --

def expert_params(H, I):
    """Parameters of one SwiGLU expert: W_gate and W_up [I,H] and W_down [H,I]
    (Moebius reading notes eq. (2))."""
    return 3 * H * I


def expert_bytes(H, I, bytes_per_param=2):
    """Bytes one touched expert streams from HBM per forward (bf16: 2 B)."""
    return expert_params(H, I) * bytes_per_param


def expected_touched(E, k, n):
    """Expected number of experts a batch of n tokens touches when each token
    picks a uniform random k-subset of E: E * (1 - (1 - k/E)^n) (CS349D
    lecture 8 notes, section 2.1 "一批 token 会碰到几个专家")."""
    return E * (1.0 - (1.0 - k / E) ** n)


def tokens_per_expert(n, k, E):
    """Average rows per expert, n*k/E (CS349D lecture 8 notes, section 2.1)."""
    return n * k / E


def ridge_rows(peak_flops, hbm_bytes_per_s):
    """Rows per expert at which an expert GEMM turns compute-bound: its
    arithmetic intensity is about m_e flops per weight byte (2 flops per
    multiply-add over 2-byte weights), so the ridge is F/B (CS349D lecture 8
    notes, section 2.1, exercise 2)."""
    return peak_flops / hbm_bytes_per_s


def expert_gemm_utilisation(m_rows, peak_flops, hbm_bytes_per_s):
    """Fraction of the tensor peak an HBM-bound expert GEMM with m rows per
    expert can reach: min(1, m / ridge)."""
    return min(1.0, m_rows / ridge_rows(peak_flops, hbm_bytes_per_s))


def algorithmic(cfg, T, counts, weight_bytes=2):
    """Algorithmic bytes and flops of one step and of the gate/up GEMM
    (weight_bytes per expert weight: 2 for bf16, 1 for FP8 codes, whose block
    exponents add 1/16384)."""
    touched = int(sum(1 for c in counts if c > 0))
    H, I, E, k = cfg.H, cfg.I, cfg.E, cfg.k
    per_expert = expert_bytes(H, I, weight_bytes)
    if weight_bytes == 1:
        per_expert += -(-expert_params(H, I) // (128 * 128))
    nsh = 1 if cfg.shared else 0
    layer_bytes = (touched + nsh) * per_expert + E * H * 4 + 2 * T * H * 2
    layer_flops = 2 * T * k * 3 * H * I + nsh * 2 * T * 3 * H * I + 2 * T * H * E
    rows = T * k + nsh * T
    # the gate/up kernel reads each token row of x once from HBM (its k-fold
    # reuse is served by L2) and writes h
    gateup_bytes = (touched + nsh) * 2 * I * H * weight_bytes + T * H * 2 + rows * I * 2
    gateup_flops = 2 * rows * 2 * I * H
    return {"touched": touched, "layer_bytes": layer_bytes, "layer_flops": layer_flops,
            "gateup_bytes": gateup_bytes, "gateup_flops": gateup_flops}


# ------------------------------------------------------------ CPU oracle --

def cpu_oracle_sample(inputs_host, n_tokens, seed=0):
    """Time the oracle (routing + layer) on a seeded sample of n tokens."""
    import numpy as np

    import oracle
    cfg, T = inputs_host.cfg, inputs_host.T
    rng = np.random.default_rng(seed)
    toks = sorted(rng.choice(T, size=min(n_tokens, T), replace=False).tolist())
    x = inputs_host.x[toks].contiguous()
    threads = oracle.max_threads()
    t0 = time.perf_counter()
    s = oracle.router_logits(x, inputs_host.w_router, threads)
    ids, w, _ = oracle.topk_gating(s, cfg.k, cfg.gating, inputs_host.sel_bias)
    oracle.layer_tokens(x, ids, w, inputs_host.w13, inputs_host.w2, range(len(toks)),
                        inputs_host.w13_shared, inputs_host.w2_shared, threads)
    dt = time.perf_counter() - t0
    return len(toks), dt, threads


def host_inputs(cfg, T, seed, experts_from_gpu=None):
    """Host copy of a workload; expert blocks are copied lazily from the GPU
    tensors when given (only the experts the oracle reads are fetched)."""
    import synth

    class Lazy(dict):
        def __init__(self, src):
            super().__init__()
            self.src = src

        def __missing__(self, e):
            v = self.src[e].cpu()
            self[e] = v
            return v

        def keys(self):
            return range(self.src.shape[0])

    if experts_from_gpu is not None:
        g = experts_from_gpu
        return synth.LayerInputs(cfg, T, seed, g.x.cpu(), g.w_router.cpu(),
                                 None if g.sel_bias is None else g.sel_bias.cpu(),
                                 Lazy(g.w13), Lazy(g.w2),
                                 None if g.w13_shared is None else g.w13_shared.cpu(),
                                 None if g.w2_shared is None else g.w2_shared.cpu())
    return synth.make_layer(cfg, T, seed, device="cpu")


# ---------------------------------------------------------------- arms --

def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        pg = dist
    return world, rank, local, pg


def max_over_ranks(value: float, pg):
    if pg is None:
        return value
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def barrier(pg):
    if pg is not None:
        pg.barrier()


def run_reference(args):
    """The oracle as the reference arm: each step is a bounded token sample of
    the same workload, timed on the host cores."""
    import synth
    world, rank, local, pg = dist_setup(args)
    if rank != 0:
        return
    cfg = layer_config(args)
    T = args.T
    import torch
    if torch.cuda.is_available():
        # inputs are generated on the GPU (untimed); the oracle reads host copies
        gen = synth.make_layer(cfg, T, args.seed, device="cuda")
        inp = host_inputs(cfg, T, args.seed, experts_from_gpu=gen)
    else:
        inp = host_inputs(cfg, T, args.seed)
    # a short probe of the oracle's rate sizes the per-step sample (about 90 s
    # over all steps) unless --cpu-tokens fixes it
    k0, dt0, _ = cpu_oracle_sample(inp, min(16, T), seed=99)
    n = args.cpu_tokens if args.cpu_tokens > 0 else int(max(16, 90.0 * k0 / dt0 / max(1, args.steps)))
    n = min(n, T)
    total_tok, total_s, threads = 0, 0.0, 1
    for step in range(args.steps):
        k, dt, threads = cpu_oracle_sample(inp, n, seed=step)
        total_tok += k
        total_s += dt
    value = total_tok / total_s
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(cfg, T),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"{n} seeded tokens of the T={T} batch per step "
                                       "(routing + expert FFNs + combine, fp64)"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def new_events(stream, n):
    import torch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record(stream)  # materialise the handles
    return evs


PATHS = {"auto": None, "chain": 1, "persistent": 2, "chain1sm": 3}

# the persistent single-kernel layer's shapes (moe_layer_forward_ex)
DECODE_MAX_T = 16


def uses_persistent(cfg, T, path):
    """Whether a forward of this shape runs as the persistent decode layer."""
    fits = T <= DECODE_MAX_T and cfg.H >= 256
    return path == "persistent" or (path == "auto" and fits)


def pair_tiles(cfg, T, path):
    """Tiles of the chain's expert GEMMs: "cta_pair" (tcgen05.mma.cta_group::2)
    or "one_sm", by the library's rule -- gate/up on pairs from 256 rows per
    routed expert on average, down from 64 when I >= 2048 (else 256); H a
    multiple of 256, H and I of 128."""
    if path in ("persistent", "chain1sm") or uses_persistent(cfg, T, path):
        return {"gateup": "one_sm", "down": "one_sm"}
    shape_ok = cfg.H % 256 == 0 and cfg.I % 128 == 0
    gu = shape_ok and T * cfg.k >= 256 * cfg.E
    dn = shape_ok and T * cfg.k >= (64 if cfg.I >= 2048 else 256) * cfg.E
    return {"gateup": "cta_pair" if gu else "one_sm", "down": "cta_pair" if dn else "one_sm"}


def time_layer(moe, d, wts, x, y, ws, lay, cfg, T, steps, warmup, pg, stream, l2_flush=False,
               path=None, capacity=0, fp8_weights=None):
    """Warm-up, then the timed region (K forwards between two events, barrier +
    synchronize on both sides), then the same K forwards with stage events and
    with per-step events.  Returns the timings, the host time per call and the
    routing counts the workspace holds afterwards.  capacity > 0: the
    capacity-limited forward; fp8_weights: the FP8-weight forward (both one
    call whose stage events all fall around it)."""
    import torch

    def fwd(stage_events=None):
        if capacity <= 0 and fp8_weights is None:
            moe.moe_layer_forward(d, wts, x, y, ws, stage_events=stage_events, path=path)
            return
        cur = torch.cuda.current_stream()
        if stage_events is not None:
            stage_events[0].record(cur)
        if fp8_weights is not None:
            moe.moe_layer_forward_fp8(d, fp8_weights, x, y, ws)
        else:
            moe.moe_layer_forward_capacity(d, wts, x, y, capacity, ws)
        if stage_events is not None:
            for e in stage_events[1:]:
                e.record(cur)

    for _ in range(warmup):
        fwd()
    torch.cuda.synchronize()
    st, raw = moe.moe_get_device_status(ws)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status {st} raw={raw:#x}")
    stage_ev = [new_events(stream, moe.MOE_STAGE_EVENTS) for _ in range(steps)]
    torch.cuda.synchronize()

    # ---- timed region: K steps, only start/end events (an event between two
    # kernels would serialise their programmatic-dependent launch) ----
    barrier(pg)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    if l2_flush:
        # each step alone, after a write larger than L2
        scratch = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for i in range(steps):
            scratch.fill_(i & 0xff)
            ev_a[i].record(stream)
            fwd()
            ev_b[i].record(stream)
        torch.cuda.synchronize()
        barrier(pg)
        ms = sum(ev_a[i].elapsed_time(ev_b[i]) for i in range(steps))
    else:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(steps):
            fwd()
        end.record(stream)
        torch.cuda.synchronize()
        barrier(pg)
        ms = start.elapsed_time(end)
    ms_max = max_over_ranks(ms, pg)
    # ---- the same K steps again with CUDA events at every stage boundary, on
    # the launching stream: per-kernel durations for the roofline ----
    for i in range(steps):
        fwd(stage_ev[i])
    torch.cuda.synchronize()
    t_wall1 = time.time()
    st, raw = moe.moe_get_device_status(ws)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status {st} raw={raw:#x}")

    # ---- the same K steps once more with an event between consecutive
    # forwards only: the spread of single-step times (p10 / p50 / p90) ----
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    step_ev[0].record(stream)
    for i in range(steps):
        fwd()
        step_ev[i + 1].record(stream)
    torch.cuda.synchronize()
    step_us = sorted(1e3 * step_ev[i].elapsed_time(step_ev[i + 1]) for i in range(steps))
    pct = lambda q: step_us[min(len(step_us) - 1, int(q * (len(step_us) - 1) + 0.5))]
    step_spread = {"p10": pct(0.1), "p50": pct(0.5), "p90": pct(0.9)}

    # ---- host time of one call (argument checks, cached tensor maps, launches;
    # the Python binding's marshalling included), the GPU kept busy ahead ----
    n_host = max(10, min(steps, 100))
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    for _ in range(n_host):
        fwd()
    host_us = 1e6 * (time.perf_counter() - h0) / n_host
    torch.cuda.synchronize()

    stage_ms = {n: 0.0 for n in moe.STAGE_NAMES}
    for ev in stage_ev:
        for j, n in enumerate(moe.STAGE_NAMES):
            stage_ms[n] += ev[j].elapsed_time(ev[j + 1])
    stage_us = {n: 1e3 * v / steps for n, v in stage_ms.items()}
    counts = moe.workspace_view(ws, lay, "counts", torch.int32, (cfg.E,)).cpu().tolist()
    gap = moe.workspace_view(ws, lay, "gap", torch.float32, (T,)).cpu()
    dropped = 0
    if capacity > 0:
        inv = moe.workspace_view(ws, lay, "inv_pos", torch.int32, (T * cfg.k,)).cpu()
        dropped = int((inv < 0).sum().item())
    near_ties = int((gap < NEAR_TIE).sum().item()) if cfg.k < cfg.E else 0
    return {"ms_max": ms_max, "stage_us": stage_us, "step_spread": step_spread,
            "host_us": host_us, "counts": counts, "near_ties": near_ties,
            "capacity": capacity, "dropped": dropped, "t_wall": (t_wall0, t_wall1)}


# top-k boundary gaps below this are near-ties (the configuration statement)
NEAR_TIE = 1e-5


def layer_line(cfg, T, args, world, tm, pk, sampler):
    """The JSON line of one layer measurement (without e2e / cpu_baseline)."""
    counts = tm["counts"]
    fp8 = getattr(args, "weights", "bf16") == "fp8"
    alg = algorithmic(cfg, T, counts, 1 if fp8 else 2)
    step_s = tm["ms_max"] / 1e3 / args.steps
    value = world * T / step_s
    stage_us = tm["stage_us"]
    # the persistent decode layer is one kernel (its stage events all fall at
    # its end): its roofline is the whole layer's
    # FP8 weights: the persistent layer up to 16 tokens, else the kernel chain
    # with FP8 GEMMs (no stage events either way: the whole layer is timed)
    fp8_chain = fp8 and not (T <= DECODE_MAX_T and cfg.H >= 256)
    persistent = ((uses_persistent(cfg, T, args.path) and not tm["capacity"]) or
                  (fp8 and not fp8_chain))
    whole = persistent or tm["capacity"] > 0 or fp8_chain
    if whole:
        kern = ("persistent decode layer (router, dispatch, tcgen05 GEMMs, combine)" if persistent
                else "FP8-weight layer forward (kernel chain: route, dispatch, fp16 gather, FP8 "
                     "GEMMs with the weight operand in TMEM, combine)" if fp8_chain
                else "capacity-limited layer forward (kernel chain)")
        kern_bytes, kern_us = alg["layer_bytes"], stage_us["route"]
    else:
        kern = "expert gate/up GEMM + SwiGLU (tcgen05)"
        kern_bytes, kern_us = alg["gateup_bytes"], stage_us["gateup"]
    gu_s = kern_us / 1e6
    gu_gbs = kern_bytes / gu_s / 1e9
    layer_t_hbm = alg["layer_bytes"] / (pk["hbm_gbs"] * 1e9)
    layer_t_tc = alg["layer_flops"] / (pk["bf16_tflops_sustained"] * 1e12)
    layer_roof = max(layer_t_hbm, layer_t_tc)
    num = max(counts) * cfg.E
    den = T * cfg.k
    traffic = None
    prof = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(prof):
        with open(prof) as f:
            tr = json.load(f).get(f"{cfg.name}_T{T}")
        if tr and tr.get("kernel_sources_sha") == kernel_sources_sha():
            traffic = tr["gateup_dram_bytes"]
    return {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tm["ms_max"] / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "weights": "fp8-e4m3, power-of-two scale per 128x128 block" if fp8 else "bf16",
        "data": "synthetic (seeded counter-based generator; random-init weights of the layer shape)",
        "config": workload_config(cfg, T, args.l2_flush),
        "roofline": {"bound": "hbm", "kernel": kern,
                     "achieved": gu_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gu_gbs / pk["hbm_gbs"], "traffic": None if whole else traffic,
                     "algorithmic_bytes": kern_bytes, "launch_us": kern_us,
                     "peak_source": pk["source"]},
        "path": "persistent" if persistent else "chain",
        "gemm_tiles": ({"gateup": "fp8, weight operand in TMEM", "down": "fp8, weight operand in TMEM"}
                       if fp8 else pair_tiles(cfg, T, getattr(args, "path", "auto"))),
        "layer_roofline": {"bound": "hbm" if layer_t_hbm >= layer_t_tc else "tensor",
                           "roof_us": layer_roof * 1e6, "step_us": step_s * 1e6,
                           "frac": layer_roof / step_s, "bytes": alg["layer_bytes"],
                           "flops": alg["layer_flops"], "touched_experts": alg["touched"],
                           "hbm_peak_gbs": pk["hbm_gbs"],
                           "tc_peak_tflops": pk["bf16_tflops_sustained"],
                           "tc_frac_of_burst": alg["layer_flops"] / step_s
                                               / (pk["bf16_tflops"] * 1e12)},
        "stages_us": stage_us,
        "step_us_spread": tm["step_spread"],
        "host_us_per_call": tm["host_us"],
        "routing": {"imbalance_ratio": num / den, "touched_experts": alg["touched"],
                    "near_ties": tm["near_ties"], "near_tie_gap": NEAR_TIE,
                    **({"capacity": tm["capacity"], "dropped_assignments": tm["dropped"]}
                       if tm["capacity"] else {})},
        "gpu_launches": (1 if persistent else launches_per_step(cfg, T, tm["capacity"] > 0))
                        * args.steps,
        "clocks": sampler.summary(*tm["t_wall"]) if sampler else None,
    }


def run_gpu(args):
    import torch

    import routed_expert_ffn_gb300 as moe
    import synth
    from routed_expert_ffn_gb300 import build as moe_build

    world, rank, local, pg = dist_setup(args)
    torch.cuda.set_device(local)
    moe_build.build()
    cfg = layer_config(args)
    T = args.T
    # every rank: the same layer weights, its own batch of tokens
    inp = synth.make_layer(cfg, T, args.seed, device="cuda")
    if rank > 0:
        inp.x = synth.make_tokens(cfg, T, args.seed + 1000 * rank, device="cuda")
    d = moe.desc(T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.gating, cfg.shared)
    ws = moe.alloc_workspace(d)
    lay = moe.moe_workspace_layout(d)
    wts = moe.layer_weights(inp.w_router, inp.w13, inp.w2, inp.sel_bias, inp.w13_shared,
                            inp.w2_shared)
    y = torch.empty((T, cfg.H), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    sampler = ClockSampler(uuid) if rank == 0 else None
    time.sleep(0.5 if sampler else 0)
    cap = (moe.moe_expert_capacity(args.capacity_factor, T, cfg.k, cfg.E)
           if args.capacity_factor > 0 else 0)
    wq = None
    if args.weights == "fp8":   # quantised once, before the timed region
        qd = moe.quantize_layer_fp8(inp.w13, inp.w2, inp.w13_shared, inp.w2_shared)
        wq = moe.layer_weights_fp8(inp.w_router, qd, inp.sel_bias)
        inp.w13 = inp.w2 = inp.w13_shared = inp.w2_shared = None   # keep only the codes
        torch.cuda.empty_cache()
    tm = time_layer(moe, d, wts, inp.x, y, ws, lay, cfg, T, args.steps, args.warmup, pg, stream,
                    args.l2_flush, PATHS[args.path], cap, wq)

    # ---- end to end: pinned host x in, host y out, through the same call ----
    # Every step copies its x from pinned host memory, runs moe_layer_forward
    # and copies its y back to pinned host memory.  The copies run on their
    # own streams with two device buffers each, so a step's copies overlap the
    # neighbouring steps' forwards (the forwards themselves share the
    # workspace and run in order on the compute stream).
    x_host = inp.x.cpu().pin_memory()
    y_host = [torch.empty((T, cfg.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(inp.x) for _ in range(2)]
    y_dev = [torch.empty_like(y) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    h2d_done, fwd_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    e_steps = max(3, min(args.steps, 50))

    def e2e_steps(n, start_event=None):
        for i in range(n):
            b = i & 1
            if start_event is not None and i == 0:
                s_in.wait_event(start_event)
            if i >= 2:
                s_in.wait_event(fwd_done[b])      # forward i-2 has read x_dev[b]
            with torch.cuda.stream(s_in):
                x_dev[b].copy_(x_host, non_blocking=True)
                h2d_done[b].record(s_in)
            stream.wait_event(h2d_done[b])
            if i >= 2:
                stream.wait_event(d2h_done[b])    # y_dev[b] of step i-2 is on the host
            if wq is not None:
                moe.moe_layer_forward_fp8(d, wq, x_dev[b], y_dev[b], ws, stream=stream)
            elif cap:
                moe.moe_layer_forward_capacity(d, wts, x_dev[b], y_dev[b], cap, ws, stream=stream)
            else:
                moe.moe_layer_forward(d, wts, x_dev[b], y_dev[b], ws, stream=stream,
                                      path=PATHS[args.path])
            fwd_done[b].record(stream)
            s_out.wait_event(fwd_done[b])
            with torch.cuda.stream(s_out):
                y_host[b].copy_(y_dev[b], non_blocking=True)
                d2h_done[b].record(s_out)
        for b in range(min(n, 2)):
            stream.wait_event(d2h_done[b])

    e2e_steps(4)
    torch.cuda.synchronize()
    barrier(pg)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_steps(e_steps, start_event=e0)
    e1.record(stream)
    torch.cuda.synchronize()
    e_ms = max_over_ranks(e0.elapsed_time(e1), pg)
    if sampler:
        sampler.stop()
    if rank != 0:
        return
    pk = peaks()
    line = layer_line(cfg, T, args, world, tm, pk, sampler)
    line["e2e"] = {"value": world * T * e_steps / (e_ms / 1e3), "unit": "tokens/s",
                   "h2d_bytes_per_step": T * cfg.H * 2, "d2h_bytes_per_step": T * cfg.H * 2}
    if not args.no_cpu_baseline:
        hin = (host_inputs(cfg, T, args.seed) if args.weights == "fp8"
               else host_inputs(cfg, T, args.seed, experts_from_gpu=inp))
        # the sample: about 15 s of oracle work (a short probe gives the rate)
        k0, dt0, _ = cpu_oracle_sample(hin, min(16, T), seed=7)
        want = args.cpu_tokens if args.cpu_tokens > 0 else int(max(48, 15.0 * k0 / dt0))
        n, dt, threads = cpu_oracle_sample(hin, min(want, T))
        line["cpu_baseline"] = {"value": n / dt, "unit": "tokens/s", "cores": threads,
                                "kind": "oracle", "cpu_model": cpu_model(),
                                "sample": f"{n} seeded tokens of the T={T} batch (routing + "
                                          "expert FFNs + combine, fp64)",
                                "tiny_layer_single_thread": tiny_single_thread()}
    print(json.dumps(line))


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        vendor = model = ""
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
            elif line.startswith("Vendor ID:"):
                vendor = line.split(":", 1)[1].strip()
        if model:
            return f"{vendor} {model}".strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def tiny_single_thread():
    """The oracle on one thread over the whole tiny layer (T=64: router, top-k
    gating, expert FFNs, combine), median of 3 runs, in tokens/s."""
    import oracle
    import synth
    cfg = synth.CONFIGS["tiny"]
    T = 64
    inp = synth.make_layer(cfg, T, 0, device="cpu")
    times = []
    for _ in range(3):
        t0 = time.perf_counter()
        oracle.layer(inp, nthreads=1)
        times.append(time.perf_counter() - t0)
    dt = statistics.median(times)
    return {"value": T / dt, "unit": "tokens/s", "cores": 1, "workload": "tiny layer, T=64",
            "seconds": dt}


# (config, T) pairs of the sweep: every layer configuration at its batch sizes
SWEEP = [("qwen3", T) for T in (1, 16, 128, 256, 1024)] + \
        [("qwen3_tp8", T) for T in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048)] + \
        [("mixtral", T) for T in (1, 8, 64, 512, 4096)] + \
        [("dsv3", T) for T in (2048, 8192)] + [("tiny", 64)]


def run_sweep(args):
    """One JSON line per (layer, T) of SWEEP, each with its own clock record and
    stage times, appended to --sweep-out (and printed)."""
    import torch

    import routed_expert_ffn_gb300 as moe
    import synth
    from routed_expert_ffn_gb300 import build as moe_build
    torch.cuda.set_device(0)
    moe_build.build()
    pk = peaks()
    uuid = "GPU-" + str(torch.cuda.get_device_properties(0).uuid)
    only = set(args.sweep_configs.split(",")) if args.sweep_configs else None
    stream = torch.cuda.current_stream()
    layers = {}
    out_path = args.sweep_out
    for name, T in SWEEP:
        if only is not None and name not in only:
            continue
        if args.sweep_max_T and T > args.sweep_max_T:
            continue
        cfg = synth.CONFIGS[name]
        if name not in layers:
            layers.clear()
            torch.cuda.empty_cache()
            torch.cuda.empty_cache()
            layers[name] = synth.make_layer(cfg, 1, args.seed, device="cuda")
        full = layers[name]
        x = synth.make_tokens(cfg, T, args.seed, device="cuda")
        w_r, b = synth.make_router(cfg, args.seed, device="cuda")
        d = moe.desc(T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.gating, cfg.shared)
        ws = moe.alloc_workspace(d)
        lay = moe.moe_workspace_layout(d)
        wts = moe.layer_weights(w_r, full.w13, full.w2, b, full.w13_shared, full.w2_shared)
        y = torch.empty((T, cfg.H), dtype=torch.bfloat16, device="cuda")
        steps = args.steps if T < 4096 else max(3, args.steps // 10)
        a = argparse.Namespace(**vars(args))
        a.steps = steps
        a.l2_flush = name == "tiny"
        sampler = ClockSampler(uuid)
        time.sleep(0.3)
        cap = (moe.moe_expert_capacity(args.capacity_factor, T, cfg.k, cfg.E)
               if args.capacity_factor > 0 else 0)
        wq = None
        if args.weights == "fp8":
            if name + "_fp8" not in layers:
                layers[name + "_fp8"] = moe.quantize_layer_fp8(full.w13, full.w2,
                                                               full.w13_shared, full.w2_shared)
            wq = moe.layer_weights_fp8(w_r, layers[name + "_fp8"], b)
        tm = time_layer(moe, d, wts, x, y, ws, lay, cfg, T, steps, args.warmup, None, stream,
                        a.l2_flush, PATHS[args.path], cap, wq)
        sampler.stop()
        line = layer_line(cfg, T, a, 1, tm, pk, sampler)
        line["sweep"] = True
        print(json.dumps(line), flush=True)
        if out_path:
            with open(out_path, "a") as f:
                f.write(json.dumps(line) + "\n")
        del ws, y, x


def launches_per_step(cfg, T, capacity=False):
    """Kernels one kernel-chain forward launches: router (one fused kernel up to
    32 tokens, else W_r split + tensor-core router + gating), dispatch (one
    kernel up to 2048 assignments, else three), [the capacity compaction],
    gather + plan, gate/up GEMM, down GEMM, combine."""
    return (1 if T <= 32 else 3) + (1 if T * cfg.k <= 2048 else 3) + 4 + (1 if capacity else 0)


def kernel_sources_sha():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "routed_expert_ffn_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def run_reshard(args):
    """EP <-> TP expert-weight reshard permute of one rank's E/P experts of the
    configuration (Moebius, section 3.1 "Weights Resharding"): pack (EP ->
    per-peer chunks) then unpack (chunks -> EP), each step both directions;
    HBM-bound, every byte read once and written once per direction."""
    import torch
    import synth
    import routed_expert_ffn_gb300 as moe
    from routed_expert_ffn_gb300 import build
    build.build()
    cfg = synth.CONFIGS[args.config]
    P = args.tp
    E_l = max(1, (args.E or cfg.E) // P)
    H, I = cfg.H, cfg.I
    g = torch.Generator(device="cuda").manual_seed(args.seed)
    w13 = torch.randint(-32768, 32767, (E_l, 2 * I, H), dtype=torch.int16, device="cuda",
                        generator=g)
    w2 = torch.randint(-32768, 32767, (E_l, H, I), dtype=torch.int16, device="cuda", generator=g)
    c13 = torch.empty((P, E_l, 2 * I // P, H), dtype=torch.int16, device="cuda")
    c2 = torch.empty((P, E_l, H, I // P), dtype=torch.int16, device="cuda")
    b13, b2 = torch.empty_like(w13), torch.empty_like(w2)
    stream = torch.cuda.current_stream()

    def step():
        moe.moe_reshard_ep_to_tp_pack(E_l, H, I, P, w13, w2, c13, c2)
        moe.moe_reshard_tp_to_ep_unpack(E_l, H, I, P, c13, c2, b13, b2)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if not (torch.equal(b13, w13) and torch.equal(b2, w2)):
        raise RuntimeError("reshard round trip changed the weights")
    uuid = "GPU-" + str(torch.cuda.get_device_properties(0).uuid)
    sampler = ClockSampler(uuid)
    time.sleep(0.5)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0 = time.time()
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    sampler.stop()
    ms = a.elapsed_time(b) / args.steps
    weight_bytes = (w13.numel() + w2.numel()) * 2
    moved = 2 * 2 * weight_bytes  # two directions, each reads and writes every byte
    gbs = moved / (ms * 1e-3) / 1e9
    pk = peaks()
    # DRAM bytes of one step (pack + unpack) from an ncu capture of the same
    # kernel sources, if one is recorded
    traffic = None
    prof = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(prof):
        with open(prof) as f:
            tr = json.load(f).get(f"reshard_{cfg.name}_P{P}")
        if tr and tr.get("kernel_sources_sha") == kernel_sources_sha():
            traffic = tr["step_dram_bytes"]
    # the oracle's permutation (numpy) on the host, same shapes, one direction each
    import oracle
    h13, h2 = w13.cpu().numpy(), w2.cpu().numpy()
    c0 = time.time()
    p13, p2 = oracle.reshard_pack(h13, h2, P)
    oracle.reshard_unpack(p13, p2, P)
    cpu_s = time.time() - c0
    line = {"metric": "EP<->TP expert-weight reshard permute, GB/s moved (read + write)",
            "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (bit copies)",
            "data": "synthetic (random 16-bit patterns)",
            "config": {"workload": f"{cfg.name} EP->TP->EP reshard of one rank, P={P}",
                       "E_local": E_l, "H": H, "I": I, "P": P,
                       "weight_bytes": weight_bytes,
                       "l2": "inputs larger than L2" if weight_bytes > (129 << 20)
                             else "inputs smaller than L2"},
            "roofline": {"bound": "hbm", "kernel": "reshard_kernel (pack + unpack)",
                         "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"], "traffic": traffic,
                         "peak_source": pk["source"]},
            "cpu_baseline": {"value": moved / cpu_s / 1e9, "unit": "GB/s", "cores": 1,
                             "kind": "oracle",
                             "sample": "one pack and one unpack of the same tensors (numpy)"},
            "gpu_launches": 2 * args.steps,
            "clocks": sampler.summary(t0, t1)}
    print(json.dumps(line))


def main():
    args = parse()
    if args.op == "reshard":
        run_reshard(args)
        return
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
