#!/usr/bin/env python3
"""Benchmark of the deterministic MoE layer forward with router replay.

One step = one full layer call (router GEMM, top-k or replay + gates, dispatch,
gather, grouped gate/up GEMM with SwiGLU, grouped down GEMM, fixed-order
combine) over one batch of synthetic tokens, through the C ABI.  The default
workload is the decode-like replay layer: T=64 tokens, d=7168, E=384 experts,
top-8, expert FFN 2048, one shared expert, bf16 weights, recorded ids from a
perturbed copy of the hidden states.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config NAME] [--mode replay|own] [--pass forward|backward]

--pass backward times the layer backward instead (MXFP8 expert GEMMs: dH and
dXp on the block-scaled FP8 MMA, quoted against the fp8 peak, the weight
gradients on bf16 MMAs; one step = the weight copies quantised along the
backward's contraction axes, then the whole backward of one batch with
recorded ids, forward recomputed), by default on the 32k-token training layer.  --pass train times a training
step of the layer: weight copies, the forward keeping its activations, and
the backward from them.

Under torchrun each rank runs its own batch on its own GPU (weak scaling, no
collective on the data path; a barrier and a max over ranks for timing).
--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (rank 0 only).

On one GPU the default (headline) run also times every other d=7168 workload
of the layer -- prefill-like Zipf (replay and own), 32k tokens (uniform and
Zipf s=1.2 routing, own), decode with own routing, MXFP8 weights, MXFP8
weights and activations, NVFP4 (own) -- one after another in the same process,
and reports each under "workloads" in the same JSON line (--no-workloads skips
them).
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

METRIC = "MoE-layer tokens/s (384-expert top-8, d=7168, replay, bf16); % of roofline"
BWD_METRIC = ("MoE-layer backward tokens/s (384-expert top-8, d=7168, MXFP8 expert GEMMs, "
              "recorded ids); % of roofline")
TRAIN_METRIC = ("MoE-layer training-step tokens/s (forward + MXFP8 backward, 384-expert top-8, "
                "d=7168, recorded ids); % of roofline")
UNIT = "tokens/s"
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DISPATCH_SEGMENT_PAIRS = 4096  # (token, slot) pairs one dispatch CTA sorts
ONE_SM_MAX_TOKENS = 128        # bf16 batches up to this size run the one-SM expert GEMMs


def kernels_per_step(T, k, wfmt="bf16", act_mx=False):
    """Launches of one layer call: router GEMM, top-k, dispatch (one kernel for
    at most one segment of pairs, else histogram, scan and scatter), gather,
    gate/up, down, combine; with NVFP4 or MXFP8 activations the gather is the
    token rows' quantiser (which writes the gathered rows too) and the rows of h
    have a quantiser of their own."""
    n = 7 if T * k <= DISPATCH_SEGMENT_PAIRS else 9
    return n + (1 if wfmt == "nvfp4" or act_mx else 0)


def launches_per_step(cfg):
    """kernels_per_step plus the shared expert's own gate/up launch when it
    runs on the second stream beside the routing."""
    n = kernels_per_step(cfg.T, cfg.k, cfg.wfmt, cfg.act_mx)
    if cfg.n_shared and cfg.wfmt == "bf16" and cfg.T > ONE_SM_MAX_TOKENS:
        n += 1
    return n


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=None,
                    help="default: c2_decode_replay (forward), c4_train_32k (backward)")
    ap.add_argument("--pass", dest="pass_", choices=["forward", "backward", "train"],
                    default="forward")
    ap.add_argument("--mode", choices=["replay", "own"], default="replay")
    ap.add_argument("--experts", type=int, default=0,
                    help="override the expert count (small captures for the profiler)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the token count (small captures for the profiler)")
    ap.add_argument("--cpu-sample", type=int, default=0,
                    help="tokens of the workload the CPU-baseline oracle runs on "
                         "(default 64 forward, 2 backward)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="forward, 1 GPU: skip timing the other d=7168 workloads beside the "
                         "headline one")
    args = ap.parse_args()
    if args.config is None:
        args.config = "c4_train_32k" if args.pass_ != "forward" else "c2_decode_replay"
    if not args.cpu_sample:
        args.cpu_sample = 2 if args.pass_ != "forward" else 64
    return args


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_desc(cfg, mode):
    act = " activations=mxfp8" if cfg.act_mx else ""
    return (f"{cfg.name}: T={cfg.T} d={cfg.d} E={cfg.E} top-{cfg.k} F={cfg.F} "
            f"shared={cfg.n_shared} weights={cfg.wfmt}{act} mode={mode}")


def weight_bytes_per_value(cfg):
    """Stored bytes per expert weight value: bf16 2; MXFP8 1 + an E8M0 scale
    per 32; NVFP4 1/2 + an E4M3 scale per 16 (the per-matrix fp32 scale is
    negligible)."""
    return {"bf16": 2.0, "mxfp8": 1 + 1 / 32, "nvfp4": 0.5 + 1 / 16}[cfg.wfmt]


def act_bytes_per_value(cfg):
    """Bytes per value of the token rows the expert GEMMs read: bf16 2; MXFP8
    activations 1 + an E8M0 scale per 32; NVFP4 1/2 + an E4M3 scale per 16."""
    if cfg.wfmt == "nvfp4":
        return 0.5 + 1 / 16
    return 1 + 1 / 32 if cfg.act_mx else 2.0


def mma_peak(cfg, bf16_tflops):
    """The expert GEMMs' tensor peak for their operand type: the measured bf16
    peak times the nominal dense ratio (fp8 4.5 / 2.25 = 2, fp4 13.5 / 2.25 =
    6) for the block-scaled kinds; bf16 for the rest (MXFP8 weights with bf16
    activations are dequantised to bf16)."""
    if cfg.wfmt == "nvfp4":
        return 6.0 * bf16_tflops, "fp4 (e2m1, block-scaled) = 6 x bf16"
    if cfg.act_mx:
        return 2.0 * bf16_tflops, "fp8 (e4m3, block-scaled) = 2 x bf16"
    return bf16_tflops, "bf16"


def layer_work(cfg, touched):
    """Algorithmic FLOPs and bytes of one layer call (touched = routed experts
    with at least one token)."""
    T, d, E, k, F, S = cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.n_shared
    flops = T * (2 * d * E + 6 * d * F * (k + S))
    wbytes = 3 * d * F * weight_bytes_per_value(cfg)
    nbytes = (touched * wbytes + S * 3 * d * F * 2 + E * d * 2 + T * d * 2 + T * d * 2
              + T * k * (4 + 4 + 4))
    return flops, nbytes


def gate_up_bytes(cfg, touched, with_shared=True):
    """Algorithmic bytes of one grouped gate/up GEMM launch: the gate and up
    weights of every touched expert (and the shared one, when it runs in the
    same launch) read once, the gathered token rows read, the SwiGLU
    activations written."""
    T, d, k, F = cfg.T, cfg.d, cfg.k, cfg.F
    S = cfg.n_shared if with_shared else 0
    rows = T * k + T * S
    wb = weight_bytes_per_value(cfg)
    return (touched + S) * 2 * F * d * wb + rows * d * act_bytes_per_value(cfg) + rows * F * 2


def down_bytes(cfg, touched):
    T, d, k, F, S = cfg.T, cfg.d, cfg.k, cfg.F, cfg.n_shared
    rows = T * k + T * S
    wb = weight_bytes_per_value(cfg)
    return ((touched + S) * d * F * wb + rows * F * act_bytes_per_value(cfg) + T * k * d * 2
            + S * T * d * 4)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, _, r in rows:
            for n, v in zip(names, r[1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


def stored_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if the
    kernel source has not changed since it was captured; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel)
    if not d:
        return None
    src = os.path.join(ROOT, "deterministic_rl_gb300", "csrc", d.get("source", "gemm.cu"))
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()[:16]
    return d.get("bytes_per_launch") if h == d.get("source_sha256_16") else None


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def host_experts(inp, ids_np):
    """The oracle's view of the experts a token sample uses, fetched to host."""
    import numpy as np
    import oracle
    from oracle import Expert, Matrix
    from deterministic_rl_gb300.synthetic import bf16_bits, u8

    def mat(w, s):
        return Matrix(bf16_bits(w)) if s is None else Matrix(u8(w), u8(s))
    cache = {}
    for e in sorted(set(np.asarray(ids_np).reshape(-1).tolist())):
        cache[e] = Expert(mat(inp.w_gate[e], None if inp.s_gate is None else inp.s_gate[e]),
                          mat(inp.w_up[e], None if inp.s_up is None else inp.s_up[e]),
                          mat(inp.w_down[e], None if inp.s_down is None else inp.s_down[e]))
    shared = []
    if inp.ws_gate is not None:
        shared = [Expert(Matrix(bf16_bits(inp.ws_gate)), Matrix(bf16_bits(inp.ws_up)),
                         Matrix(bf16_bits(inp.ws_down)))]
    return cache, shared


def oracle_sample(inp, tokens, mode):
    """Inputs of an oracle run over the given token indices: hidden states,
    router, recorded ids (the oracle's routing of the perturbed copy) and the
    experts they touch, all on the host."""
    import numpy as np
    import torch
    import oracle
    from deterministic_rl_gb300.synthetic import bf16_bits
    idx = torch.as_tensor(tokens, device=inp.x.device)
    x = bf16_bits(inp.x[idx])
    wr = bf16_bits(inp.w_router)
    bias = None if inp.router_bias is None else inp.router_bias.cpu().numpy()
    if mode == "replay":
        lg = oracle.router_logits(bf16_bits(inp.x_replay_src[idx]), wr, bias)
        rid = oracle.select_topk(lg, inp.cfg.k)
        need = rid
    else:
        rid = None
        need = oracle.select_topk(oracle.router_logits(x, wr, bias), inp.cfg.k)
    cache, shared = host_experts(inp, need)
    return x, wr, bias, rid, cache, shared


def time_oracle(inp, tokens, mode, min_seconds=10.0):
    """The oracle on the sample, repeated until about min_seconds of CPU work."""
    import oracle
    x, wr, bias, rid, cache, shared = oracle_sample(inp, tokens, mode)
    cores = oracle.set_threads(os.cpu_count() or 1)
    passes = 0
    t0 = time.perf_counter()
    while True:
        oracle.layer_forward(x, wr, bias, lambda e: cache[e], shared, inp.cfg.k, replay_ids=rid)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or passes >= 100:
            break
    return len(tokens) * passes / dt, cores, dt, passes


def run_reference(args):
    """The fp64 CPU oracle as it stands, on a bounded sample of the workload."""
    import torch
    import oracle
    from deterministic_rl_gb300.synthetic import CONFIGS, make_layer
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    cfg = CONFIGS[args.config]
    if args.experts:
        cfg = cfg.with_(name=f"{cfg.name}_E{args.experts}", E=args.experts)
    if args.tokens:
        cfg = cfg.with_(name=f"{cfg.name}_T{args.tokens}", T=args.tokens)
    oracle.build()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = make_layer(cfg, dev)  # same seeded bytes as the GPU arm
    per_step = 1
    pool = list(range(min(cfg.T, 8)))
    x, wr, bias, rid, cache, shared = oracle_sample(inp, pool, args.mode)
    cores = oracle.set_threads(os.cpu_count() or 1)

    def step(i):
        j = i % len(pool)
        oracle.layer_forward(x[j:j + per_step], wr, bias, lambda e: cache[e], shared, cfg.k,
                             replay_ids=None if rid is None else rid[j:j + per_step])
    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    value = args.steps * per_step / dt
    sample = (f"{per_step} token per step, cycling over the first {len(pool)} tokens of "
              f"{cfg.name} ({args.mode}); fp64 oracle on {cores} host threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_desc(cfg, args.mode)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def time_forward(cfg, mode, K, warmup, world, local):
    """Time K layer calls of workload cfg (own or replay mode) after `warmup`
    untimed ones, on this rank's GPU: CUDA events on the launching stream,
    barrier and synchronize on both sides, clocks sampled during the timed
    region.  Returns the measurements and the layer (for the e2e leg)."""
    import torch
    from deterministic_rl_gb300 import MoELayer, binding as B
    from deterministic_rl_gb300.synthetic import make_layer
    rank = int(os.environ.get("RANK", "0"))
    # weak scaling: every rank runs its own batch (seed offset by rank)
    inp = make_layer(cfg.with_(seed=cfg.seed + 1000 * rank) if rank else cfg, "cuda")
    layer = MoELayer.from_inputs(inp)
    T = cfg.T
    # weight preparation at load time (untimed): the SM-pair forward reads the
    # gate/up weights from one packed tensor
    packed = cfg.wfmt == "bf16" and T > ONE_SM_MAX_TOKENS
    if packed:
        layer.pack_weights()
    replay = None
    if mode == "replay":
        rid, _ = layer.route(inp.x_replay_src)  # recorded at "inference": untimed
        replay = rid.clone()
    outs = layer.outputs(T)

    def step(x=inp.x, ids=replay):
        layer.forward(x, replay_ids=ids, outputs=outs)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if layer.status() != 0:
        raise RuntimeError(f"device status after warm-up: {B.status_str(layer.status())}")
    cnt = layer.intermediates(T)["cnt"].cpu()
    touched = int((cnt > 0).sum())
    flops, nbytes = layer_work(cfg, touched)
    need_flush = nbytes < 2 * L2_BYTES
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda") if need_flush else None

    ns = len(B.STAGES)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * ns)] for _ in range(K)]
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    for row in evs:
        for e in row:
            e.record()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record()
        for i in range(K):
            if need_flush:
                flush.zero_()
            step_ev[i][0].record()
            B.moe_set_stage_events(evs[i])
            step()
            step_ev[i][1].record()
        end.record()
        torch.cuda.synchronize()
    B.moe_set_stage_events(None)
    barrier(world)
    if layer.status() != 0:
        raise RuntimeError(f"device status after timing: {B.status_str(layer.status())}")
    if need_flush:
        elapsed = sum(a.elapsed_time(b) for a, b in step_ev)
    else:
        elapsed = start.elapsed_time(end)
    t_ms = max_over_ranks(world, elapsed)
    ms_per_step = t_ms / K
    value = world * T * K / (t_ms / 1e3)
    stage_ms = {name: statistics.fmean(evs[i][2 * j].elapsed_time(evs[i][2 * j + 1]) for i in range(K))
                for j, name in enumerate(B.STAGES)}

    pk, pk_kind = peaks()
    hbm = float(pk["hbm_gbs"])
    tensor = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    t_mma, mma_kind = mma_peak(cfg, tensor)
    # the dominant kernel: the grouped gate/up GEMM (+ SwiGLU)
    one_sm = cfg.wfmt == "bf16" and T <= ONE_SM_MAX_TOKENS
    block_scaled = cfg.wfmt == "nvfp4" or cfg.act_mx
    # on SM pairs with bf16 weights the shared expert's gate/up runs on a second
    # stream beside the routing, outside the timed gate/up stage
    shared_in = not (cfg.n_shared and not one_sm and cfg.wfmt == "bf16")
    gu_bytes = gate_up_bytes(cfg, touched, shared_in)
    gu_flops = 4.0 * cfg.d * cfg.F * (T * cfg.k + (T * cfg.n_shared if shared_in else 0))
    gu_ms = stage_ms["gate_up"]
    if one_sm:
        kname = "grouped_gemm_kernel<GEMM_SWIGLU> (one-SM grouped gate/up GEMM + SwiGLU)"
    elif block_scaled:
        kname = (f"bs_pair_kernel<GEMM_SWIGLU, {'nvfp4' if cfg.wfmt == 'nvfp4' else 'mxfp8'}> "
                 "(SM-pair block-scaled gate/up GEMM + SwiGLU)")
    else:
        kname = f"pair_gemm_kernel<GEMM_SWIGLU, {cfg.wfmt}> (SM-pair grouped gate/up GEMM + SwiGLU)"
    if gu_flops / (t_mma * 1e12) > gu_bytes / (hbm * 1e9):
        achieved = gu_flops / (gu_ms / 1e3) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": t_mma, "unit": "TFLOP/s",
                    "frac": achieved / t_mma, "traffic": None,
                    "algorithmic_flops_per_launch": gu_flops, "mma": mma_kind,
                    "peak_source": (f"{pk_kind} (MEASURED_PEAKS.json bf16_tflops, burst)"
                                    if pk_kind == "measured" else "fallback 1.9 PFLOP/s")
                    + ("" if t_mma == tensor else f", scaled: {mma_kind}")}
    else:
        achieved = gu_bytes / (gu_ms / 1e3) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                    "frac": achieved / hbm,
                    # the committed DRAM capture is of the one-SM gate/up kernel
                    "traffic": stored_traffic("gate_up") if one_sm else None,
                    "peak_source": f"{pk_kind} (MEASURED_PEAKS.json hbm_gbs)"
                    if pk_kind == "measured" else "fallback 6.8 TB/s"}
    roofline.update({"kernel": kname, "algorithmic_bytes_per_launch": gu_bytes,
                     "avg_launch_ms": gu_ms})
    # the router GEMM runs in bf16, the expert GEMMs at their operand type's rate
    r_flops = 2.0 * T * cfg.d * cfg.E
    t_tensor = r_flops / (tensor * 1e12) + (flops - r_flops) / (t_mma * 1e12)
    t_nom = r_flops / 2.25e15 + (flops - r_flops) / (2.25e15 * t_mma / tensor)
    t_roof = max(t_tensor, nbytes / (hbm * 1e9))
    layer_roof = {"flops": flops, "bytes": nbytes, "touched_experts": touched,
                  "bound": "tensor" if t_tensor > nbytes / (hbm * 1e9) else "hbm",
                  "roofline_ms": 1e3 * t_roof, "frac": 1e3 * t_roof / ms_per_step,
                  "frac_nominal_8tbs": 1e3 * max(t_nom, nbytes / 8e12) / ms_per_step,
                  "expert_mma": mma_kind,
                  "peaks": f"{pk_kind}: {hbm} GB/s, {tensor} TFLOP/s bf16"}
    return {"inp": inp, "layer": layer, "replay": replay, "outs": outs, "packed": packed,
            "value": value, "ms_per_step": ms_per_step, "nbytes": nbytes, "need_flush": need_flush,
            "roofline": roofline, "layer_roofline": layer_roof, "stages_ms": stage_ms,
            "clocks": clk.summary()}


# Every d = 7168 workload of the layer beside the headline one, timed in the
# same run: (workload, mode, zipf override or None).
EXTRA_WORKLOADS = [("c2_decode_replay", "own", None),
                   ("c3_prefill_zipf", "replay", None), ("c3_prefill_zipf", "own", None),
                   ("c4_train_32k", "own", None), ("c4_train_32k", "own", 1.2),
                   ("c5_mxfp8", "own", None), ("c5_mxfp8_act", "own", None),
                   ("c6_nvfp4", "own", None)]


def run_workloads(args, world, local):
    """The other d = 7168 workloads, each timed like the headline one (same
    warm-up, at most 20 timed steps, clocks sampled), one after another with
    the previous one's memory released."""
    import torch
    from deterministic_rl_gb300.synthetic import CONFIGS
    res = []
    for name, mode, zipf in EXTRA_WORKLOADS:
        cfg = CONFIGS[name]
        if zipf is not None:
            cfg = cfg.with_(zipf=zipf, name=f"{name}_zipf{zipf}")
        K = max(1, min(args.steps, 20))
        r = time_forward(cfg, mode, K, args.warmup, world, local)
        entry = {"workload": workload_desc(cfg, mode), "steps": K, "warmup": args.warmup,
                 "ms_per_step": r["ms_per_step"], "tokens_per_s": r["value"],
                 "layer_roofline_frac": r["layer_roofline"]["frac"],
                 "layer_roofline": r["layer_roofline"],
                 "dominant_kernel": {k: r["roofline"][k] for k in
                                     ("kernel", "bound", "achieved", "peak", "unit", "frac",
                                      "avg_launch_ms")},
                 "stages_ms": r["stages_ms"], "clocks": r["clocks"],
                 "gpu_launches": launches_per_step(cfg) * K,
                 "weights": ("gate/up packed once at load (moe_pack_weights, untimed)"
                             if r["packed"] else "as given")}
        if cfg.near_tie_frac:
            entry["note"] = ("near-tie tokens are not constructed here: they change no "
                             "kernel's work (the parity tests construct them)")
        res.append(entry)
        del r
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return res


def run_ours(args):
    import torch
    from deterministic_rl_gb300 import build as lib_build
    from deterministic_rl_gb300.synthetic import CONFIGS
    world, rank, local = dist_setup(args)
    lib_build.build()
    cfg = CONFIGS[args.config]
    if args.experts:
        cfg = cfg.with_(name=f"{cfg.name}_E{args.experts}", E=args.experts)
    if args.tokens:
        cfg = cfg.with_(name=f"{cfg.name}_T{args.tokens}", T=args.tokens)
    T, K = cfg.T, args.steps
    r = time_forward(cfg, args.mode, K, args.warmup, world, local)
    inp, layer, replay, outs = r["inp"], r["layer"], r["replay"], r["outs"]

    e2e = None
    if not args.no_e2e:
        x_h = inp.x.cpu().pin_memory()
        rid_h = replay.cpu().pin_memory() if replay is not None else None
        out_h = torch.empty(outs[0].shape, dtype=outs[0].dtype, pin_memory=True)
        ids_h = torch.empty(outs[1].shape, dtype=outs[1].dtype, pin_memory=True)
        g_h = torch.empty(outs[2].shape, dtype=outs[2].dtype, pin_memory=True)
        x_d = torch.empty_like(inp.x)
        rid_d = torch.empty_like(replay) if replay is not None else None
        Ke = max(1, min(K, 100))
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(Ke):
            x_d.copy_(x_h, non_blocking=True)
            if rid_d is not None:
                rid_d.copy_(rid_h, non_blocking=True)
            layer.forward(x_d, replay_ids=rid_d, outputs=outs)
            out_h.copy_(outs[0], non_blocking=True)
            ids_h.copy_(outs[1], non_blocking=True)
            g_h.copy_(outs[2], non_blocking=True)
            torch.cuda.current_stream().synchronize()
        dt = max_over_ranks(world, time.perf_counter() - t0)
        h2d = x_h.numel() * 2 + (rid_h.numel() * 4 if rid_h is not None else 0)
        d2h = out_h.numel() * out_h.element_size() + ids_h.numel() * 4 + g_h.numel() * 4
        e2e = {"value": world * T * Ke / dt, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": Ke,
               "api": f"MoELayer.forward -> {'moe_forward_replay' if rid_h is not None else 'moe_forward'}"
                      " (C ABI), pinned host buffers"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tokens = list(range(min(T, args.cpu_sample)))
        v, cores, dt, passes = time_oracle(inp, tokens, args.mode)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"first {len(tokens)} tokens of {cfg.name} ({args.mode}), {passes} fp64 "
                         f"oracle layer passes, {dt:.1f} s"}

    workloads = None
    if (world == 1 and args.config == "c2_decode_replay" and not args.no_workloads
            and not args.experts and not args.tokens):
        del inp, layer, replay, outs, r["inp"], r["layer"], r["outs"], r["replay"]
        torch.cuda.empty_cache()
        workloads = run_workloads(args, world, local)

    if rank == 0:
        line = {"metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": world, "steps": K,
                "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": workload_desc(cfg, args.mode), "tokens_per_step": T,
                           "weights": ("gate/up packed once at load (moe_pack_weights, untimed)"
                                       if r["packed"] else "as given"),
                           "parallelism": f"replicas x{world} (own batch per GPU, no collective)",
                           "l2": ("L2 flushed between steps" if r["need_flush"] else
                                  f"inputs larger than L2: {r['nbytes'] / 1e9:.1f} GB read per step")},
                "roofline": r["roofline"], "layer_roofline": r["layer_roofline"],
                "stages_ms": r["stages_ms"], "clocks": r["clocks"], "e2e": e2e,
                "gpu_launches": launches_per_step(cfg) * K, "cpu_baseline": cpu}
        if workloads is not None:
            line["workloads"] = workloads
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ---- backward ----------------------------------------------------------------------

def backward_kernel_flops(cfg, train=False):
    """Algorithmic FLOPs of each grouped-GEMM launch of one backward (train:
    of one training step, whose down GEMM also forms the shared rows)."""
    T, d, k, F, S = cfg.T, cfg.d, cfg.k, cfg.F, cfg.n_shared
    rows = T * k + T * S
    return {"gate_up": 4.0 * d * F * rows, "down": 2.0 * d * F * (rows if train else T * k),
            "dh": 2.0 * d * F * rows,
            "dxp": 4.0 * d * F * rows, "wgrad_down": 2.0 * d * F * rows,
            "wgrad_gate_up": 4.0 * d * F * rows}


# the backward GEMMs on the block-scaled MXFP8 MMA, and its nominal rate over bf16
BS_BWD_KERNELS = ("dh", "dxp")
FP8_OVER_BF16 = 2.0


def backward_work(cfg, train=False):
    """Algorithmic FLOPs and bytes of one backward step (train: of one training
    step): the grouped GEMMs, the router and gate gradients; every expert weight
    read once, every weight gradient written once (fp32), x and dout read, dx
    (and the layer output) written."""
    T, d, E, k, F, S = cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.n_shared
    flops = sum(backward_kernel_flops(cfg, train).values()) + 2.0 * T * E * d + 6.0 * T * k * d
    nbytes = ((E + S) * 3 * d * F * (2 + 4) + E * d * (2 + 4) + T * d * (2 + 2 + 4)
              + T * k * 4 + (T * d * 2 if train else 0))
    return flops, nbytes


def backward_launches(cfg, train=False):
    """Our kernels per backward step: weight copies (3, +3 for the shared
    expert); router GEMM, top-k; dispatch (1 or 3); padded offsets and the
    tile -> group table; gather; gate/up and down (recomputed, or the training
    forward's); gate backward; router weight gradient; dY quantised along d (token
    order) and along tokens; dH; SwiGLU backward; dXp; dx; token-major Xp and H;
    two weight-gradient GEMMs."""
    prep = 3 + 3 * cfg.n_shared
    disp = 1 if cfg.T * cfg.k <= DISPATCH_SEGMENT_PAIRS else 3
    # train: + the combine of the forward's output
    return prep + 2 + disp + 2 + 1 + 2 + 2 + 2 + 1 + 1 + 1 + 1 + 2 + 2 + (1 if train else 0)


def backward_roofline(cfg, stage_ms, ms_per_step, pk, pk_kind, train=False):
    """Per-kernel fractions, the dominant kernel's roofline and the layer roofline
    of one backward (or training) step from its per-stage times (ms): each grouped
    GEMM against the peak of the MMA it runs on -- dH and dXp on the block-scaled
    MXFP8 MMA at the fp8 peak (the measured bf16 figure times the nominal 2x), the
    others at the bf16 peak -- and the layer's tensor time as the sum of those."""
    flops, nbytes = backward_work(cfg, train)
    hbm = float(pk["hbm_gbs"])
    tensor = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    tensor_s = float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    kf = backward_kernel_flops(cfg, train)
    # dH and dXp run on the block-scaled MXFP8 MMA: the fp8 peak, the measured
    # bf16 figure times the nominal 2x ratio; the rest on bf16 MMAs
    kpeak = {n: tensor * (FP8_OVER_BF16 if n in BS_BWD_KERNELS else 1.0) for n in kf}
    kernels = {n: {"ms": stage_ms[n], "tflops": kf[n] / (stage_ms[n] / 1e3) / 1e12,
                   "peak_tflops": kpeak[n],
                   "frac": kf[n] / (stage_ms[n] / 1e3) / 1e12 / kpeak[n]} for n in kf}
    dom = max(kf, key=lambda n: stage_ms[n])
    knames = {"gate_up": "pair_gemm_kernel<GEMM_SWIGLU, bf16> (gate/up, keeps pre-activations)",
              "down": "pair_gemm_kernel<GEMM_DOWN, bf16> (expert outputs)",
              "dh": "bs_pair_kernel<GEMM_DOWN, MXFP8> (dH = Q(dY) Q(Wd), block-scaled, fp32 rows)",
              "dxp": "bs_pair_kernel<GEMM_DOWN, MXFP8> (dXp, K = 2F, block-scaled, fp32 rows)",
              "wgrad_down": "wgrad_kernel (dWd, ragged K)",
              "wgrad_gate_up": "wgrad_kernel (dWg and dWu, ragged K)"}
    achieved = kernels[dom]["tflops"]
    roofline = {"bound": "tensor", "achieved": achieved, "peak": kpeak[dom], "unit": "TFLOP/s",
                "frac": achieved / kpeak[dom], "traffic": None, "kernel": knames[dom],
                "algorithmic_flops_per_launch": kf[dom], "avg_launch_ms": stage_ms[dom],
                "frac_of_sustained": achieved / (tensor_s * kpeak[dom] / tensor),
                "peak_source": (f"{pk_kind} (MEASURED_PEAKS.json bf16_tflops, burst)"
                                if pk_kind == "measured" else "fallback 1.9 PFLOP/s")
                + (" x 2 (fp8 over bf16, nominal)" if dom in BS_BWD_KERNELS else "")}
    # tensor time: each grouped GEMM at its own peak, the router and gate work at bf16
    t_tensor = (sum(kf[n] / kpeak[n] for n in kf) + (flops - sum(kf.values())) / tensor) / 1e12
    t_tensor_s = t_tensor * tensor / tensor_s
    t_roof = max(t_tensor, nbytes / (hbm * 1e9))
    layer_roof = {"flops": flops, "bytes": nbytes,
                  "bound": "tensor" if t_tensor > nbytes / (hbm * 1e9) else "hbm",
                  "roofline_ms": 1e3 * t_roof, "frac": 1e3 * t_roof / ms_per_step,
                  "frac_of_sustained": 1e3 * max(t_tensor_s, nbytes / (hbm * 1e9)) / ms_per_step,
                  "peaks": f"{pk_kind}: {hbm} GB/s, {tensor} TFLOP/s bf16 burst, "
                           f"{tensor_s} sustained; fp8 = 2 x bf16",
                  "note": "dH and dXp at the fp8 peak (block-scaled MXFP8 MMA); the weight "
                          "gradients and the forward recompute at the bf16 peak (bf16 MMAs of "
                          "the exact MXFP8 values, and the bf16 forward)"}
    return kernels, roofline, layer_roof


def _bwd_cfg(args):
    from deterministic_rl_gb300.synthetic import CONFIGS
    cfg = CONFIGS[args.config]
    if args.experts:
        cfg = cfg.with_(name=f"{cfg.name}_E{args.experts}", E=args.experts)
    if args.tokens:
        cfg = cfg.with_(name=f"{cfg.name}_T{args.tokens}", T=args.tokens)
    return cfg


def backward_workload_desc(cfg, train=False):
    what = "training step (forward + backward)" if train else "backward"
    return (f"{cfg.name} {what}: T={cfg.T} d={cfg.d} E={cfg.E} top-{cfg.k} F={cfg.F} "
            f"shared={cfg.n_shared} bf16 weights, MXFP8 expert GEMMs, recorded ids")


def oracle_backward_sample(inp, n):
    """Host inputs of the backward oracle on the first n tokens: fp64 values of
    x, the router, dout, the recorded ids and the experts they use."""
    import numpy as np
    import torch
    from oracle.backward import ExpertValues
    from deterministic_rl_gb300.synthetic import make_dout, make_replay_ids
    f64 = lambda t: t.detach().to(torch.float64).cpu().numpy()  # noqa: E731
    cfg = inp.cfg
    ids = make_replay_ids(cfg)[:n].numpy()
    dout = f64(make_dout(cfg, device=inp.x.device)[:n])
    cache = {e: ExpertValues(f64(inp.w_gate[e]), f64(inp.w_up[e]), f64(inp.w_down[e]))
             for e in sorted(set(ids.reshape(-1).tolist()))}
    shared = ([ExpertValues(f64(inp.ws_gate), f64(inp.ws_up), f64(inp.ws_down))]
              if inp.ws_gate is not None else [])
    bias = None if inp.router_bias is None else f64(inp.router_bias)
    return f64(inp.x[:n]), f64(inp.w_router), bias, ids, dout, cache, shared


def time_oracle_backward(inp, n, min_seconds=10.0):
    """The backward oracle (every gradient of an n-token batch) repeated until
    about min_seconds of CPU work; tokens/s."""
    from oracle import backward as OB
    x, wr, bias, ids, dout, cache, shared = oracle_backward_sample(inp, n)
    passes = 0
    t0 = time.perf_counter()
    while True:
        OB.layer_backward(x, wr, bias, lambda e: cache[e], shared, ids, dout)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or passes >= 100:
            break
    return n * passes / dt, os.cpu_count() or 1, dt, passes


def run_backward_reference(args):
    """The backward oracle as it stands on host cores: each step is the whole
    backward of one token of the workload (cycling over the first 4)."""
    import torch
    from oracle import backward as OB
    from deterministic_rl_gb300.synthetic import make_layer
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    cfg = _bwd_cfg(args)
    inp = make_layer(cfg, "cuda" if torch.cuda.is_available() else "cpu")
    pool = 4
    x, wr, bias, ids, dout, cache, shared = oracle_backward_sample(inp, pool)

    def step(i):
        j = i % pool
        OB.layer_backward(x[j:j + 1], wr, bias, lambda e: cache[e], shared, ids[j:j + 1],
                          dout[j:j + 1])
    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    value = args.steps / dt
    cores = os.cpu_count() or 1
    sample = (f"1 token per step, cycling over the first {pool} tokens of {cfg.name}; fp64 numpy "
              f"backward oracle (the token's forward activations and every gradient), up to "
              f"{cores} host threads")
    train = args.pass_ == "train"
    line = {"impl": "reference", "metric": TRAIN_METRIC if train else BWD_METRIC, "value": value,
            "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": backward_workload_desc(cfg, train)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_backward_ours(args):
    import torch
    from deterministic_rl_gb300 import MoELayer, binding as B, build as lib_build
    from deterministic_rl_gb300.synthetic import make_dout, make_layer, make_replay_ids
    world, rank, local = dist_setup(args)
    lib_build.build()
    cfg = _bwd_cfg(args)
    # weak scaling: every rank runs its own batch (seed offset by rank)
    rcfg = cfg.with_(seed=cfg.seed + 1000 * rank) if rank else cfg
    inp = make_layer(rcfg, "cuda")
    layer = MoELayer.from_inputs(inp)
    T, K = cfg.T, args.steps
    ids = make_replay_ids(rcfg, device="cuda")
    dout = make_dout(rcfg, device="cuda")
    grads = layer.alloc_grads()
    dx = torch.empty((T, cfg.d), dtype=torch.float32, device="cuda")

    train = args.pass_ == "train"
    outs = layer.outputs(T)

    def step(x=inp.x, i=ids, g=dout):
        layer.prepare_backward()
        if train:
            layer.forward_train(x, replay_ids=i, outputs=outs)
            layer.backward_saved(g, grads=grads, dx=dx)
        else:
            layer.backward(x, i, g, grads=grads, dx=dx)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if layer.backward_status() != 0:
        raise RuntimeError(f"device status after warm-up: {B.status_str(layer.backward_status())}")
    _, nbytes = backward_work(cfg, train)
    ns = len(B.BWD_STAGES)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * ns)] for _ in range(K)]
    for row in evs:
        for e in row:
            e.record()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record()
        for i in range(K):
            B.moe_set_backward_stage_events(evs[i])
            step()
        end.record()
        torch.cuda.synchronize()
    B.moe_set_backward_stage_events(None)
    barrier(world)
    if layer.backward_status() != 0:
        raise RuntimeError(f"device status after timing: {B.status_str(layer.backward_status())}")
    t_ms = max_over_ranks(world, start.elapsed_time(end))
    ms_per_step = t_ms / K
    value = world * T * K / (t_ms / 1e3)
    stage_ms = {name: statistics.fmean(evs[i][2 * j].elapsed_time(evs[i][2 * j + 1])
                                       for i in range(K))
                for j, name in enumerate(B.BWD_STAGES)}

    pk, pk_kind = peaks()
    kernels, roofline, layer_roof = backward_roofline(cfg, stage_ms, ms_per_step, pk, pk_kind,
                                                      train)

    e2e = None
    if not args.no_e2e:
        x_h = inp.x.cpu().pin_memory()
        ids_h = ids.cpu().pin_memory()
        dout_h = dout.cpu().pin_memory()
        dx_h = torch.empty(dx.shape, dtype=dx.dtype, pin_memory=True)
        out_h = torch.empty(outs[0].shape, dtype=outs[0].dtype, pin_memory=True)
        x_d, ids_d, dout_d = torch.empty_like(inp.x), torch.empty_like(ids), torch.empty_like(dout)
        Ke = max(1, min(K, 20))
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(Ke):
            x_d.copy_(x_h, non_blocking=True)
            ids_d.copy_(ids_h, non_blocking=True)
            dout_d.copy_(dout_h, non_blocking=True)
            step(x_d, ids_d, dout_d)
            dx_h.copy_(dx, non_blocking=True)
            if train:
                out_h.copy_(outs[0], non_blocking=True)
            torch.cuda.current_stream().synchronize()
        dt = max_over_ranks(world, time.perf_counter() - t0)
        e2e = {"value": world * T * Ke / dt, "unit": UNIT,
               "h2d_bytes_per_step": x_h.numel() * 2 + ids_h.numel() * 4 + dout_h.numel() * 2,
               "d2h_bytes_per_step": dx_h.numel() * 4 + (out_h.numel() * 2 if train else 0),
               "steps": Ke,
               "api": ("MoELayer.prepare_backward + forward_train + backward_saved -> "
                       "moe_backward_prepare_weights + moe_forward_train + moe_backward_saved"
                       if train else
                       "MoELayer.prepare_backward + MoELayer.backward -> "
                       "moe_backward_prepare_weights + moe_backward")
                      + " (C ABI), pinned host buffers; weight gradients stay on the device"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n = min(T, args.cpu_sample)
        v, cores, dt, passes = time_oracle_backward(inp, n)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"first {n} tokens of {cfg.name} (every gradient of that batch), "
                         f"{passes} fp64 numpy backward-oracle passes, {dt:.1f} s"}

    if rank == 0:
        line = {"metric": TRAIN_METRIC if train else BWD_METRIC, "value": value, "unit": UNIT,
                "n_gpus": world, "steps": K,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": backward_workload_desc(cfg, train), "tokens_per_step": T,
                           "parallelism": f"replicas x{world} (own batch per GPU, no collective)",
                           "l2": f"inputs larger than L2: {nbytes / 1e9:.1f} GB moved per step"},
                "roofline": roofline, "layer_roofline": layer_roof, "kernels": kernels,
                "stages_ms": stage_ms, "clocks": clk.summary(), "e2e": e2e,
                "gpu_launches": backward_launches(cfg, train) * K, "cpu_baseline": cpu}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.pass_ != "forward":
        if args.impl == "reference":
            return run_backward_reference(args)
        return run_backward_ours(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
