#!/usr/bin/env python
"""MoE-layer forward benchmark on B300: tokens/s and fraction of the roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--impl ours|reference] [--reroute R] [--fp8 [--fp8-down]]

One step = one moe_forward (router, top-k/softmax, dispatch, grouped SwiGLU
experts, combine) over one batch of the workload's T tokens, inputs resident
in HBM.  The default workload is the Mixtral-8x7B-shaped prefill layer
(T=16384, d=4096, f=14336, N=8, k=2, router bias N(0, 0.5^2)); --config picks
another of the five (tiny, mixtral_decode, mixtral_prefill, deepseek,
capacity).  Weights and activations are synthetic and seeded.

N > 1 (torchrun): every rank runs an independent replica of the layer on its
own batch (the layer is token-parallel; there is no exchange), so scaling is
weak and value = all ranks' tokens / the slowest rank's time.

--impl reference times the fp64 CPU oracle (the only reference there is) on
the host cores, on a bounded sample of the same workload per step.

--reroute R re-routes capacity overflow in R rounds (layers with a capacity);
--fp8 runs the routed gate/up projections with E4M3 weights and token rows
(--fp8-down the down projection too) and reports them against their own
roofline (E4M3 bytes, FP8 FLOPs at twice the measured bf16 rate).  `e2e` is
the same layer through the host-buffer call with pinned x in and y out, the
copies overlapped with token chunks of the layer where that cannot change y.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_mixture_experts_63_b300 import binding as B  # noqa: E402
from sparse_mixture_experts_63_b300 import roofline as RL  # noqa: E402
from sparse_mixture_experts_63_b300.configs import CONFIGS  # noqa: E402
from sparse_mixture_experts_63_b300.inputs import make_inputs, make_x  # noqa: E402

L2_FLUSH_BYTES = 256 << 20   # > 126 MB L2
BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def parse():
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="mixtral_prefill", choices=sorted(CONFIGS))
    ap.add_argument("--y-dtype", choices=["f32", "bf16"], default="f32")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override T (smaller cases for profiling captures)")
    ap.add_argument("--experts", type=int, default=0,
                    help="override N (smaller profiling cases with the same per-expert shape)")
    ap.add_argument("--ffn-dim", type=int, default=0,
                    help="override f (e.g. tiny experts to profile the router alone)")
    ap.add_argument("--reroute", type=int, default=0,
                    help="re-route capacity overflow to the next-best expert in R rounds "
                         "(layers with a capacity factor only)")
    ap.add_argument("--fp8", action="store_true",
                    help="routed gate/up projections in FP8 E4M3 (per-channel weight and "
                         "per-token activation scales); the down projection stays bf16")
    ap.add_argument("--fp8-down", action="store_true",
                    help="with --fp8: the down projection in FP8 E4M3 too (h quantised per row)")
    ap.add_argument("--forward-only", action="store_true",
                    help="time moe_forward only (no stage, end-to-end or CPU legs)")
    return ap.parse_args()


# ---------------------------------------------------------------- clocks ----
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(),
                                 f"moe_bench_clocks_gpu{gpu_index}_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as fh:
            for line in fh:
                p = [q.strip() for q in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------- helpers ----
def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(v, ws):
    """The slowest rank's value (NCCL on GPUs, gloo on CPU)."""
    if ws == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(ws, tokens_per_rank, ms_max):
    """tokens/s of the whole job: every rank's batch over the slowest rank's time."""
    return ws * tokens_per_rank / (ms_max / 1e3)


def cfg_desc(cfg):
    s = f"{cfg.name}: T={cfg.T} d={cfg.d} f={cfg.f} N={cfg.N} k={cfg.k}"
    if cfg.fs:
        s += f" shared fs={cfg.fs}"
    if cfg.cf:
        s += f" capacity factor {cfg.cf}"
    if cfg.bias_std:
        s += f" router bias N(0,{cfg.bias_std}^2)"
    return s + f" {cfg.dtype}"


def traffic_from_profiles(cfg_name):
    """dram bytes per launch of the dominant kernel from the committed ncu summary,
    or None when absent or taken on kernel sources that have changed since."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None, None
    with open(p) as fh:
        d = json.load(fh)
    ent = d.get(cfg_name)
    if not ent:
        return None, None
    import hashlib
    h = hashlib.sha256()
    for f in ent.get("sources", []):
        fp = os.path.join(ROOT, f)
        if not os.path.exists(fp):
            return None, None
        h.update(open(fp, "rb").read())
    if h.hexdigest()[:16] != ent.get("sources_sha"):
        return None, None
    return ent.get("bytes_per_launch"), ent.get("kernel")


# ----------------------------------------------------------- CPU oracle -----
def oracle_sample(inp, S, fetch):
    """Oracle forward over the first S tokens: routing, grouping, experts, combine."""
    import oracle
    cfg = inp["cfg"]
    x = inp["x"][:S]
    logits = oracle.router_logits(x, inp["W_g"], inp["bias"])
    idx, w = oracle.topk_softmax(logits, cfg.k)
    g = oracle.group(idx, cfg.N, oracle.capacity(cfg.cf, S, cfg.k, cfg.N))
    y = oracle.forward_rows(x, idx, w, g["inv_pos"], fetch, shared=inp["shared"])
    return y


def host_layer(cfg, dev_inp, S_max):
    """Host copies of what the oracle needs for a sample of S_max tokens."""
    x = dev_inp.x[:S_max].cpu()
    W_g = dev_inp.W_g.cpu()
    bias = None if dev_inp.bias is None else dev_inp.bias.cpu()
    shared = None
    if cfg.fs:
        shared = (dev_inp.Ws_gate.cpu(), dev_inp.Ws_up.cpu(), dev_inp.Ws_down.cpu())
    cache = {}

    def fetch(e):
        if e not in cache:
            cache[e] = (dev_inp.W_gate[e].cpu(), dev_inp.W_up[e].cpu(), dev_inp.W_down[e].cpu())
        return cache[e]
    return dict(cfg=cfg, x=x, W_g=W_g, bias=bias, shared=shared), fetch, cache


def prefetch(inp, S, fetch):
    import oracle
    cfg = inp["cfg"]
    logits = oracle.router_logits(inp["x"][:S], inp["W_g"], inp["bias"])
    idx, _ = oracle.topk_softmax(logits, cfg.k)
    for e in sorted(set(idx.ravel().tolist())):
        fetch(e)


def calibrate_sample(inp, fetch, T, seconds, cap):
    """Token count whose oracle pass takes about `seconds` (grown geometrically
    from a tiny sample, since fixed costs dominate the smallest ones)."""
    S = min(T, 2 if inp["cfg"].d * inp["cfg"].f > 1 << 24 else 16)
    while True:
        prefetch(inp, S, fetch)
        t = time.perf_counter()
        oracle_sample(inp, S, fetch)
        dt = time.perf_counter() - t
        if dt >= seconds / 4 or S >= cap:
            return int(min(cap, max(1, S * seconds / max(dt, 1e-4))))
        S = min(cap, S * 4)


def cpu_baseline(cfg, dev_inp, seconds):
    """Times the oracle on the host cores on a bounded token sample; returns dict."""
    import oracle
    S_cap = min(cfg.T, 4096)
    inp, fetch, _ = host_layer(cfg, dev_inp, S_cap)
    S = calibrate_sample(inp, fetch, cfg.T, seconds, S_cap)
    prefetch(inp, S, fetch)
    t = time.perf_counter()
    oracle_sample(inp, S, fetch)
    dt = time.perf_counter() - t
    return {"value": S / dt, "unit": "tokens/s", "cores": oracle.default_threads(),
            "kind": "oracle",
            "sample": (f"first {S} of {cfg.T} tokens of the same layer, full oracle pass "
                       f"(fp64 router, top-k, grouping, SwiGLU experts, combine), {dt:.1f} s")}


# ------------------------------------------------------------ our arm -------
def run_ours(args, ws, rank, local):
    cfg = CONFIGS[args.config]
    if args.tokens:
        cfg = cfg.scaled(T=args.tokens)
    if args.experts:
        cfg = cfg.scaled(N=args.experts)
    if args.ffn_dim:
        cfg = cfg.scaled(f=args.ffn_dim, fs=args.ffn_dim if cfg.fs else 0)
    dev = torch.device("cuda", local)
    inp = make_inputs(cfg, device=dev)
    # each rank gets its own batch of the same layer
    if rank > 0:
        inp.x = make_x(cfg, device=dev, seed=cfg.seed * 1000 + rank)
    y_dtype = torch.float32 if args.y_dtype == "f32" else torch.bfloat16
    layer = B.MoELayer(inp.W_g, inp.W_gate, inp.W_up, inp.W_down, cfg.k, bias=inp.bias,
                       Ws_gate=inp.Ws_gate, Ws_up=inp.Ws_up, Ws_down=inp.Ws_down,
                       capacity_factor=cfg.cf, y_dtype=y_dtype, reroute_rounds=args.reroute,
                       fp8=args.fp8, fp8_down=args.fp8 and args.fp8_down)
    y = torch.empty((cfg.T, cfg.d), dtype=y_dtype, device=dev)
    outs = layer.outputs_for(cfg.T, dev)
    a = layer.args(inp.x, y, outs)
    wsbuf = layer.workspace(a, dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        B.moe_forward(a, wsbuf, stream)

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    def timed_loop():
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        barrier(ws)
        torch.cuda.synchronize()
        l0 = B.moe_launch_counter()
        for s, e in evs:
            flush.fill_(1)               # evict L2 between steps (outside the events)
            s.record(stream)
            step()
            e.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        launches = B.moe_launch_counter() - l0
        return sum(s.elapsed_time(e) for s, e in evs) / args.steps, launches

    ms, launches = timed_loop()
    if args.forward_only:
        clocks = sampler.stop()
        ms_max = reduce_max(ms, ws)
        if rank == 0:
            return {"config": cfg_desc(cfg), "ms_per_step": round(ms_max, 4),
                    "value": round(ws * cfg.T / (ms_max / 1e3), 1), "unit": "tokens/s",
                    "gpu_launches": int(launches), "clocks": clocks, "forward_only": True}
        return None

    # per-stage times through the stage entry points (same inputs, same stream)
    k, N = cfg.k, cfg.N
    cap = B.moe_capacity(cfg.cf, cfg.T, k, N)
    A_max = cfg.T * k if cap == 0 else min(cfg.T * k, N * cap)
    idx, w = B.moe_router_topk(inp.x, inp.W_g, k, bias=inp.bias)
    perm = B.moe_permute(idx, N, x=inp.x, topk_w=w, capacity=cap, A_max=A_max)
    y_perm = torch.empty((A_max, cfg.d), dtype=inp.x.dtype, device=dev)
    torch.cuda.synchronize()

    def time_stage(fn, reps):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        fn()
        for s, e in evs:
            flush.fill_(1)
            s.record(stream)
            fn()
            e.record(stream)
        torch.cuda.synchronize()
        return sum(s.elapsed_time(e) for s, e in evs) / reps

    reps = max(3, min(args.steps, 20))
    stage_ms = {
        "router_topk": time_stage(lambda: B.moe_router_topk(inp.x, inp.W_g, k, bias=inp.bias,
                                                            topk_idx=idx, topk_w=w), reps),
        "permute": time_stage(lambda: B.moe_permute(idx, N, x=inp.x, topk_w=w, capacity=cap,
                                                    A_max=A_max), reps),
        "expert_ffn": time_stage(lambda: B.moe_expert_ffn(perm["x_perm"], perm["offsets"],
                                                          inp.W_gate, inp.W_up, inp.W_down,
                                                          row_scale=perm["row_scale"],
                                                          y_perm=y_perm, A_max=A_max), reps),
        "combine": time_stage(lambda: B.moe_combine(y_perm, perm["inv_pos"], y=y), reps),
    }
    if args.fp8:
        # the FP8 layer's FFN: E4M3 rows of the permuted tokens, E4M3 gate/up
        qg, sg, qu, su = layer.fp8[:4]
        qd, sd = layer.fp8[4:6] if len(layer.fp8) > 4 else (None, None)
        xq, sx = B.quantize_rows_e4m3(inp.x)
        A_kept = int(perm["offsets"][-1].item())          # rows past it hold no token
        xq_perm = torch.zeros((A_max, cfg.d), dtype=torch.uint8, device=dev)
        xq_perm[:A_kept] = xq[perm["perm_token"][:A_kept].long()]
        stage_ms["quantize_rows"] = time_stage(lambda: B.quantize_rows_e4m3(inp.x), reps)
        stage_ms["expert_ffn_bf16"] = stage_ms["expert_ffn"]
        stage_ms["expert_ffn"] = time_stage(lambda: B.moe_expert_ffn_fp8(
            xq_perm, sx, perm["perm_token"], perm["offsets"], qg, sg, qu, su,
            W_down=None if qd is not None else inp.W_down, Wq_down=qd, wscale_down=sd,
            row_scale=perm["row_scale"], y_perm=y_perm, A_max=A_max), reps)
    if args.reroute > 0:
        cand, cand_w = B.moe_router_topk(inp.x, inp.W_g, k + args.reroute, bias=inp.bias)
        stage_ms["permute_reroute"] = time_stage(
            lambda: B.moe_permute_reroute(cand, cand_w, N, k, cap, x=inp.x), reps)
    # routing diagnostics from the router's logits and the pre-capacity counts
    lg_buf = torch.empty((cfg.T, N), dtype=torch.float32, device=inp.x.device)
    B.moe_router_topk(inp.x, inp.W_g, k, bias=inp.bias, logits=lg_buf)
    stage_ms["routing_stats"] = time_stage(lambda: B.moe_routing_stats(perm["counts"], lg_buf),
                                           reps)
    if cfg.fs > 0:
        sh_off = torch.tensor([0, cfg.T], dtype=torch.int32, device=inp.x.device)
        ys = torch.empty((cfg.T, cfg.d), dtype=inp.x.dtype, device=inp.x.device)
        stage_ms["shared_ffn"] = time_stage(
            lambda: B.moe_expert_ffn(inp.x, sh_off, inp.Ws_gate[None], inp.Ws_up[None],
                                     inp.Ws_down[None], y_perm=ys), reps)

    # end to end through the host-buffer entry point (pinned host x in, y out)
    x_host = inp.x.cpu().pin_memory()
    y_host = torch.empty((cfg.T, cfg.d), dtype=y_dtype).pin_memory()
    x_stage = torch.empty_like(inp.x)
    a_h = layer.args(x_stage, y, outs)
    e2e_serial_ms = time_stage(lambda: B.moe_forward_host_io(a_h, x_host, y_host, wsbuf, stream),
                               reps)
    # the same with the copies overlapped with the layer (token chunks; y only)
    a_o = layer.args(x_stage, y, {"device_status": outs["device_status"]})
    chunks = B.moe_forward_overlap_chunks(a_o) if not (cfg.cf > 0 or args.reroute) else 1
    ws_o = layer.workspace(a_o, dev)    # routing outputs live in the workspace here
    e2e_ms = time_stage(lambda: B.moe_forward_host_io_overlapped(a_o, x_host, y_host, ws_o,
                                                                 chunks, stream), reps)
    clocks = sampler.stop()
    if any(r in clocks.get("reasons", []) for r in BAD_REASONS):
        # one re-measurement of the main loop
        sampler = ClockSampler(local)
        sampler.start()
        ms, launches = timed_loop()
        clocks = sampler.stop()
        clocks["remeasured"] = True

    ms_max = reduce_max(ms, ws)
    e2e_max = reduce_max(e2e_ms, ws)
    if rank != 0:
        return None

    # work and roofline
    counts = outs["counts"].cpu()
    offsets = outs["offsets"].cpu()
    kept = (offsets[1:] - offsets[:-1])
    A = int(offsets[-1].item())
    touched = int((kept > 0).sum().item())
    esz = 2 if cfg.dtype == "bf16" else 4
    fp8_down = args.fp8 and args.fp8_down
    work = RL.layer_work(cfg.T, cfg.d, cfg.f, N, k, A, touched, cfg.fs, esz,
                         fp8_gate_up=args.fp8, fp8_down=fp8_down)
    pk = RL.peaks()
    fp8_flop = (4.0 if args.fp8 else 0.0) * cfg.d * cfg.f * A + (2.0 if fp8_down else 0.0) * cfg.d * cfg.f * A
    t_roof, bound, t_flop, t_bytes = RL.roofline_time_s(work, pk, fp8_flop=fp8_flop)
    value = whole_job_value(ws, cfg.T, ms_max)

    # dominant kernel: the grouped expert FFN (gate/up + SwiGLU, down + gate scale)
    ffn_ms = stage_ms["expert_ffn"]
    ffn_flop = 6.0 * cfg.d * cfg.f * A
    ffn_bytes = touched * (RL.expert_params(cfg.d, cfg.f) * esz if not args.fp8
                           else 2 * cfg.d * cfg.f + 2 * cfg.f * 4 +
                           (cfg.d * cfg.f + cfg.d * 4 if fp8_down else cfg.d * cfg.f * esz))
    # FP8 layers: 2/3 of the FFN FLOPs (gate/up) run at the FP8 rate, so the
    # FFN's peak is the bf16 peak scaled by FLOPs over bf16-equivalent FLOPs
    fp8_share = (1.0 if fp8_down else 2 / 3) if args.fp8 else 0.0
    peak_scale = 1.0 / ((1 - fp8_share) + fp8_share / RL.FP8_OVER_BF16)
    if bound == "tensor":
        achieved = ffn_flop / (ffn_ms / 1e3) / 1e12
        peak = round(pk["bf16_tflops"] * peak_scale, 1)
        unit = "TFLOP/s"
    else:
        achieved = ffn_bytes / (ffn_ms / 1e3) / 1e9
        peak = pk["hbm_gbs"]
        unit = "GB/s"
    traffic, tkernel = traffic_from_profiles(
        cfg.name + ("_fp8_all" if fp8_down else "_fp8" if args.fp8 else ""))
    line = {
        "metric": "MoE-layer tokens/s on 1 B300 and % of roofline (active FLOPs vs expert bytes)",
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("e4m3 experts + bf16" if fp8_down else "e4m3 gate/up + bf16" if args.fp8 else
                  "bf16" if cfg.dtype == "bf16" else "f32"),
        "data": "synthetic (seeded Gaussian x and N(0,1/fan_in) weights of the workload's shape)",
        "config": {"workload": cfg_desc(cfg) + (f", overflow re-routed in {args.reroute} rounds"
                                                 if args.reroute else "")
                   + (", gate/up" + (" and down" if fp8_down else "") +
                      " in FP8 E4M3 (per-channel / per-row absmax scales)" if args.fp8 else ""),
                   "fp8_gate_up": bool(args.fp8), "fp8_down": bool(fp8_down),
                   "reroute_rounds": args.reroute, "T": cfg.T, "d": cfg.d, "f": cfg.f, "N": N,
                   "k": k, "fs": cfg.fs, "capacity_factor": cfg.cf, "bias_std": cfg.bias_std,
                   "y_dtype": args.y_dtype, "parallelism": f"replicas x{ws} (no exchange)",
                   "l2": "256 MB L2 flush write between steps, outside the timed events; "
                         "weights also exceed L2"},
        "layer_roofline": {"bound": bound, "roofline_ms": round(t_roof * 1e3, 4),
                           "flop_ms": round(t_flop * 1e3, 4), "bytes_ms": round(t_bytes * 1e3, 4),
                           "frac": round(t_roof * 1e3 / ms_max, 4),
                           "tokens_per_s_at_roofline": round(cfg.T / t_roof, 1),
                           "active_flop": work.flop, "weight_bytes": work.weight_bytes,
                           "activation_bytes": work.activation_bytes,
                           "peaks": f"{pk['source']}: {pk['bf16_tflops']} TFLOP/s bf16, "
                                    f"{pk['hbm_gbs']} GB/s"},
        "roofline": {"kernel": "grouped expert FFN (gate/up+SwiGLU and down+gate-scale launches)",
                     "bound": "tensor" if bound == "tensor" else "hbm",
                     "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "per_launch_ms": round(ffn_ms, 4),
                     "algorithmic": (f"{ffn_flop:.4g} FLOP" if unit == "TFLOP/s"
                                     else f"{ffn_bytes:.4g} B"),
                     "peak_source": f"{pk['source']} (burst)" + (
                         "; gate/up at the bf16 peak x the nominal FP8/bf16 ratio"
                         if args.fp8 and unit == "TFLOP/s" else ""),
                     # context only: the same kernel against the measured sustained
                     # (power-capped) cuBLAS rate; the bench runs back to back for
                     # seconds, so its clocks sit in that regime
                     **({"peak_sustained": round(pk["bf16_tflops_sustained"] * peak_scale, 1),
                         "frac_of_sustained": round(
                             achieved / (pk["bf16_tflops_sustained"] * peak_scale), 4)}
                        if unit == "TFLOP/s" else {})},
        "stages_ms": {k_: round(v, 4) for k_, v in stage_ms.items()},
        "routing": {"kept_rows": A, "dropped": int(outs["dropped"].item()),
                    "rerouted": int(outs["rerouted"].item()), "reroute_rounds": args.reroute,
                    "touched_experts": touched, "max_rows_per_expert": int(kept.max().item()),
                    "min_rows_per_expert": int(kept.min().item())},
        "e2e": {"value": round(ws * cfg.T / (e2e_max / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": cfg.T * cfg.d * esz,
                "d2h_bytes_per_step": cfg.T * cfg.d * (4 if args.y_dtype == "f32" else 2),
                "ms_per_step": round(e2e_max, 4),
                "api": f"moe_forward_host_io_overlapped (pinned host x, y; {chunks} token "
                       f"chunk{'s' if chunks > 1 else ''}, copies on two side streams)",
                "serial_copies_ms_per_step": round(e2e_serial_ms, 4)},
        "gpu_launches": int(launches),
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, inp, args.cpu_seconds)
    return line


# ------------------------------------------------------- reference arm ------
def run_reference(args, ws, rank):
    if rank != 0:
        return None
    import oracle
    cfg = CONFIGS[args.config]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    dinp = make_inputs(cfg, device=dev)
    per_step = max(0.5, min(6.0, 150.0 / max(1, args.steps + args.warmup)))
    inp, fetch, _ = host_layer(cfg, dinp, min(cfg.T, 4096))
    S = calibrate_sample(inp, fetch, cfg.T, per_step, min(cfg.T, 4096))
    prefetch(inp, S, fetch)
    for _ in range(args.warmup):
        oracle_sample(inp, S, fetch)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample(inp, S, fetch)
    dt = (time.perf_counter() - t) / args.steps
    v = S / dt
    sample = (f"first {S} of {cfg.T} tokens per step, full fp64 oracle pass "
              f"(router, top-k, grouping, SwiGLU experts, combine)")
    return {
        "impl": "reference",
        "metric": "MoE-layer tokens/s on 1 B300 and % of roofline (active FLOPs vs expert bytes)",
        "value": round(v, 3), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg_desc(cfg), "T": cfg.T, "d": cfg.d, "f": cfg.f, "N": cfg.N,
                   "k": cfg.k, "fs": cfg.fs, "capacity_factor": cfg.cf,
                   "bias_std": cfg.bias_std},
        "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s",
                         "cores": oracle.default_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    ws, rank, local = dist_setup(args)
    if args.impl == "reference":
        line = run_reference(args, ws, rank)
    else:
        line = run_ours(args, ws, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
