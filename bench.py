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

--ffn-vs-cublas R times only the routed expert FFN of the workload's expert
shape on exactly R rows per expert, against cuBLAS batched GEMMs of the same
shapes (context: what the library reaches on this power-capped chip).

--ep-emulate G times the expert-parallel layer over G ranks emulated on this
one GPU (the all-to-alls as device copies) against the one-GPU layer on the
same tokens: the device-side cost of the expert-parallel path.
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
METRIC = "MoE-layer tokens/s on 1 B300 and % of roofline (active FLOPs vs expert bytes)"
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
    ap.add_argument("--ffn-vs-cublas", type=int, default=0, metavar="R",
                    help="time only the routed expert FFN of the layer's expert shape with "
                         "exactly R rows per expert, against cuBLAS batched GEMMs (torch.bmm) "
                         "of the same shapes with the SwiGLU in torch (context for the chip's "
                         "power-capped GEMM rate; one JSON line)")
    ap.add_argument("--ep-emulate", type=int, default=0, metavar="G",
                    help="time the expert-parallel layer over G ranks emulated on this one GPU "
                         "(every rank's layer and batch in one process, the all-to-alls as "
                         "device copies) against the one-GPU layer on the same tokens "
                         "(a context line)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the forward-only timing of the other bf16 workloads that the "
                         "default (prefill) run appends as `workloads`")
    return ap.parse_args()


# ---------------------------------------------------------------- clocks ----
class ClockSampler:
    """SM clock and clock-event reasons of one GPU, read (never set) through
    NVML every 10 ms on a background thread while the benchmark runs; the
    summary covers the samples taken inside the timed window only.  Falls
    back to `nvidia-smi -lms 100` when NVML cannot be loaded."""
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
            "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, torch_index, period_s=0.01):
        self.torch_index = torch_index
        self.period = period_s
        self.samples = []          # (host time, sm MHz, max sm MHz, reason bits)
        self.window = None
        self._stop = None
        self._thread = None
        self._proc = None
        self.source = "unsampled"
        self.nvml_error = None

    def _nvml(self):
        """Read-only NVML calls through ctypes on the library nvidia-smi uses:
        returns (SM clock, max SM clock, clock-event reason bits) readers."""
        import ctypes
        L = ctypes.CDLL("libnvidia-ml.so.1")
        if L.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        h = ctypes.c_void_p()
        uuid = None
        try:
            uuid = str(torch.cuda.get_device_properties(self.torch_index).uuid)
        except Exception:   # noqa: BLE001 -- older torch: no uuid, match by index
            pass
        rc = 1
        if uuid:
            u = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            rc = L.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h))
        if rc != 0 and L.nvmlDeviceGetHandleByIndex_v2(self.torch_index, ctypes.byref(h)) != 0:
            raise RuntimeError("no NVML handle for the device")
        NVML_CLOCK_SM = 1
        get_reasons = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            L.nvmlDeviceGetCurrentClocksThrottleReasons

        def clock():
            c = ctypes.c_uint()
            if L.nvmlDeviceGetClockInfo(h, NVML_CLOCK_SM, ctypes.byref(c)) != 0:
                raise RuntimeError("nvmlDeviceGetClockInfo failed")
            return float(c.value)

        def max_clock():
            c = ctypes.c_uint()
            if L.nvmlDeviceGetMaxClockInfo(h, NVML_CLOCK_SM, ctypes.byref(c)) != 0:
                raise RuntimeError("nvmlDeviceGetMaxClockInfo failed")
            return float(c.value)

        def reasons():
            r = ctypes.c_ulonglong()
            if get_reasons(h, ctypes.byref(r)) != 0:
                raise RuntimeError("clock-event reasons unavailable")
            return int(r.value)
        clock(), reasons()   # both readable, or fall back
        return clock, max_clock(), reasons

    def start(self):
        import threading
        try:
            clock, smax, reasons = self._nvml()
        except Exception as exc:   # noqa: BLE001 -- any NVML failure: use nvidia-smi
            self.nvml_error = f"{type(exc).__name__}: {exc}"[:200]
            return self._start_smi()
        self.source = f"nvml every {self.period * 1e3:.0f} ms"
        self._stop = threading.Event()

        def run():
            while not self._stop.is_set():
                try:
                    self.samples.append((time.perf_counter(), clock(), smax, reasons()))
                except Exception:   # noqa: BLE001 -- a failed read drops one sample
                    pass
                self._stop.wait(self.period)
        self._thread = threading.Thread(target=run, daemon=True)
        self._thread.start()

    def _start_smi(self):
        self.path = os.path.join(tempfile.gettempdir(),
                                 f"moe_bench_clocks_{os.getpid()}_{self.torch_index}.csv")
        try:
            self.fh = open(self.path, "w")
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.torch_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            self.source = "nvidia-smi every 100 ms"
        except (OSError, FileNotFoundError):
            self._proc = None

    def mark(self, t0, t1):
        """The timed window, in time.perf_counter() seconds."""
        self.window = (t0, t1)

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=2)
            rows = list(self.samples)
        elif self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
            self.fh.close()
            rows = []
            with open(self.path) as fh:   # no host timestamps: the whole run counts
                for line in fh:
                    p = [q.strip() for q in line.split(",")]
                    try:
                        bits = sum(self.BITS[n] for n, v in zip(
                            ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                             "sw_power_cap"), p[5:9]) if v.lower() == "active")
                        rows.append((None, float(p[1]), float(p[2]), bits))
                    except (ValueError, IndexError):
                        continue
        else:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return self.summary(rows)

    def summary(self, rows):
        """Summary of (host time or None, SM MHz, max SM MHz, reason bits)
        samples: those inside the timed window when the rows carry host times."""
        if self.window is not None and rows and rows[0][0] is not None:
            t0, t1 = self.window
            inside = [r for r in rows if t0 <= r[0] <= t1]
        else:
            inside = rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"],
                    "source": self.source}
        counts = {n: sum(1 for r in inside if r[3] & b) for n, b in self.BITS.items()}
        extra = {"nvml_error": self.nvml_error} if self.nvml_error else {}
        return {**extra, "sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside),
                "sm_min_mhz": min(r[1] for r in inside),
                "samples": len(inside), "reasons": sorted(n for n, c in counts.items() if c),
                "reason_samples": {n: c for n, c in counts.items() if c},
                "source": self.source + ", timed window only"}


STUCK_LOW = 0.75   # median SM clock under this fraction of max, with no reason: a clock lock


def clocks_rejected(clocks):
    """A run to measure again: the GPU slowed itself down (hardware or thermal
    slowdown), or its SM clock sat well below its maximum with no clock-event
    reason at all (a clock lock left by someone else).  A power cap alone
    (`sw_power_cap`) is kept."""
    reasons = clocks.get("reasons") or []
    if any(r in reasons for r in BAD_REASONS):
        return True
    mhz, top = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    return bool(mhz and top and mhz < STUCK_LOW * top and not reasons)


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
WORKLOADS_ALSO = ("deepseek", "mixtral_decode", "capacity")


def resolve_cfg(args):
    cfg = CONFIGS[args.config]
    if args.tokens:
        cfg = cfg.scaled(T=args.tokens)
    if args.experts:
        cfg = cfg.scaled(N=args.experts)
    if args.ffn_dim:
        cfg = cfg.scaled(f=args.ffn_dim, fs=args.ffn_dim if cfg.fs else 0)
    return cfg


def dtype_name(cfg, fp8, fp8_down):
    if fp8_down:
        return "e4m3 experts + bf16"
    if fp8:
        return "e4m3 gate/up + bf16"
    return "bf16" if cfg.dtype == "bf16" else "f32"


def config_dict(cfg, ws, fp8=False, fp8_down=False, reroute=0, y_dtype="f32"):
    """The workload as both arms name it (same keys and values)."""
    return {"workload": cfg_desc(cfg) + (f", overflow re-routed in {reroute} rounds"
                                         if reroute else "")
            + (", gate/up" + (" and down" if fp8_down else "") +
               " in FP8 E4M3 (per-channel / per-row absmax scales)" if fp8 else ""),
            "fp8_gate_up": bool(fp8), "fp8_down": bool(fp8_down), "reroute_rounds": reroute,
            "T": cfg.T, "d": cfg.d, "f": cfg.f, "N": cfg.N, "k": cfg.k, "fs": cfg.fs,
            "capacity_factor": cfg.cf, "bias_std": cfg.bias_std, "y_dtype": y_dtype,
            "parallelism": f"replicas x{ws} (no exchange)",
            "l2": "256 MB L2 flush write between steps, outside the timed events; "
                  "weights also exceed L2"}


class Bench:
    """One layer set up for timing: inputs, weights, outputs, workspace."""

    def __init__(self, cfg, dev, rank=0, reroute=0, fp8=False, fp8_down=False,
                 y_dtype=torch.float32):
        self.cfg = cfg
        self.inp = make_inputs(cfg, device=dev)
        if rank > 0:   # each rank gets its own batch of the same layer
            self.inp.x = make_x(cfg, device=dev, seed=cfg.seed * 1000 + rank)
        inp = self.inp
        self.layer = B.MoELayer(inp.W_g, inp.W_gate, inp.W_up, inp.W_down, cfg.k, bias=inp.bias,
                                Ws_gate=inp.Ws_gate, Ws_up=inp.Ws_up, Ws_down=inp.Ws_down,
                                capacity_factor=cfg.cf, y_dtype=y_dtype, reroute_rounds=reroute,
                                fp8=fp8, fp8_down=fp8 and fp8_down)
        self.y = torch.empty((cfg.T, cfg.d), dtype=y_dtype, device=dev)
        self.outs = self.layer.outputs_for(cfg.T, dev)
        self.a = self.layer.args(inp.x, self.y, self.outs)
        self.wsbuf = self.layer.workspace(self.a, dev)

    def step(self, stream):
        B.moe_forward(self.a, self.wsbuf, stream)

    def timed(self, steps, stream, flush, ws, ffn_events=False):
        """`steps` steps between a barrier and a synchronize on both sides, an L2
        flush before each (outside its events).  Returns the median step time,
        the median time of the routed expert FFN inside those same steps (CUDA
        events that moe_forward records around its grouped-GEMM launches; None
        unless ffn_events), the library launches counted, and the host window."""
        E = lambda: torch.cuda.Event(enable_timing=True)   # noqa: E731
        evs = [(E(), E()) for _ in range(steps)]
        fev = [(E(), E()) for _ in range(steps)] if ffn_events else None
        for pair in fev or ():
            pair[0].record(stream)     # creates the events moe_forward will re-record
            pair[1].record(stream)
        barrier(ws)
        torch.cuda.synchronize()
        l0 = B.moe_launch_counter()
        t0 = time.perf_counter()
        for i, (s, e) in enumerate(evs):
            flush.fill_(1)
            if fev:
                self.a.ffn_event_begin = fev[i][0].cuda_event
                self.a.ffn_event_end = fev[i][1].cuda_event
            s.record(stream)
            self.step(stream)
            e.record(stream)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        barrier(ws)
        launches = B.moe_launch_counter() - l0
        self.a.ffn_event_begin = self.a.ffn_event_end = None
        ms = statistics.median(s.elapsed_time(e) for s, e in evs)
        ffn_ms = statistics.median(s.elapsed_time(e) for s, e in fev) if fev else None
        return ms, ffn_ms, launches, (t0, t1)

    def routing(self):
        offsets = self.outs["offsets"].cpu()
        kept = offsets[1:] - offsets[:-1]
        return dict(A=int(offsets[-1].item()), touched=int((kept > 0).sum().item()),
                    kept=kept)

    def layer_roofline(self, ms, fp8=False, fp8_down=False):
        cfg = self.cfg
        r = self.routing()
        esz = 2 if cfg.dtype == "bf16" else 4
        work = RL.layer_work(cfg.T, cfg.d, cfg.f, cfg.N, cfg.k, r["A"], r["touched"], cfg.fs,
                             esz, fp8_gate_up=fp8, fp8_down=fp8_down)
        pk = RL.peaks()
        fp8_flop = ((4.0 if fp8 else 0.0) + (2.0 if fp8_down else 0.0)) * cfg.d * cfg.f * r["A"]
        t_roof, bound, t_flop, t_bytes = RL.roofline_time_s(work, pk, fp8_flop=fp8_flop)
        return {"bound": bound, "roofline_ms": round(t_roof * 1e3, 4),
                "flop_ms": round(t_flop * 1e3, 4), "bytes_ms": round(t_bytes * 1e3, 4),
                "frac": round(t_roof * 1e3 / ms, 4),
                "tokens_per_s_at_roofline": round(cfg.T / t_roof, 1),
                "active_flop": work.flop, "weight_bytes": work.weight_bytes,
                "activation_bytes": work.activation_bytes,
                "peaks": f"{pk['source']}: {pk['bf16_tflops']} TFLOP/s bf16, "
                         f"{pk['hbm_gbs']} GB/s"}

    def free(self):
        del self.inp, self.layer, self.y, self.outs, self.a, self.wsbuf
        torch.cuda.empty_cache()


def run_workloads(names, local, flush, stream, steps, warmup):
    """Forward-only, clock-sampled timing of further bf16 workloads (one GPU):
    median step, tokens/s and the fraction of each layer's roofline."""
    rec = {}
    dev = torch.device("cuda", local)
    for name in names:
        cfg = CONFIGS[name]
        bn = Bench(cfg, dev)
        for _ in range(warmup):
            bn.step(stream)
        torch.cuda.synchronize()
        # enough steps for ~0.3 s of timed work, so the clock record has samples
        t = time.perf_counter()
        bn.step(stream)
        torch.cuda.synchronize()
        est = max(time.perf_counter() - t, 1e-5)
        n = int(min(400, max(steps, 0.3 / est)))
        sampler = ClockSampler(local)
        sampler.start()
        ms, _, launches, win = bn.timed(n, stream, flush, 1)
        sampler.mark(*win)
        clocks = sampler.stop()
        if clocks_rejected(clocks):
            sampler = ClockSampler(local)
            sampler.start()
            ms, _, launches, win = bn.timed(n, stream, flush, 1)
            sampler.mark(*win)
            clocks = sampler.stop()
            clocks["remeasured"] = True
        r = bn.routing()
        rec[name] = {"ms_per_step": round(ms, 4), "value": round(cfg.T / (ms / 1e3), 1),
                     "unit": "tokens/s", "steps": n, "warmup": warmup,
                     "config": config_dict(cfg, 1), "dtype": dtype_name(cfg, False, False),
                     "layer_roofline": bn.layer_roofline(ms),
                     "routing": {"kept_rows": r["A"], "touched_experts": r["touched"],
                                 "dropped": int(bn.outs["dropped"].item()),
                                 "max_rows_per_expert": int(r["kept"].max().item()),
                                 "min_rows_per_expert": int(r["kept"].min().item())},
                     "gpu_launches": int(launches), "clocks": clocks,
                     "timing": "moe_forward only, median of CUDA events per step"}
        bn.free()
    return rec


def run_ours(args, ws, rank, local):
    cfg = resolve_cfg(args)
    dev = torch.device("cuda", local)
    fp8, fp8_down = bool(args.fp8), bool(args.fp8 and args.fp8_down)
    y_dtype = torch.float32 if args.y_dtype == "f32" else torch.bfloat16
    bn = Bench(cfg, dev, rank, args.reroute, fp8, fp8_down, y_dtype)
    inp, layer, outs = bn.inp, bn.layer, bn.outs
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    cdict = config_dict(cfg, ws, fp8, fp8_down, args.reroute, args.y_dtype)

    for _ in range(args.warmup):
        bn.step(stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    ffn_events = not args.forward_only
    ms, ffn_ms, launches, win = bn.timed(args.steps, stream, flush, ws, ffn_events)
    sampler.mark(*win)
    clocks = sampler.stop()
    if clocks_rejected(clocks):
        # one re-measurement of the timed loop
        sampler = ClockSampler(local)
        sampler.start()
        ms, ffn_ms, launches, win = bn.timed(args.steps, stream, flush, ws, ffn_events)
        sampler.mark(*win)
        clocks = sampler.stop()
        clocks["remeasured"] = True
    ms_max = reduce_max(ms, ws)
    if args.forward_only:
        if rank != 0:
            return None
        return {"metric": METRIC, "value": round(whole_job_value(ws, cfg.T, ms_max), 1),
                "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(ms_max, 4), "dtype": dtype_name(cfg, fp8, fp8_down),
                "config": cdict, "layer_roofline": bn.layer_roofline(ms_max, fp8, fp8_down),
                "gpu_launches": int(launches), "clocks": clocks, "forward_only": True,
                "timing": "moe_forward only, median of CUDA events per step"}

    # per-stage times through the stage entry points (context: separate legs)
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
        return statistics.median(s.elapsed_time(e) for s, e in evs)

    reps = max(3, min(args.steps, 20))
    stage_ms = {
        "router_topk": time_stage(lambda: B.moe_router_topk(inp.x, inp.W_g, k, bias=inp.bias,
                                                            topk_idx=idx, topk_w=w), reps),
        "permute": time_stage(lambda: B.moe_permute(idx, N, x=inp.x, topk_w=w, capacity=cap,
                                                    A_max=A_max), reps),
        "combine": time_stage(lambda: B.moe_combine(y_perm, perm["inv_pos"], y=bn.y), reps),
    }
    if args.reroute > 0:
        cand, cand_w = B.moe_router_topk(inp.x, inp.W_g, k + args.reroute, bias=inp.bias)
        stage_ms["permute_reroute"] = time_stage(
            lambda: B.moe_permute_reroute(cand, cand_w, N, k, cap, x=inp.x), reps)
    # routing diagnostics from the router's logits and the pre-capacity counts
    lg_buf = torch.empty((cfg.T, N), dtype=torch.float32, device=dev)
    B.moe_router_topk(inp.x, inp.W_g, k, bias=inp.bias, logits=lg_buf)
    stage_ms["routing_stats"] = time_stage(lambda: B.moe_routing_stats(perm["counts"], lg_buf),
                                           reps)
    if cfg.fs > 0:
        sh_off = torch.tensor([0, cfg.T], dtype=torch.int32, device=dev)
        ys = torch.empty((cfg.T, cfg.d), dtype=inp.x.dtype, device=dev)
        stage_ms["shared_ffn"] = time_stage(
            lambda: B.moe_expert_ffn(inp.x, sh_off, inp.Ws_gate[None], inp.Ws_up[None],
                                     inp.Ws_down[None], y_perm=ys), reps)

    # end to end through the host-buffer entry point (pinned host x in, y out)
    x_host = inp.x.cpu().pin_memory()
    y_host = torch.empty((cfg.T, cfg.d), dtype=y_dtype).pin_memory()
    x_stage = torch.empty_like(inp.x)
    a_h = layer.args(x_stage, bn.y, outs)
    e2e_serial_ms = time_stage(lambda: B.moe_forward_host_io(a_h, x_host, y_host, bn.wsbuf,
                                                             stream), reps)
    # the same with the copies overlapped with the layer (token chunks; y only)
    a_o = layer.args(x_stage, bn.y, {"device_status": outs["device_status"]})
    chunks = B.moe_forward_overlap_chunks(a_o) if not (cfg.cf > 0 or args.reroute) else 1
    ws_o = layer.workspace(a_o, dev)    # routing outputs live in the workspace here
    e2e_ms = time_stage(lambda: B.moe_forward_host_io_overlapped(a_o, x_host, y_host, ws_o,
                                                                 chunks, stream), reps)
    e2e_max = reduce_max(e2e_ms, ws)
    ffn_max = reduce_max(ffn_ms, ws)
    if rank != 0:
        return None

    # dominant kernel: the routed grouped expert FFN (gate/up + SwiGLU, down +
    # gate scale), timed inside the step loop above
    r = bn.routing()
    A, touched = r["A"], r["touched"]
    esz = 2 if cfg.dtype == "bf16" else 4
    lr = bn.layer_roofline(ms_max, fp8, fp8_down)
    pk = RL.peaks()
    ffn_flop = 6.0 * cfg.d * cfg.f * A
    ffn_bytes = touched * (RL.expert_params(cfg.d, cfg.f) * esz if not fp8
                           else 2 * cfg.d * cfg.f + 2 * cfg.f * 4 +
                           (cfg.d * cfg.f + cfg.d * 4 if fp8_down else cfg.d * cfg.f * esz))
    # FP8 layers: 2/3 of the FFN FLOPs (gate/up) run at the FP8 rate, so the
    # FFN's peak is the bf16 peak scaled by FLOPs over bf16-equivalent FLOPs
    fp8_share = (1.0 if fp8_down else 2 / 3) if fp8 else 0.0
    peak_scale = 1.0 / ((1 - fp8_share) + fp8_share / RL.FP8_OVER_BF16)
    if lr["bound"] == "tensor":
        achieved = ffn_flop / (ffn_max / 1e3) / 1e12
        peak = round(pk["bf16_tflops"] * peak_scale, 1)
        unit = "TFLOP/s"
    else:
        achieved = ffn_bytes / (ffn_max / 1e3) / 1e9
        peak = pk["hbm_gbs"]
        unit = "GB/s"
    traffic, _ = traffic_from_profiles(
        cfg.name + ("_fp8_all" if fp8_down else "_fp8" if fp8 else ""))
    line = {
        "metric": METRIC,
        "value": round(whole_job_value(ws, cfg.T, ms_max), 1),
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_name(cfg, fp8, fp8_down),
        "data": "synthetic (seeded Gaussian x and N(0,1/fan_in) weights of the workload's shape)",
        "config": cdict,
        "timing": "median of per-step CUDA events on the launching stream",
        "layer_roofline": lr,
        "roofline": {"kernel": "grouped expert FFN (gate/up+SwiGLU and down+gate-scale launches)",
                     "bound": "tensor" if lr["bound"] == "tensor" else "hbm",
                     "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "per_launch_ms": round(ffn_max, 4),
                     "timed": "inside the timed steps: CUDA events moe_forward records around "
                              "its routed grouped-GEMM launches (median per step)",
                     "algorithmic": (f"{ffn_flop:.4g} FLOP" if unit == "TFLOP/s"
                                     else f"{ffn_bytes:.4g} B"),
                     "peak_source": f"{pk['source']} (burst)" + (
                         "; gate/up at the bf16 peak x the nominal FP8/bf16 ratio"
                         if fp8 and unit == "TFLOP/s" else ""),
                     # context only: the same kernel against the measured sustained
                     # (power-capped) cuBLAS rate; the bench runs back to back for
                     # seconds, so its clocks sit in that regime
                     **({"peak_sustained": round(pk["bf16_tflops_sustained"] * peak_scale, 1),
                         "frac_of_sustained": round(
                             achieved / (pk["bf16_tflops_sustained"] * peak_scale), 4)}
                        if unit == "TFLOP/s" else {})},
        "stages_ms": {k_: round(v, 4) for k_, v in stage_ms.items()},
        "stages_note": "stage entry points timed in separate legs after the timed steps "
                       "(context only)",
        "routing": {"kept_rows": A, "dropped": int(outs["dropped"].item()),
                    "rerouted": int(outs["rerouted"].item()), "reroute_rounds": args.reroute,
                    "touched_experts": touched, "max_rows_per_expert": int(r["kept"].max().item()),
                    "min_rows_per_expert": int(r["kept"].min().item())},
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
    if (ws == 1 and not args.no_workloads and args.config == "mixtral_prefill" and
            not (args.tokens or args.experts or args.ffn_dim or fp8 or args.reroute)):
        bn.free()
        del flush, x_host, y_host, x_stage, y_perm, perm, lg_buf
        torch.cuda.empty_cache()
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        line["workloads"] = run_workloads(WORKLOADS_ALSO, local, flush, stream,
                                          steps=30, warmup=max(3, args.warmup))
    return line


# ------------------------------------------------------- reference arm ------
def run_reference(args, ws, rank):
    if rank != 0:
        return None
    import oracle
    cfg = resolve_cfg(args)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    dinp = make_inputs(cfg, device=dev)
    per_step = max(0.5, min(6.0, 150.0 / max(1, args.steps + args.warmup)))
    inp, fetch, _ = host_layer(cfg, dinp, min(cfg.T, 4096))
    S = calibrate_sample(inp, fetch, cfg.T, per_step, min(cfg.T, 4096))
    prefetch(inp, S, fetch)
    for _ in range(args.warmup):
        oracle_sample(inp, S, fetch)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle_sample(inp, S, fetch)
        times.append(time.perf_counter() - t)
    dt = statistics.median(times)
    v = S / dt
    sample = (f"first {S} of {cfg.T} tokens per step, full fp64 oracle pass "
              f"(router, top-k, grouping, SwiGLU experts, combine)")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(v, 3), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(cfg, ws, bool(args.fp8), bool(args.fp8 and args.fp8_down),
                              args.reroute, args.y_dtype),
        "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s",
                         "cores": oracle.default_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_ffn_vs_cublas(args, local):
    """The routed FFN (both grouped-GEMM launches, SwiGLU and gate scale fused)
    on N experts of exactly R rows each, against the same FFN as cuBLAS
    batched GEMMs: x_e [N,R,d] x [W_gate|W_up] [N,d,2f], SiLU(gate)*up in
    torch, then h [N,R,f] x W_down [N,f,d]; and the two cuBLAS GEMMs alone.
    Rounds of `steps` back-to-back calls per leg, the order rotated; medians
    of CUDA events.  Useful FLOP 6*N*R*d*f in every leg."""
    cfg = resolve_cfg(args)
    dev = torch.device("cuda", local)
    inp = make_inputs(cfg, device=dev)
    N, d, f, R = cfg.N, cfg.d, cfg.f, args.ffn_vs_cublas
    A = N * R
    gen = torch.Generator(device=dev).manual_seed(cfg.seed)
    x = torch.randn(A, d, device=dev, generator=gen).to(torch.bfloat16)
    off = torch.arange(0, A + 1, R, dtype=torch.int32, device=dev)
    y = torch.empty(A, d, dtype=torch.bfloat16, device=dev)
    Wgu = torch.cat([inp.W_gate, inp.W_up], dim=2)
    xe = x.view(N, R, d)
    g = torch.empty(N, R, 2 * f, dtype=torch.bfloat16, device=dev)
    h = torch.empty(N, R, f, dtype=torch.bfloat16, device=dev)
    y2 = torch.empty(N, R, d, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    launches0 = B.moe_launch_counter()

    def ours():
        B.moe_expert_ffn(x, off, inp.W_gate, inp.W_up, inp.W_down, y_perm=y)

    def cublas_gemms():
        torch.bmm(xe, Wgu, out=g)
        torch.bmm(h, inp.W_down, out=y2)

    def cublas():
        torch.bmm(xe, Wgu, out=g)
        torch.mul(torch.nn.functional.silu(g[..., :f]), g[..., f:], out=h)
        torch.bmm(h, inp.W_down, out=y2)

    def timed(fn):
        E = lambda: torch.cuda.Event(enable_timing=True)   # noqa: E731
        evs = [(E(), E()) for _ in range(args.steps)]
        for s, e in evs:
            s.record(stream)
            fn()
            e.record(stream)
        torch.cuda.synchronize()
        return statistics.median(s.elapsed_time(e) for s, e in evs)

    for _ in range(args.warmup):
        ours()
        cublas()
    torch.cuda.synchronize()
    rel = ((y.float() - y2.view(A, d).float()).norm() / y2.float().norm()).item()
    sampler = ClockSampler(local)
    sampler.start()
    t0 = time.perf_counter()
    legs = (ours, cublas, cublas_gemms)
    rounds = []
    for r in range(3):   # each round starts with a different leg
        t = {}
        for j in range(3):
            fn = legs[(r + j) % 3]
            t[fn.__name__] = timed(fn)
        rounds.append(t)
    sampler.mark(t0, time.perf_counter())
    clocks = sampler.stop()
    flop = 6.0 * A * d * f
    med = {k: statistics.median(t[k] for t in rounds) for k in rounds[0]}
    return {"metric": "routed expert FFN TFLOP/s, ours vs cuBLAS batched GEMMs",
            "workload": f"{cfg.name} expert shape: N={N} experts x {R} rows, d={d}, f={f}, bf16",
            "ours_ms": round(med["ours"], 4), "ours_tflops": round(flop / med["ours"] / 1e9, 1),
            "cublas_ms": round(med["cublas"], 4),
            "cublas_tflops": round(flop / med["cublas"] / 1e9, 1),
            "cublas_gemms_only_ms": round(med["cublas_gemms"], 4),
            "cublas_gemms_only_tflops": round(flop / med["cublas_gemms"] / 1e9, 1),
            "rounds_ms": [{k: round(v, 4) for k, v in t.items()} for t in rounds],
            "rel_frobenius_ours_vs_cublas": float(f"{rel:.3g}"),
            "gpu_launches": int(B.moe_launch_counter() - launches0), "clocks": clocks,
            "timing": f"3 rounds of {args.steps} back-to-back calls per leg, the leg order "
                      "rotated each round; median of CUDA events; weights larger than L2",
            "legs": "ours = moe_expert_ffn (SwiGLU fused); cublas = two torch.bmm + SiLU(gate)*up "
                    "in torch; cublas_gemms = the two torch.bmm alone (no SwiGLU: h is stale)"}


def run_ep_emulated(args, local):
    """Expert parallelism over G ranks, emulated on one GPU: every rank's
    ExpertParallelMoE (its N/G experts) with its own batch of T tokens, the
    exchanges done as device copies (the bytes an all-to-all moves, at copy
    speed rather than a link's).  Timed against moe_forward of the one-GPU
    layer on the same G*T tokens.  Both run on one GPU, so the ratio is the
    expert-parallel path's device-side cost (regroup, return, G sets of
    launches, the host reads of the split sizes), not a multi-GPU time."""
    from sparse_mixture_experts_63_b300 import expert_parallel as EP
    cfg = resolve_cfg(args)
    G = args.ep_emulate
    if cfg.N % G or cfg.cf:
        raise SystemExit("--ep-emulate needs N divisible by G and no capacity limit "
                         "(a capacity applies per rank's batch)")
    dev = torch.device("cuda", local)
    inp = make_inputs(cfg, device=dev)
    Ne = cfg.N // G
    layers = [EP.ExpertParallelMoE(inp.W_g, inp.W_gate[r * Ne:(r + 1) * Ne],
                                   inp.W_up[r * Ne:(r + 1) * Ne], inp.W_down[r * Ne:(r + 1) * Ne],
                                   cfg.k, r, G, bias=inp.bias, Ws_gate=inp.Ws_gate,
                                   Ws_up=inp.Ws_up, Ws_down=inp.Ws_down)
              for r in range(G)]
    xs = [make_x(cfg, device=dev, seed=cfg.seed * 1000 + r + 1) for r in range(G)]
    x_all = torch.cat(xs)
    one = B.MoELayer(inp.W_g, inp.W_gate, inp.W_up, inp.W_down, cfg.k, bias=inp.bias,
                     Ws_gate=inp.Ws_gate, Ws_up=inp.Ws_up, Ws_down=inp.Ws_down)
    y_all = torch.empty((G * cfg.T, cfg.d), dtype=torch.float32, device=dev)
    outs = one.outputs_for(G * cfg.T, dev)
    a = one.args(x_all, y_all, outs)
    wsb = one.workspace(a, dev)
    stream = torch.cuda.current_stream()
    launches0 = B.moe_launch_counter()
    state = {}

    def ep():
        state["ys"] = EP.run_ranks_in_one_process(layers, xs)

    def single():
        B.moe_forward(a, wsb, stream)

    def timed(fn):
        E = lambda: torch.cuda.Event(enable_timing=True)   # noqa: E731
        evs = [(E(), E()) for _ in range(args.steps)]
        for s_, e_ in evs:
            s_.record(stream)
            fn()
            e_.record(stream)
        torch.cuda.synchronize()
        return statistics.median(s_.elapsed_time(e_) for s_, e_ in evs)

    for _ in range(args.warmup):
        ep()
        single()
    torch.cuda.synchronize()
    diff = max(float((state["ys"][r] - y_all[r * cfg.T:(r + 1) * cfg.T]).abs().max())
               for r in range(G))
    # rows each rank sent to other ranks, one forward (x rows + gate weights out, y rows back)
    sent = 0
    for L, x in zip(layers, xs):
        st = L.dispatch(x)
        sent += sum(n for q, n in enumerate(st.send_rows) if q != L.rank)
    esize = 2 if cfg.dtype == "bf16" else 4
    rounds = [(timed(ep), timed(single)) for _ in range(3)]
    ep_ms = statistics.median(r[0] for r in rounds)
    one_ms = statistics.median(r[1] for r in rounds)
    return {"metric": "expert-parallel layer emulated on one GPU (all-to-alls as device copies)",
            "workload": f"{cfg_desc(cfg)}; {G} ranks x {cfg.T} tokens, {Ne} experts per rank",
            "value": round(G * cfg.T / (ep_ms / 1e3), 1), "unit": "tokens/s",
            "ep_ms": round(ep_ms, 4), "one_gpu_layer_ms": round(one_ms, 4),
            "ep_over_one_gpu": round(ep_ms / one_ms, 4),
            "rows_exchanged_per_step": int(sent),
            "bytes_exchanged_per_step": int(sent * (2 * cfg.d * esize + 4)),
            "max_abs_ep_vs_one_gpu": diff,
            "rounds_ms": [[round(x, 4), round(y, 4)] for x, y in rounds],
            "gpu_launches": int(B.moe_launch_counter() - launches0),
            "timing": f"3 rounds of {args.steps} back-to-back forwards per leg, medians of CUDA "
                      "events; both legs on one GPU: not a multi-GPU time"}


def main():
    args = parse()
    if args.ep_emulate > 0:
        print(json.dumps(run_ep_emulated(args, 0)), flush=True)
        return
    if args.ffn_vs_cublas > 0:
        print(json.dumps(run_ffn_vs_cublas(args, 0)), flush=True)
        return
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
