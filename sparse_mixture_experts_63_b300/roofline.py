"""Algorithmic work of one MoE layer forward and its B300 roofline.

Work counted is what the method must do, not the dense work it avoids
("MoE 推理：激活参数 vs 总参数与专家路由", section 直接答案: FLOPs follow the
active parameters, memory the total; section 深入原理: at small batch the
weights actually read are those of the distinct experts the batch touches):

  FLOP  = 2*T*d*N             router
        + 6*d*f*A             routed SwiGLU (three GEMMs of 2*d*f per row)
        + 6*d*fs*T            shared expert
  bytes = sum over experts with >= 1 kept row of 3*d*f*esize
        + d*N*esize (W_g) + 3*d*fs*esize (shared)

With FP8 E4M3 expert weights a matrix counts one byte per weight plus one
fp32 scale per output channel, and its FLOPs run at twice the bf16 rate (the
nominal FP8/bf16 ratio of the dense tensor peaks).

A = kept (token, expert) rows.  Activations are left out of the roofline
bytes and reported separately.  Roofline time = max(FLOP / tensor peak,
bytes / HBM bandwidth); the fraction reported is roofline time / measured time.
"""
import json
import os
from dataclasses import dataclass

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def peaks():
    """Measured B300 peaks (MEASURED_PEAKS.json) or the documented fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(FALLBACK, source="fallback")


def expert_params(d, f):
    """Parameters of one SwiGLU expert: W_gate, W_up [d,f] and W_down [f,d]."""
    return 3 * d * f


def active_fraction(N, k):
    """Share of routed-expert parameters one token uses (k of N experts)."""
    return (k * expert_params(1, 1)) / (N * expert_params(1, 1))


@dataclass
class Work:
    flop: float
    weight_bytes: float
    activation_bytes: float
    flop_ffn: float


def layer_work(T, d, f, N, k, A, touched, fs=0, esize=2, fp8_gate_up=False, fp8_down=False):
    """Algorithmic work of one forward: A kept rows, `touched` experts with >=1 row.
    fp8_gate_up / fp8_down: those routed weights are 1-byte E4M3 codes plus one
    fp32 scale per output channel (the others keep `esize`)."""
    flop_router = 2.0 * T * d * N
    flop_ffn = 6.0 * d * f * A
    flop_shared = 6.0 * d * fs * T
    per_expert = ((2 * d * f + 2 * f * 4) if fp8_gate_up else 2 * d * f * esize) + \
        ((d * f + d * 4) if fp8_down else d * f * esize)
    wbytes = touched * per_expert + d * N * esize + expert_params(d, fs) * esize
    # x read twice (router, gather), x_perm written+read, h written+read (gate/up -> down),
    # y_perm written+read, y written in fp32 (+ shared y written + read)
    act = (2 * T * d + 2 * A * d + 2 * A * f + 2 * A * d) * esize + T * d * 4
    if fs:
        act += (2 * T * fs + 2 * T * d) * esize
    return Work(flop_router + flop_ffn + flop_shared, float(wbytes), float(act),
                flop_ffn + flop_shared)


# Dense FP8 over dense bf16 tensor rate, nominal (4.5 vs 2.25 PFLOP/s).
FP8_OVER_BF16 = 2.0


def roofline_time_s(work: Work, pk=None, sustained=False, fp8_flop=0.0):
    """fp8_flop: the part of work.flop that runs on FP8 tensor cores (at the
    bf16 peak times the nominal FP8/bf16 ratio)."""
    pk = pk or peaks()
    tc = pk["bf16_tflops_sustained" if sustained else "bf16_tflops"] * 1e12
    bw = pk["hbm_gbs"] * 1e9
    t_flop = (work.flop - fp8_flop) / tc + fp8_flop / (tc * FP8_OVER_BF16)
    t_bytes = work.weight_bytes / bw
    return max(t_flop, t_bytes), ("tensor" if t_flop >= t_bytes else "hbm"), t_flop, t_bytes
