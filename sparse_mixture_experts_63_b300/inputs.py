"""Seeded synthetic inputs for one MoE layer.

This module draws random numbers and nothing else: it holds none of the
layer's arithmetic, so both the CUDA path and the CPU oracle can take their
inputs from it.

Recipe (the same on every device; the stream differs between CPU and CUDA
generators, so a case is identified by (config, seed, device)):
  * one torch.Generator seeded with cfg.seed, drawing in the fixed order
    x, W_g, bias, then per expert e: W_gate[e], W_up[e], W_down[e], then the
    shared expert's Ws_gate, Ws_up, Ws_down;
  * x ~ N(0, 1); every weight ~ N(0, 1/fan_in), i.e. fp32 randn scaled by
    1/sqrt(fan_in), fan_in = d for W_g, W_gate, W_up (and the shared ones),
    f (fs) for W_down (Ws_down);
  * bias[e] ~ N(0, bias_std^2) in fp32 when bias_std > 0;
  * for bf16 layers each fp32 draw is rounded to bf16 (round to nearest even);
    one expert is drawn at a time, so the largest layer never holds an fp32
    copy of all its weights.
"""
import math
from dataclasses import dataclass
from typing import Optional

import torch

from .configs import MoEConfig


@dataclass
class MoEInputs:
    cfg: MoEConfig
    x: torch.Tensor                   # [T, d]
    W_g: torch.Tensor                 # [d, N]
    bias: Optional[torch.Tensor]      # [N] fp32 or None
    W_gate: torch.Tensor              # [N, d, f]
    W_up: torch.Tensor                # [N, d, f]
    W_down: torch.Tensor              # [N, f, d]
    Ws_gate: Optional[torch.Tensor]   # [d, fs] or None
    Ws_up: Optional[torch.Tensor]     # [d, fs] or None
    Ws_down: Optional[torch.Tensor]   # [fs, d] or None

    def tensors(self):
        return dict(x=self.x, W_g=self.W_g, bias=self.bias, W_gate=self.W_gate,
                    W_up=self.W_up, W_down=self.W_down, Ws_gate=self.Ws_gate,
                    Ws_up=self.Ws_up, Ws_down=self.Ws_down)


def torch_dtype(cfg: MoEConfig):
    return torch.float32 if cfg.dtype == "f32" else torch.bfloat16


def _draw(shape, std, g, device, dtype):
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32)
            .mul_(std).to(dtype))


def make_inputs(cfg: MoEConfig, device="cuda", seed: Optional[int] = None) -> MoEInputs:
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(cfg.seed if seed is None else seed)
    dt = torch_dtype(cfg)
    T, d, f, N = cfg.T, cfg.d, cfg.f, cfg.N
    x = _draw((T, d), 1.0, g, device, dt)
    W_g = _draw((d, N), 1.0 / math.sqrt(d), g, device, dt)
    bias = None
    if cfg.bias_std > 0:
        bias = _draw((N,), cfg.bias_std, g, device, torch.float32)
    W_gate = torch.empty((N, d, f), device=device, dtype=dt)
    W_up = torch.empty((N, d, f), device=device, dtype=dt)
    W_down = torch.empty((N, f, d), device=device, dtype=dt)
    for e in range(N):
        W_gate[e] = _draw((d, f), 1.0 / math.sqrt(d), g, device, dt)
        W_up[e] = _draw((d, f), 1.0 / math.sqrt(d), g, device, dt)
        W_down[e] = _draw((f, d), 1.0 / math.sqrt(f), g, device, dt)
    Ws_gate = Ws_up = Ws_down = None
    if cfg.fs > 0:
        Ws_gate = _draw((d, cfg.fs), 1.0 / math.sqrt(d), g, device, dt)
        Ws_up = _draw((d, cfg.fs), 1.0 / math.sqrt(d), g, device, dt)
        Ws_down = _draw((cfg.fs, d), 1.0 / math.sqrt(cfg.fs), g, device, dt)
    return MoEInputs(cfg, x, W_g, bias, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down)


def make_x(cfg: MoEConfig, device="cuda", seed: int = 0) -> torch.Tensor:
    """A fresh activation batch [T, d] for an existing layer (e.g. per bench step)."""
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(seed)
    return _draw((cfg.T, cfg.d), 1.0, g, torch.device(device), torch_dtype(cfg))
