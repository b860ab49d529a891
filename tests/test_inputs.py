"""The seeded input recipe (CPU generator): shapes and dtypes per workload,
the same draw for the same seed, the stated spreads (x ~ N(0,1), weights
~ N(0, 1/fan_in), router bias ~ N(0, bias_std^2)), and bf16 rounding."""
import math

import pytest
import torch

from sparse_mixture_experts_63_b300.configs import CONFIGS
from sparse_mixture_experts_63_b300.inputs import make_inputs, make_x

SMALL = {  # the workloads' structure at sizes a CPU draws in well under a second
    "tiny": CONFIGS["tiny"],
    "deepseek": CONFIGS["deepseek"].scaled(T=64, d=512, f=256, N=16, fs=256),
    "capacity": CONFIGS["capacity"].scaled(T=128, d=512, f=384, N=16),
    "mixtral_prefill": CONFIGS["mixtral_prefill"].scaled(T=128, d=512, f=768),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_shapes_dtypes_and_optional_parts(name):
    cfg = SMALL[name]
    inp = make_inputs(cfg, device="cpu")
    dt = torch.float32 if cfg.dtype == "f32" else torch.bfloat16
    assert inp.x.shape == (cfg.T, cfg.d) and inp.x.dtype == dt
    assert inp.W_g.shape == (cfg.d, cfg.N) and inp.W_g.dtype == dt
    assert inp.W_gate.shape == inp.W_up.shape == (cfg.N, cfg.d, cfg.f)
    assert inp.W_down.shape == (cfg.N, cfg.f, cfg.d)
    assert (inp.bias is None) == (cfg.bias_std == 0)
    if inp.bias is not None:
        assert inp.bias.shape == (cfg.N,) and inp.bias.dtype == torch.float32
    assert (inp.Ws_gate is None) == (cfg.fs == 0)
    if cfg.fs:
        assert inp.Ws_gate.shape == inp.Ws_up.shape == (cfg.d, cfg.fs)
        assert inp.Ws_down.shape == (cfg.fs, cfg.d)


def test_same_seed_same_draw_other_seed_other_draw():
    cfg = SMALL["capacity"]
    a, b = make_inputs(cfg, device="cpu"), make_inputs(cfg, device="cpu")
    for k, v in a.tensors().items():
        if v is not None:
            assert torch.equal(v, b.tensors()[k]), k
    c = make_inputs(cfg, device="cpu", seed=cfg.seed + 1)
    assert not torch.equal(a.x, c.x) and not torch.equal(a.W_down, c.W_down)
    assert torch.equal(make_x(cfg, "cpu", seed=7), make_x(cfg, "cpu", seed=7))
    assert not torch.equal(make_x(cfg, "cpu", seed=7), make_x(cfg, "cpu", seed=8))


def _std(t):
    return t.float().std().item()


def test_spreads_follow_fan_in():
    cfg = SMALL["deepseek"]
    inp = make_inputs(cfg, device="cpu")
    assert _std(inp.x) == pytest.approx(1.0, rel=0.03)
    for w, fan_in in ((inp.W_g, cfg.d), (inp.W_gate, cfg.d), (inp.W_up, cfg.d),
                      (inp.W_down, cfg.f), (inp.Ws_gate, cfg.d), (inp.Ws_up, cfg.d),
                      (inp.Ws_down, cfg.fs)):
        assert _std(w) == pytest.approx(1.0 / math.sqrt(fan_in), rel=0.05)
        assert abs(w.float().mean().item()) < 0.05 / math.sqrt(fan_in)
    # experts are distinct draws, not copies
    assert not torch.equal(inp.W_gate[0], inp.W_gate[1])


def test_router_bias_spread():
    cfg = CONFIGS["capacity"].scaled(T=8, d=64, f=64, N=4096)   # many experts, one bias each
    inp = make_inputs(cfg, device="cpu")
    assert _std(inp.bias) == pytest.approx(cfg.bias_std, rel=0.05)
    pre = make_inputs(CONFIGS["mixtral_prefill"].scaled(T=8, d=64, f=64, N=4096), device="cpu")
    assert _std(pre.bias) == pytest.approx(0.5, rel=0.05)


def test_bf16_layers_hold_rounded_values():
    cfg = SMALL["capacity"]
    inp = make_inputs(cfg, device="cpu")
    g = torch.Generator().manual_seed(cfg.seed)
    x32 = torch.randn((cfg.T, cfg.d), generator=g)   # the first draw of the recipe
    assert torch.equal(inp.x, x32.to(torch.bfloat16))
