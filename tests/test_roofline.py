"""The roofline arithmetic the benchmark reports, checked on the CPU against
closed forms of the five workloads (no GPU needed)."""
import math

import pytest

from sparse_mixture_experts_63_b300 import roofline as RL

PK = dict(hbm_gbs=6491.8, bf16_tflops=1777.7, bf16_tflops_sustained=1399.6, source="test")


def test_prefill_work_and_bound():
    # 16384 tokens, top-2 of 8 experts of 4096 x 14336, every expert touched
    w = RL.layer_work(16384, 4096, 14336, 8, 2, A=32768, touched=8)
    assert w.flop == 2.0 * 16384 * 4096 * 8 + 6.0 * 4096 * 14336 * 32768
    assert w.weight_bytes == 8 * 3 * 4096 * 14336 * 2 + 4096 * 8 * 2
    t, bound, t_flop, t_bytes = RL.roofline_time_s(w, PK)
    assert bound == "tensor" and t == t_flop
    assert math.isclose(t_flop, w.flop / 1777.7e12)
    assert math.isclose(t_bytes, w.weight_bytes / 6491.8e9)


def test_decode_is_bandwidth_bound():
    w = RL.layer_work(32, 4096, 14336, 8, 2, A=64, touched=8)
    t, bound, _, t_bytes = RL.roofline_time_s(w, PK)
    assert bound == "hbm" and t == t_bytes


def test_shared_expert_adds_its_flops_and_bytes():
    a = RL.layer_work(8192, 7168, 2048, 256, 8, A=65536, touched=256)
    b = RL.layer_work(8192, 7168, 2048, 256, 8, A=65536, touched=256, fs=2048)
    assert b.flop - a.flop == 6.0 * 7168 * 2048 * 8192
    assert b.weight_bytes - a.weight_bytes == 3 * 7168 * 2048 * 2


@pytest.mark.parametrize("down", [False, True])
def test_fp8_weight_bytes(down):
    """E4M3 codes are one byte plus one fp32 scale per output channel; the
    matrices left in bf16 keep two bytes."""
    d, f, touched = 4096, 14336, 8
    w = RL.layer_work(32, d, f, 8, 2, A=64, touched=touched, fp8_gate_up=True, fp8_down=down)
    per = 2 * d * f + 2 * f * 4 + ((d * f + d * 4) if down else d * f * 2)
    assert w.weight_bytes == touched * per + d * 8 * 2


def test_fp8_flops_run_at_twice_the_bf16_rate():
    w = RL.layer_work(16384, 4096, 14336, 8, 2, A=32768, touched=8, fp8_gate_up=True)
    fp8_flop = 4.0 * 4096 * 14336 * 32768
    _, _, t_flop, _ = RL.roofline_time_s(w, PK, fp8_flop=fp8_flop)
    assert math.isclose(t_flop, (w.flop - fp8_flop) / 1777.7e12 + fp8_flop / (2 * 1777.7e12))


def test_active_fraction():
    # k of N experts' parameters per token
    assert RL.active_fraction(8, 2) == 0.25
    assert RL.active_fraction(256, 8) == 8 / 256
