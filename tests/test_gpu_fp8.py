"""GPU parity of the FP8 (E4M3) expert path against the fp64 oracle.

Quantisation is byte work: the codes and scales must match the oracle's bit
for bit.  The FFN and the layer are compared with the oracle's fp64 layer on
the same E4M3 values (its own quantisation of the inputs), within the bf16
layer tolerance: with a bf16 down projection h is rounded to bf16 between the
GEMMs, as in the bf16 path; with an E4M3 down projection the oracle quantises
its exact h per row and the kernels quantise their fp32 h.
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_mixture_experts_63_b300 import binding as B
from sparse_mixture_experts_63_b300.configs import CONFIGS, MoEConfig
from sparse_mixture_experts_63_b300.inputs import make_inputs

import parity

pytestmark = pytest.mark.gpu

SMALL = {
    "mixtral_small": MoEConfig("mixtral_small", T=300, d=512, f=1024, N=8, k=2, bias_std=0.5,
                               seed=31),
    "deepseek_small": MoEConfig("deepseek_small", T=200, d=256, f=256, N=256, k=8, fs=256,
                                seed=41),
    "capacity_small": MoEConfig("capacity_small", T=512, d=256, f=192, N=32, k=2, cf=1.25,
                                bias_std=1.0, seed=51),
    "wide_tiles": MoEConfig("wide_tiles", T=1200, d=256, f=192, N=8, k=2, bias_std=0.4, seed=77),
    "ragged_k": MoEConfig("ragged_k", T=257, d=272, f=200, N=8, k=2, seed=78),
    "one_token": MoEConfig("one_token", T=1, d=64, f=64, N=8, k=2, seed=71),
}


@pytest.mark.parametrize("R,C,scale", [(1, 16, 1.0), (333, 272, 3.0), (64, 4096, 1e-3),
                                       (5, 64, 300.0)])
def test_quantize_rows_bit_exact(R, C, scale):
    g = torch.Generator().manual_seed(R + C)
    x = (torch.randn((R, C), generator=g) * scale).to(torch.bfloat16)
    x[0, :] = 0                                   # an all-zero row: scale 1
    if R > 2:
        x[1, 3] = 1e4                             # one large element
    q, s = B.quantize_rows_e4m3(x.cuda())
    torch.cuda.synchronize()
    qo, so = oracle.quantize_rows_e4m3(x)
    np.testing.assert_array_equal(q.cpu().numpy(), qo)
    np.testing.assert_array_equal(s.cpu().numpy(), so)


@pytest.mark.parametrize("N,d,f", [(1, 16, 1), (3, 272, 200), (2, 128, 64), (4, 4096, 96)])
def test_quantize_weights_bit_exact(N, d, f):
    g = torch.Generator().manual_seed(N * d + f)
    W = (torch.randn((N, d, f), generator=g) * d ** -0.5).to(torch.bfloat16)
    W[0, :, 0] = 0                                # an all-zero channel
    q, s = B.quantize_weights_e4m3(W.cuda())
    torch.cuda.synchronize()
    qo, so = oracle.quantize_weights_e4m3(W)
    np.testing.assert_array_equal(q.cpu().numpy(), qo)
    np.testing.assert_array_equal(s.cpu().numpy(), so)


@pytest.mark.parametrize("down", [False, True], ids=["bf16_down", "fp8_down"])
@pytest.mark.parametrize("counts", [
    [0, 1, 256, 257, 288, 320, 321, 600, 641, 100, 0, 960],
    [0, 1, 160, 161, 255, 256, 257, 288, 320, 321, 600, 641, 100, 0, 960, 200],
    [3, 17, 64, 0, 31],
])
def test_expert_ffn_fp8_crafted_counts(counts, down):
    """FP8 gate/up on expert sizes at every tiling edge (empty, one row, one
    and two sub-tiles, experts split into several tiles), tokens repeated in
    any order, against the oracle's fp64 expert on the same E4M3 values."""
    N, d, f = len(counts), 256, 192
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    A = int(off[-1])
    g = torch.Generator().manual_seed(79)
    T = A // 2 + 3
    x = (torch.randn((T, d), generator=g) * 0.5).to(torch.bfloat16)
    pt = torch.randint(0, T, (A,), generator=g, dtype=torch.int32)
    Wg = (torch.randn((N, d, f), generator=g) * d ** -0.5).to(torch.bfloat16)
    Wu = (torch.randn((N, d, f), generator=g) * d ** -0.5).to(torch.bfloat16)
    Wd = (torch.randn((N, f, d), generator=g) * f ** -0.5).to(torch.bfloat16)
    rs = torch.rand((A,), generator=g) + 0.5
    qx, sx = oracle.quantize_rows_e4m3(x)
    (qg, sg), (qu, su) = oracle.quantize_weights_e4m3(Wg), oracle.quantize_weights_e4m3(Wu)
    ptn = pt.numpy()
    qd, sd = oracle.quantize_weights_e4m3(Wd) if down else (None, None)
    gpu = lambda a: None if a is None else torch.from_numpy(a).cuda()
    y = B.moe_expert_ffn_fp8(gpu(qx[ptn]), gpu(sx), pt.cuda(), gpu(off), gpu(qg), gpu(sg),
                             gpu(qu), gpu(su), W_down=None if down else Wd.cuda(),
                             Wq_down=gpu(qd), wscale_down=gpu(sd), row_scale=rs.cuda(), A_max=A)
    torch.cuda.synchronize()
    ref = np.zeros((A, d))
    for e in range(N):
        if counts[e]:
            rows = ptn[off[e]:off[e + 1]]
            ref[off[e]:off[e + 1]] = oracle.expert_rows_fp8(
                qg[e], sg[e], qu[e], su[e], Wd[e], qx[rows], sx[rows],
                None if qd is None else qd[e], None if sd is None else sd[e])
    ref *= rs.double().numpy()[:, None]
    parity.assert_y_close(y[:A].float().cpu().numpy(), ref, "bf16")


@pytest.mark.parametrize("down", [False, True], ids=["bf16_down", "fp8_down"])
@pytest.mark.parametrize("name", list(SMALL))
def test_layer_fp8_reduced(name, down):
    cfg = SMALL[name]
    if down and cfg.f % 16:
        pytest.skip("an E4M3 down projection needs f % 16 == 0")
    inp = make_inputs(cfg, device=torch.device("cuda"))
    print(name, down, parity.check_layer_fp8(cfg, inp, down=down))


@pytest.mark.parametrize("down", [False, True], ids=["bf16_down", "fp8_down"])
@pytest.mark.parametrize("name,rows", [("mixtral_decode", None), ("capacity", None),
                                       ("mixtral_prefill", 512), ("deepseek", 256)])
def test_layer_fp8_full_size(name, rows, down):
    """The FP8 layer at the sizes the benchmark times: codes and scales of
    every weight bit-exact, routing and the output of sampled rows (all rows
    on the decode and capacity layers; seeded rows with the first and last
    token on the prefill (512) and DeepSeek (256: 2048 routed rows, every
    expert touched) layers) against the oracle."""
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, device=torch.device("cuda"))
    sel = None
    if rows is not None:
        sel = np.sort(np.random.default_rng(cfg.seed).choice(cfg.T, size=rows, replace=False))
        sel[0], sel[-1] = 0, cfg.T - 1
    print(name, down, parity.check_layer_fp8(cfg, inp, sel, down=down))
    del inp
    torch.cuda.empty_cache()


def test_layer_fp8_with_reroute_matches_stage_path():
    """FP8 gate/up with overflow re-routing: the same rows go to the FFN."""
    cfg = SMALL["capacity_small"]
    inp = make_inputs(cfg, device=torch.device("cuda"))
    mk = lambda fp8: B.MoELayer(inp.W_g, inp.W_gate, inp.W_up, inp.W_down, cfg.k, bias=inp.bias,
                                capacity_factor=cfg.cf, reroute_rounds=2, fp8=fp8)
    a, b = mk(False), mk(True)
    ya, yb = a(inp.x), b(inp.x)
    torch.cuda.synchronize()
    for key in ("topk_idx", "counts", "inv_pos", "rerouted"):
        assert torch.equal(a.last[key], b.last[key]), key
    rel = float((yb - ya).norm() / ya.norm())
    assert rel < 0.1, rel
