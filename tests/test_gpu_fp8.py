"""GPU parity of the FP8 (E4M3) gate/up path against the fp64 oracle.

Quantisation is byte work: the codes and scales must match the oracle's bit
for bit.  The FFN and the layer are compared with the oracle's fp64 layer on
the same E4M3 values (its own quantisation of the inputs), within the bf16
layer tolerance (h is rounded to bf16 between the GEMMs, as in the bf16 path).
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


def _fp8_fetch(inp, qw):
    (qg, sg), (qu, su) = qw[:2]
    qd = qw[2] if len(qw) > 2 else None

    def fetch(e):
        w = (qg[e], sg[e], qu[e], su[e], inp.W_down[e].cpu())
        return w if qd is None else w + (qd[0][e], qd[1][e])
    return fetch


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


def _check_fp8_layer(cfg, inp, rows=None, down=False):
    layer = B.MoELayer(inp.W_g, inp.W_gate, inp.W_up, inp.W_down, cfg.k, bias=inp.bias,
                       Ws_gate=inp.Ws_gate, Ws_up=inp.Ws_up, Ws_down=inp.Ws_down,
                       capacity_factor=cfg.cf, fp8=True, fp8_down=down)
    y = layer(inp.x)
    torch.cuda.synchronize()
    out = layer.last
    assert int(out["device_status"].item()) == 0
    # the layer's quantised weights are the oracle's, byte for byte
    qw = [oracle.quantize_weights_e4m3(inp.W_gate.cpu()), oracle.quantize_weights_e4m3(inp.W_up.cpu())]
    if down:
        qw.append(oracle.quantize_weights_e4m3(inp.W_down.cpu()))
    for (qo, so), i in zip(qw, (0, 2, 4)):
        np.testing.assert_array_equal(layer.fp8[i].cpu().numpy(), qo)
        np.testing.assert_array_equal(layer.fp8[i + 1].cpu().numpy(), so)
    x_c = inp.x.cpu()
    lo = oracle.router_logits(x_c, inp.W_g.cpu(), None if inp.bias is None else inp.bias.cpu())
    idx_o, w_o = oracle.topk_softmax(lo, cfg.k)
    idx_g = out["topk_idx"].cpu().numpy()
    flipped = np.unique(np.nonzero(np.sort(idx_g, 1) != np.sort(idx_o, 1))[0])
    C = oracle.capacity(cfg.cf, cfg.T, cfg.k, cfg.N)
    g_o = oracle.group(idx_o, cfg.N, C)
    sel = np.arange(cfg.T) if rows is None else np.asarray(rows)
    skip = np.zeros(cfg.T, dtype=bool)
    skip[flipped] = True
    if C > 0 and flipped.size:
        ex = np.unique(np.concatenate([idx_g[flipped].ravel(), idx_o[flipped].ravel()]))
        skip |= np.isin(idx_o, ex).any(1)
    assert int(skip[sel].sum()) <= max(2, len(sel) // 100)
    sel = sel[~skip[sel]]
    qx, sx = oracle.quantize_rows_e4m3(x_c)
    shared = None if not cfg.fs else (inp.Ws_gate.cpu(), inp.Ws_up.cpu(), inp.Ws_down.cpu())
    y_o = oracle.forward_rows_fp8(qx[sel], sx[sel], idx_o[sel], w_o[sel], g_o["inv_pos"][sel],
                                  _fp8_fetch(inp, qw), shared=shared,
                                  x_rows=x_c[torch.as_tensor(sel)])
    y_g = y[torch.as_tensor(sel, device=y.device)].float().cpu().numpy()
    max_abs, fro = parity.assert_y_close(y_g, y_o, "bf16")
    # how far E4M3 moves the layer from its bf16 definition (reported; a
    # loose bound catches a lost or misplaced scale)
    y_b = oracle.forward_rows(x_c[torch.as_tensor(sel)], idx_o[sel], w_o[sel],
                              g_o["inv_pos"][sel], parity.fetcher(inp), shared=shared)
    q_err = float(np.linalg.norm(y_g - y_b) / max(np.linalg.norm(y_b), 1e-30))
    assert q_err < (0.15 if down else 0.1), f"FP8 layer {q_err:.3f} (rel-fro) away from the bf16 layer"
    return dict(max_abs=max_abs, rel_fro=fro, fp8_vs_bf16_rel_fro=q_err, rows=len(sel))


@pytest.mark.parametrize("down", [False, True], ids=["bf16_down", "fp8_down"])
@pytest.mark.parametrize("name", list(SMALL))
def test_layer_fp8_reduced(name, down):
    cfg = SMALL[name]
    if down and cfg.f % 16:
        pytest.skip("an E4M3 down projection needs f % 16 == 0")
    inp = make_inputs(cfg, device=torch.device("cuda"))
    print(name, down, _check_fp8_layer(cfg, inp, down=down))


@pytest.mark.parametrize("down", [False, True], ids=["bf16_down", "fp8_down"])
@pytest.mark.parametrize("name,rows", [("mixtral_decode", None), ("capacity", 256)])
def test_layer_fp8_full_size(name, rows, down):
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, device=torch.device("cuda"))
    sel = None
    if rows is not None:
        sel = np.sort(np.random.default_rng(cfg.seed).choice(cfg.T, size=rows, replace=False))
    print(name, down, _check_fp8_layer(cfg, inp, sel, down=down))
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
