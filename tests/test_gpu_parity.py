"""GPU parity: every stage and the whole layer, through the C ABI, against the
fp64 CPU oracle, on seeded synthetic layers.

Reduced layers span several tiles and ragged tails and are checked on every
row; the full-size workloads (the launch configuration the benchmark times)
are checked on all tokens for routing and grouping, and for the layer output
on every row of the decode and capacity layers and on a seeded 1024-token
subset of the prefill and DeepSeek layers.
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

REDUCED = {
    "tiny": CONFIGS["tiny"],
    "mixtral_small": MoEConfig("mixtral_small", T=300, d=512, f=1024, N=8, k=2, bias_std=0.5,
                               seed=31),
    "deepseek_small": MoEConfig("deepseek_small", T=200, d=256, f=256, N=256, k=8, fs=256,
                                seed=41),
    "capacity_small": MoEConfig("capacity_small", T=512, d=256, f=192, N=32, k=2, cf=1.25,
                                bias_std=1.0, seed=51),
    "f32_wide": MoEConfig("f32_wide", T=129, d=128, f=72, N=16, k=3, bias_std=0.3, dtype="f32",
                          seed=61),
    "one_token": MoEConfig("one_token", T=1, d=64, f=64, N=8, k=2, seed=71),
    "three_tokens_shared": MoEConfig("three_tokens_shared", T=3, d=128, f=128, N=16, k=4,
                                     fs=64, seed=72),
    "ragged_257": MoEConfig("ragged_257", T=257, d=136, f=200, N=8, k=2, seed=73),
    "k_equals_n": MoEConfig("k_equals_n", T=64, d=64, f=64, N=4, k=4, seed=74),
    "many_rows": MoEConfig("many_rows", T=2048, d=256, f=320, N=4, k=2, bias_std=1.0, seed=75),
    "odd_dims": MoEConfig("odd_dims", T=173, d=200, f=136, N=6, k=2, fs=72, seed=76),
    # ~300 rows per expert: tiles of one 256-row and one <=64-row token sub-tile
    "wide_tiles": MoEConfig("wide_tiles", T=1200, d=256, f=192, N=8, k=2, bias_std=0.4,
                            seed=77),
}


def _cuda():
    return torch.device("cuda")


@pytest.mark.parametrize("name", list(REDUCED))
def test_layer_reduced(name):
    inp = make_inputs(REDUCED[name], device=_cuda())
    res = parity.check_layer(inp)
    print(name, res)


@pytest.mark.parametrize("name,rows", [("mixtral_decode", None), ("capacity", None),
                                       ("mixtral_prefill", 1024), ("deepseek", 1024)])
def test_layer_full_size(name, rows):
    """The layers the benchmark times, at full size: routing and grouping on
    every token; the output on every row of the decode and capacity layers and
    on a seeded subset of 1024 tokens (with the first and the last) of the
    prefill and DeepSeek layers -- each token's output row depends on that
    token alone, so the subset's rows are exact comparisons."""
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, device=_cuda())
    sel = None
    if rows is not None:
        sel = np.sort(np.random.default_rng(cfg.seed).choice(cfg.T, size=rows, replace=False))
        sel[0], sel[-1] = 0, cfg.T - 1
    res = parity.check_layer(inp, rows=sel)
    print(name, res)
    del inp
    torch.cuda.empty_cache()


def test_bf16_output_variant():
    inp = make_inputs(REDUCED["mixtral_small"], device=_cuda())
    y32, _ = parity.run_forward(inp, y_dtype=torch.float32)
    y16, _ = parity.run_forward(inp, y_dtype=torch.bfloat16)
    assert torch.equal(y16, y32.to(torch.bfloat16))


# --------------------------------------------------------------- stages ----
@pytest.mark.parametrize("name", ["tiny", "mixtral_small", "deepseek_small", "capacity_small",
                                  "f32_wide"])
def test_router_stage(name):
    cfg = REDUCED[name]
    inp = make_inputs(cfg, device=_cuda())
    logits = torch.empty((cfg.T, cfg.N), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, w = B.moe_router_topk(inp.x, inp.W_g, cfg.k, bias=inp.bias, logits=logits,
                               device_status=status)
    torch.cuda.synchronize()
    lo = oracle.router_logits(inp.x.cpu(), inp.W_g.cpu(),
                              None if inp.bias is None else inp.bias.cpu())
    rep = parity.check_routing(lo, idx.cpu().numpy(), w.cpu().numpy(), cfg.k)
    assert not rep.unexplained and rep.w_max_rel <= parity.W_REL
    assert int(status.item()) == 0
    # fp32 logits against fp64: within a few ulps of the accumulation bound
    assert np.abs(logits.cpu().double().numpy() - lo).max() < 1e-4


def test_router_ties_and_nan():
    """Exact ties go to the lower expert id; NaN logits rank last and are flagged."""
    T, d, N, k = 4, 64, 8, 3
    x = torch.zeros((T, d), dtype=torch.float32, device="cuda")
    Wg = torch.zeros((d, N), dtype=torch.float32, device="cuda")
    bias = torch.tensor([1.0, 2.0, 2.0, 0.5, 2.0, -1.0, 0.0, 3.0], device="cuda")
    idx, w = B.moe_router_topk(x, Wg, k, bias=bias)
    torch.cuda.synchronize()
    assert idx.cpu().tolist() == [[7, 1, 2]] * T
    bias2 = torch.tensor([float("nan"), 2.0, 2.0, 0.5, 2.0, -1.0, 0.0, 3.0], device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx2, _ = B.moe_router_topk(x, Wg, 8, bias=bias2, device_status=status)
    torch.cuda.synchronize()
    assert idx2.cpu().tolist()[0] == [7, 1, 2, 4, 3, 6, 5, 0]
    assert int(status.item()) & B.MOE_DEV_NAN_LOGIT


@pytest.mark.parametrize("T,N,k,cap,skew", [(1000, 8, 2, 0, 0.0), (2049, 256, 8, 0, 0.5),
                                            (4096, 128, 2, 80, 3.0), (300, 4, 4, 0, 0.0),
                                            (777, 32, 3, 50, 2.0), (1, 8, 2, 0, 0.0),
                                            (513, 64, 1, 1, 0.0), (256, 256, 8, 0, 0.5),
                                            (200, 32, 3, 5, 2.0), (64, 1024, 2, 0, 1.0),
                                            (32, 8, 2, 0, 0.0)])
def test_permute_stage_bit_exact(T, N, k, cap, skew):
    rng = np.random.default_rng(T + N)
    p = np.exp(skew * rng.normal(size=N)); p /= p.sum()
    idx = np.stack([rng.choice(N, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    d = 64
    x = torch.randn((T, d), device="cuda").to(torch.bfloat16)
    w = torch.rand((T, k), device="cuda")
    out = B.moe_permute(torch.from_numpy(idx).cuda(), N, x=x, topk_w=w, capacity=cap)
    torch.cuda.synchronize()
    g = oracle.group(idx, N, cap)
    A = g["offsets"][-1]
    np.testing.assert_array_equal(out["counts"].cpu().numpy(), g["counts"])
    np.testing.assert_array_equal(out["offsets"].cpu().numpy(), g["offsets"])
    np.testing.assert_array_equal(out["inv_pos"].cpu().numpy(), g["inv_pos"])
    np.testing.assert_array_equal(out["perm_token"][:A].cpu().numpy(), g["perm_token"])
    assert int(out["dropped"].item()) == g["dropped"]
    pt = torch.from_numpy(g["perm_token"].astype(np.int64)).cuda()
    assert torch.equal(out["x_perm"][:A], x[pt])
    slots = torch.from_numpy(g["perm_slot"].astype(np.int64)).cuda()
    assert torch.equal(out["row_scale"][:A], w[pt, slots])


def test_permute_all_tokens_one_expert_and_empty_experts():
    T, N, k = 1000, 16, 1
    idx = np.full((T, k), 5, dtype=np.int32)
    out = B.moe_permute(torch.from_numpy(idx).cuda(), N, capacity=0)
    torch.cuda.synchronize()
    off = out["offsets"].cpu().numpy()
    assert off.tolist() == [0] * 6 + [T] * 11
    assert out["perm_token"][:T].cpu().tolist() == list(range(T))


def test_permute_bad_expert_id_sets_status():
    idx = torch.tensor([[0, 1], [9, 2], [-3, 0]], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = B.moe_permute(idx, 4, capacity=0, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & B.MOE_DEV_BAD_EXPERT_ID
    g = oracle.group(idx.cpu().numpy(), 4, 0)
    np.testing.assert_array_equal(out["inv_pos"].cpu().numpy(), g["inv_pos"])
    assert int(out["dropped"].item()) == 2


def test_permute_repeat_bit_identical():
    rng = np.random.default_rng(5)
    idx = torch.from_numpy(np.stack([rng.choice(256, 8, replace=False) for _ in range(3000)])
                           .astype(np.int32)).cuda()
    a = B.moe_permute(idx, 256, capacity=0)
    b = B.moe_permute(idx, 256, capacity=0)
    torch.cuda.synchronize()
    for key in ("counts", "offsets", "inv_pos", "perm_token"):
        assert torch.equal(a[key], b[key])


@pytest.mark.parametrize("name", ["tiny", "mixtral_small", "deepseek_small", "f32_wide",
                                  "many_rows", "odd_dims", "ragged_257", "wide_tiles"])
def test_expert_ffn_stage(name):
    """y_perm rows = row_scale * SwiGLU_e(x_perm) against the oracle's expert
    rows; the stage's inputs (x_perm, offsets, row scales) are built on the
    CPU from the oracle's routing and grouping of the layer's inputs."""
    cfg = REDUCED[name]
    inp = make_inputs(cfg, device=_cuda())
    x_c = inp.x.cpu()
    lo = oracle.router_logits(x_c, inp.W_g.cpu(), None if inp.bias is None else inp.bias.cpu())
    idx_o, w_o = oracle.topk_softmax(lo, cfg.k)
    g = oracle.group(idx_o, cfg.N, 0)
    off = g["offsets"]
    pt = torch.from_numpy(g["perm_token"].astype(np.int64))
    xp = x_c[pt].contiguous()
    rs = torch.from_numpy(w_o[g["perm_token"], g["perm_slot"]]).float()
    y_perm = B.moe_expert_ffn(xp.cuda(), torch.from_numpy(off).cuda(), inp.W_gate, inp.W_up,
                              inp.W_down, row_scale=rs.cuda())
    torch.cuda.synchronize()
    ref = np.zeros((off[-1], cfg.d))
    for e in range(cfg.N):
        if off[e + 1] > off[e]:
            ref[off[e]:off[e + 1]] = oracle.expert_rows(inp.W_gate[e].cpu(), inp.W_up[e].cpu(),
                                                        inp.W_down[e].cpu(), xp[off[e]:off[e + 1]])
    ref *= rs.double().numpy()[:, None]
    parity.assert_y_close(y_perm[:off[-1]].float().cpu().numpy(), ref, cfg.dtype)


@pytest.mark.parametrize("counts", [
    # ~340 rows per expert: 256-row tiles; experts split into 2-4 tiles
    [0, 1, 256, 257, 288, 320, 321, 600, 641, 100, 0, 960],
    # ~280 rows per expert: wide tiles (two balanced sub-tiles above 160 rows)
    [0, 1, 160, 161, 255, 256, 257, 288, 320, 321, 600, 641, 100, 0, 960, 200],
])
def test_expert_ffn_crafted_counts(counts):
    """Expert sizes on every tiling edge of the grouped GEMMs: empty, one row,
    one sub-tile, two sub-tiles, and experts split into two or three tiles."""
    N, d, f = len(counts), 256, 192
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    A = int(off[-1])
    g = torch.Generator().manual_seed(78)
    xp = (torch.randn((A, d), generator=g) * 0.5).to(torch.bfloat16)
    Wg = (torch.randn((N, d, f), generator=g) * d ** -0.5).to(torch.bfloat16)
    Wu = (torch.randn((N, d, f), generator=g) * d ** -0.5).to(torch.bfloat16)
    Wd = (torch.randn((N, f, d), generator=g) * f ** -0.5).to(torch.bfloat16)
    rs = torch.rand((A,), generator=g) + 0.5
    y = B.moe_expert_ffn(xp.cuda(), torch.from_numpy(off).cuda(), Wg.cuda(), Wu.cuda(),
                         Wd.cuda(), row_scale=rs.cuda())
    torch.cuda.synchronize()
    ref = np.zeros((A, d))
    for e in range(N):
        if counts[e]:
            ref[off[e]:off[e + 1]] = oracle.expert_rows(Wg[e], Wu[e], Wd[e], xp[off[e]:off[e + 1]])
    ref *= rs.double().numpy()[:, None]
    parity.assert_y_close(y[:A].float().cpu().numpy(), ref, "bf16")


def test_combine_stage():
    T, k, d = 333, 3, 128
    A = T * k
    y_perm = torch.randn((A, d), device="cuda").to(torch.bfloat16)
    inv = torch.randperm(A, device="cuda").int().view(T, k)
    inv[::7, 1] = -1
    shared = torch.randn((T, d), device="cuda").to(torch.bfloat16)
    y = B.moe_combine(y_perm, inv, shared_y=shared)
    torch.cuda.synchronize()
    ones = np.ones((T, k))
    invn = inv.cpu().numpy()
    o = y_perm.double().cpu().numpy()[np.maximum(invn, 0)]
    ref = oracle.combine_rows(invn, ones, o, shared.double().cpu().numpy())
    np.testing.assert_allclose(y.cpu().double().numpy(), ref, rtol=1e-6, atol=1e-5)


@pytest.mark.parametrize("y_dtype", [torch.float32, torch.bfloat16])
def test_forward_equals_stage_calls(y_dtype):
    """moe_forward equals, bit for bit, its stage entry points run one after
    another (router, dispatch, routed FFN, shared-expert FFN, combine)."""
    cfg = REDUCED["deepseek_small"]
    inp = make_inputs(cfg, device=_cuda())
    y_forward, outs = parity.run_forward(inp, y_dtype=y_dtype)
    A_max = cfg.T * cfg.k
    idx, w = B.moe_router_topk(inp.x, inp.W_g, cfg.k, bias=inp.bias)
    perm = B.moe_permute(idx, cfg.N, x=inp.x, topk_w=w, capacity=0, A_max=A_max)
    y_perm = B.moe_expert_ffn(perm["x_perm"], perm["offsets"], inp.W_gate, inp.W_up, inp.W_down,
                              row_scale=perm["row_scale"], A_max=A_max)
    sh_off = torch.tensor([0, cfg.T], dtype=torch.int32, device="cuda")
    ys = B.moe_expert_ffn(inp.x, sh_off, inp.Ws_gate[None], inp.Ws_up[None], inp.Ws_down[None])
    y_staged = B.moe_combine(y_perm, perm["inv_pos"], shared_y=ys, y_dtype=y_dtype)
    torch.cuda.synchronize()
    assert torch.equal(outs["topk_idx"], idx)
    assert torch.equal(y_forward, y_staged)


def test_forward_repeat_bit_identical():
    inp = make_inputs(REDUCED["deepseek_small"], device=_cuda())
    y1, o1 = parity.run_forward(inp)
    y2, o2 = parity.run_forward(inp)
    assert torch.equal(y1, y2)
    for key in ("topk_idx", "topk_w", "counts", "offsets", "inv_pos"):
        assert torch.equal(o1[key], o2[key])


def test_host_io_variant_matches_device_call():
    cfg = REDUCED["capacity_small"]
    inp = make_inputs(cfg, device=_cuda())
    y_dev, _ = parity.run_forward(inp, logits=False)
    layer = B.MoELayer(inp.W_g, inp.W_gate, inp.W_up, inp.W_down, cfg.k, bias=inp.bias,
                       capacity_factor=cfg.cf)
    x_stage = torch.empty_like(inp.x)
    y_stage = torch.empty((cfg.T, cfg.d), dtype=torch.float32, device="cuda")
    o = layer.outputs_for(cfg.T, inp.x.device)
    a = layer.args(x_stage, y_stage, o)
    x_host = inp.x.cpu().pin_memory()
    y_host = torch.empty((cfg.T, cfg.d), dtype=torch.float32).pin_memory()
    B.moe_forward_host_io(a, x_host, y_host, layer.workspace(a, inp.x.device))
    torch.cuda.synchronize()
    assert torch.equal(y_host, y_dev.cpu())


def _stats_close(got, ref, rel=2e-5):
    for key in ("entropy_bits", "entropy_max_bits", "top3_share", "max_share", "freq_cv"):
        assert got[key] == pytest.approx(ref[key], rel=rel, abs=1e-6), key
    if np.isnan(ref["balance"]):
        assert np.isnan(got["balance"])
    else:
        assert got["balance"] == pytest.approx(ref["balance"], rel=rel), "balance"
    assert got["top3"] == ref["top3"].tolist()


@pytest.mark.parametrize("T,N,skew,with_logits", [
    (1000, 8, 1.0, True), (8192, 256, 0.5, True), (4096, 128, 3.0, True), (513, 1024, 1.0, True),
    (300, 2, 0.0, True), (1, 1, 0.0, True), (0, 16, 0.0, False), (2049, 64, 2.0, False)])
def test_routing_stats_stage(T, N, skew, with_logits):
    """Synthetic counts and logits (test inputs) on both sides; counts with ties."""
    rng = np.random.default_rng(T + N)
    p = np.exp(skew * rng.normal(size=N))
    counts = rng.multinomial(2 * max(T, 1), p / p.sum()).astype(np.int32)
    half = N // 2
    counts[half:2 * half] = counts[:half]            # equal counts: the tie rule decides
    logits = (rng.normal(size=(T, N)) * 2).astype(np.float32) if with_logits else None
    st, freq, prob = B.moe_routing_stats(torch.from_numpy(counts).cuda(),
                                         None if logits is None else torch.from_numpy(logits).cuda())
    torch.cuda.synchronize()
    got = B.routing_stats_dict(st)
    ref = oracle.routing_stats(counts, None if logits is None else logits.astype(np.float64))
    _stats_close(got, ref)
    assert got["assignments"] == int(counts.sum())
    np.testing.assert_allclose(freq.cpu().numpy(), ref["freq"], rtol=1e-6, atol=0)
    if with_logits:
        np.testing.assert_allclose(prob.cpu().numpy(), ref["prob_mean"], rtol=2e-5, atol=1e-9)


def test_routing_stats_no_assignments_and_one_expert():
    z = torch.zeros(8, dtype=torch.int32, device="cuda")
    st, _, _ = B.moe_routing_stats(z)
    got = B.routing_stats_dict(st)
    assert got["entropy_bits"] == 0 and got["max_share"] == 0 and got["freq_cv"] == 0
    assert got["top3"] == [0, 1, 2]
    one = torch.tensor([0, 0, 0, 9, 0, 0, 0, 0], dtype=torch.int32, device="cuda")
    got = B.routing_stats_dict(B.moe_routing_stats(one)[0])
    assert got["entropy_bits"] == 0 and got["max_share"] == 1 and got["top3"] == [3, 0, 1]
    assert got["freq_cv"] == pytest.approx(np.sqrt(7.0), rel=1e-6)


@pytest.mark.parametrize("name", ["mixtral_small", "deepseek_small", "capacity_small"])
def test_routing_stats_on_a_layer(name):
    """Router logits and pre-capacity counts from the library, against the
    oracle's statistics of the oracle's own routing of the same inputs."""
    cfg = REDUCED[name]
    inp = make_inputs(cfg, device=_cuda())
    logits = torch.empty((cfg.T, cfg.N), dtype=torch.float32, device="cuda")
    idx, w = B.moe_router_topk(inp.x, inp.W_g, cfg.k, bias=inp.bias, logits=logits)
    C = oracle.capacity(cfg.cf, cfg.T, cfg.k, cfg.N)
    perm = B.moe_permute(idx, cfg.N, capacity=C)
    st, _, prob = B.moe_routing_stats(perm["counts"], logits)
    torch.cuda.synchronize()
    got = B.routing_stats_dict(st)
    lo = oracle.router_logits(inp.x.cpu(), inp.W_g.cpu(), None if inp.bias is None else inp.bias.cpu())
    idx_o, _ = oracle.topk_softmax(lo, cfg.k)
    g = oracle.group(idx_o, cfg.N, C)
    np.testing.assert_array_equal(perm["counts"].cpu().numpy(), g["counts"])
    ref = oracle.routing_stats(g["counts"], lo)
    _stats_close(got, ref, rel=1e-4)
    np.testing.assert_allclose(prob.cpu().numpy(), ref["prob_mean"], rtol=1e-4, atol=1e-8)


def _reroute_inputs(T, N, k, R, skew, seed):
    """Test inputs built on the CPU: logits with a skew towards some experts,
    each token's k+R candidates by rank and the softmax over them (fp32)."""
    rng = np.random.default_rng(seed)
    lg = rng.normal(size=(T, N)) + skew * rng.normal(size=N)
    cand, w = oracle.topk_softmax(lg, k + R)
    return lg, cand.astype(np.int32), w.astype(np.float32)


# N <= 512 with every 256-token chunk resident at once: one cooperative
# launch (40000 tokens = 157 chunks, more than one CTA on some SMs); N = 600:
# the round-by-round launches.
@pytest.mark.parametrize("T,N,k,R,cap,skew", [(1000, 8, 2, 2, 200, 1.0), (4096, 128, 2, 2, 80, 1.0),
                                              (777, 32, 3, 4, 50, 2.0), (300, 4, 1, 3, 60, 1.5),
                                              (513, 64, 1, 1, 1, 0.0), (1, 8, 2, 2, 1, 0.0),
                                              (40000, 64, 2, 3, 700, 1.5),
                                              (3000, 512, 4, 2, 12, 1.0),
                                              (2000, 600, 2, 2, 5, 1.0)])
def test_permute_reroute_stage(T, N, k, R, cap, skew):
    lg, cand, cw = _reroute_inputs(T, N, k, R, skew, T + N + R)
    d = 64
    x = torch.randn((T, d), device="cuda").to(torch.bfloat16)
    out = B.moe_permute_reroute(torch.from_numpy(cand).cuda(), torch.from_numpy(cw).cuda(), N, k,
                                cap, x=x, demand=True)
    torch.cuda.synchronize()
    ref = oracle.reroute(cand, k, R, N, cap, logits=lg)
    np.testing.assert_array_equal(out["final_idx"].cpu().numpy(), ref["final_idx"])
    assert int(out["rerouted"].item()) == ref["rerouted"]
    np.testing.assert_allclose(out["final_w"].cpu().numpy(), ref["final_w"], rtol=2e-6, atol=1e-7)
    np.testing.assert_array_equal(out["demand"].cpu().numpy(), np.bincount(cand[:, :k].ravel(),
                                                                           minlength=N))
    g = oracle.group(ref["final_idx"], N, 0)
    A = int(g["offsets"][-1])
    np.testing.assert_array_equal(out["counts"].cpu().numpy(), g["counts"])
    np.testing.assert_array_equal(out["offsets"].cpu().numpy(), g["offsets"])
    np.testing.assert_array_equal(out["inv_pos"].cpu().numpy(), g["inv_pos"])
    np.testing.assert_array_equal(out["perm_token"][:A].cpu().numpy(), g["perm_token"])
    assert int(out["dropped"].item()) == T * k - A
    pt = torch.from_numpy(g["perm_token"].astype(np.int64)).cuda()
    assert torch.equal(out["x_perm"][:A], x[pt])
    slots = torch.from_numpy(g["perm_slot"].astype(np.int64)).cuda()
    assert torch.equal(out["row_scale"][:A], out["final_w"][pt, slots])


def test_permute_reroute_repeat_bit_identical():
    _, cand, cw = _reroute_inputs(4096, 128, 2, 3, 2.0, 9)
    c, w = torch.from_numpy(cand).cuda(), torch.from_numpy(cw).cuda()
    a = B.moe_permute_reroute(c, w, 128, 2, 40)
    b = B.moe_permute_reroute(c, w, 128, 2, 40)
    torch.cuda.synchronize()
    for key in ("final_idx", "final_w", "counts", "offsets", "inv_pos", "rerouted"):
        assert torch.equal(a[key], b[key]), key
    A = int(a["offsets"][-1].item())
    assert torch.equal(a["perm_token"][:A], b["perm_token"][:A])
    assert torch.equal(a["row_scale"][:A], b["row_scale"][:A])


@pytest.mark.parametrize("name,R", [("capacity_small", 2), ("capacity_small", 1),
                                    ("mixtral_small", 2), ("capacity", 2)])
def test_layer_with_reroute(name, R):
    """moe_forward with overflow re-routing against the oracle: routing to k+R
    candidates, re-routing rounds, grouping and the layer output, all from the
    oracle's own fp64 logits."""
    cfg = REDUCED[name] if name in REDUCED else CONFIGS[name]
    cf = cfg.cf if cfg.cf > 0 else 0.5
    inp = make_inputs(cfg, device=_cuda())
    layer = B.MoELayer(inp.W_g, inp.W_gate, inp.W_up, inp.W_down, cfg.k, bias=inp.bias,
                       capacity_factor=cf, reroute_rounds=R)
    y = layer(inp.x)
    torch.cuda.synchronize()
    out = layer.last
    x_c = inp.x.cpu()
    lo = oracle.router_logits(x_c, inp.W_g.cpu(), None if inp.bias is None else inp.bias.cpu())
    cand, _ = oracle.topk_softmax(lo, cfg.k + R)
    # The candidates' rank order decides the re-routing.  Near-equal logits
    # (1e-4 relative) may rank either way; the library's ranking is compared
    # with the oracle's (nothing of it goes into the oracle): when they agree,
    # every later step must match exactly.
    cand_g, _ = B.moe_router_topk(inp.x, inp.W_g, cfg.k + R, bias=inp.bias)
    cand_g = cand_g.cpu().numpy()
    if not np.array_equal(cand_g, cand):
        srt = np.sort(lo, axis=1)[:, ::-1][:, :cfg.k + R + 1]
        gaps = np.abs(np.diff(srt, axis=1)) < parity.TIE_REL * np.abs(srt[:, :-1])
        diff = np.nonzero((cand_g != cand).any(1))[0]
        assert gaps[diff].any(1).all(), "candidate ranks differ beyond near-ties"
        pytest.skip(f"{diff.size} near-tie token(s) ranked the other way; exact re-routing not comparable")
    C = oracle.capacity(cf, cfg.T, cfg.k, cfg.N)
    ref = oracle.reroute(cand, cfg.k, R, cfg.N, C, logits=lo)
    np.testing.assert_array_equal(out["topk_idx"].cpu().numpy(), ref["final_idx"])
    assert int(out["rerouted"].item()) == ref["rerouted"]
    np.testing.assert_allclose(out["topk_w"].cpu().numpy(), ref["final_w"], rtol=1e-5)
    g = oracle.group(ref["final_idx"], cfg.N, 0)
    np.testing.assert_array_equal(out["counts"].cpu().numpy(), g["counts"])
    np.testing.assert_array_equal(out["inv_pos"].cpu().numpy(), g["inv_pos"])
    assert int(out["dropped"].item()) == cfg.T * cfg.k - int(g["offsets"][-1])
    idx = np.where(ref["final_idx"] >= 0, ref["final_idx"], 0)
    sel = np.arange(cfg.T)           # every row (the full capacity layer too)
    y_o = oracle.forward_rows(x_c[torch.as_tensor(sel)], idx[sel], ref["final_w"][sel],
                              g["inv_pos"][sel], parity.fetcher(inp))
    parity.assert_y_close(y[torch.as_tensor(sel, device=y.device)].float().cpu().numpy(), y_o,
                          cfg.dtype)
    print(name, R, "rerouted", ref["rerouted"], "dropped", int(out["dropped"].item()))


@pytest.mark.parametrize("name,R", [("capacity_small", 0), ("deepseek_small", 0),
                                    ("capacity_small", 2)])
def test_forward_captures_into_a_cuda_graph(name, R):
    """moe_forward only enqueues work (no sync, no host read-back), so it can
    be captured into a CUDA graph; a replay gives the direct call's output.
    With re-routing the graph holds the cooperative single-launch rounds."""
    cfg = REDUCED[name]
    inp = make_inputs(cfg, device=_cuda())
    layer = B.MoELayer(inp.W_g, inp.W_gate, inp.W_up, inp.W_down, cfg.k, bias=inp.bias,
                       Ws_gate=inp.Ws_gate, Ws_up=inp.Ws_up, Ws_down=inp.Ws_down,
                       capacity_factor=cfg.cf, reroute_rounds=R)
    y = torch.empty((cfg.T, cfg.d), dtype=torch.float32, device="cuda")
    o = layer.outputs_for(cfg.T, y.device)
    a = layer.args(inp.x, y, o)
    ws = layer.workspace(a, y.device)
    B.moe_forward(a, ws)
    torch.cuda.synchronize()
    y_direct = y.clone()
    y.zero_()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        B.moe_forward(a, ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        B.moe_forward(a, ws)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, y_direct)


@pytest.mark.parametrize("name,chunks", [("mixtral_small", 3), ("deepseek_small", 2),
                                         ("mixtral_small", 0), ("capacity_small", 4)])
def test_overlapped_host_io_equals_forward(name, chunks):
    """Host buffers in and out with the copies overlapped with token chunks of
    the layer: y equals the single device call bit for bit (each token's row
    depends on that token alone; with a capacity the call runs one chunk)."""
    cfg = REDUCED[name]
    inp = make_inputs(cfg, device=_cuda())
    layer = B.MoELayer(inp.W_g, inp.W_gate, inp.W_up, inp.W_down, cfg.k, bias=inp.bias,
                       Ws_gate=inp.Ws_gate, Ws_up=inp.Ws_up, Ws_down=inp.Ws_down,
                       capacity_factor=cfg.cf)
    y_dev = layer(inp.x)
    x_stage = torch.empty_like(inp.x)
    y = torch.empty_like(y_dev)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = layer.args(x_stage, y, {"device_status": st})
    ws = layer.workspace(a, y.device)
    x_host = inp.x.cpu().pin_memory()
    y_host = torch.full(tuple(y.shape), float("nan"), dtype=y.dtype).pin_memory()
    B.moe_forward_host_io_overlapped(a, x_host, y_host, ws, chunks)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(y_host, y_dev.cpu())
