"""Pins for the fp64 CPU oracle, against what the pages and the mathematics fix.

None of these re-derive the oracle's formulas: each checks a worked example
printed on the pages, a closed form, an invariant, a special case with a known
answer, or a brute-force count on tiny inputs, chosen so that a dropped term,
a wrong sign, a wrong index or a transposed operand anywhere in the oracle
fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_mixture_experts_63_b300.configs import TINY, CAPACITY
from sparse_mixture_experts_63_b300.inputs import make_inputs

from conftest import GOLDEN


def golden(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def rand_f32(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).float()


# ---------------------------------------------------------------- routing ---
def test_worked_example_step6_weights():
    """Experts 2 and 5 chosen with scores 0.6 / 0.4 ("動態 token 路由", step 6)."""
    gd = golden("p1_step6_combine.json")
    N, k = 8, 2
    logits = np.full((1, N), -3.0)
    logits[0, 5] = 0.25
    logits[0, 2] = 0.25 + math.log(1.5)
    idx, w = oracle.topk_softmax(logits, k)
    assert list(idx[0]) == gd["experts"]
    np.testing.assert_allclose(w[0], gd["weights"], rtol=0, atol=1e-15)
    # and the combine takes 60% / 40% of the two experts' outputs
    o = np.array([[[1.0, 0.0, 2.0], [0.0, 1.0, -3.0]]])
    y = oracle.combine_rows(np.array([[0, 1]]), w, o)
    np.testing.assert_allclose(y[0], [0.6, 0.4, 0.6 * 2.0 - 0.4 * 3.0], atol=1e-15)


def test_combine_ignores_dropped_slots():
    """A dropped slot (row -1) adds nothing even when an output sits behind it,
    and the kept weight is not renormalised."""
    o = np.array([[[1.0, 2.0], [100.0, 100.0]], [[5.0, 0.0], [0.0, 7.0]]])
    w = np.array([[0.7, 0.3], [0.5, 0.5]])
    inv = np.array([[3, -1], [-1, -1]])
    sh = np.array([[0.25, 0.5], [1.0, 2.0]])
    y = oracle.combine_rows(inv, w, o, sh)
    np.testing.assert_allclose(y, [[0.7 + 0.25, 1.4 + 0.5], [1.0, 2.0]], atol=1e-15)


def _brute_rank_topk(l, k):
    """Slot j holds the expert whose rank is j, rank(e) = number of experts that
    come before e: larger logit, or equal logit and smaller id (NaN lowest)."""
    key = np.where(np.isnan(l), -np.inf, l)
    N = len(l)
    rank = np.array([sum(1 for q in range(N) if key[q] > key[e] or (key[q] == key[e] and q < e))
                     for e in range(N)])
    return [int(np.nonzero(rank == j)[0][0]) for j in range(k)]


@pytest.mark.parametrize("N,k", [(8, 2), (8, 8), (16, 5), (7, 1), (33, 8)])
def test_topk_brute_force_with_ties_and_nan(N, k):
    rng = np.random.default_rng(N * 100 + k)
    T = 200
    logits = rng.integers(-3, 4, size=(T, N)).astype(np.float64)  # many exact ties
    logits[rng.random((T, N)) < 0.05] = np.nan
    idx, w = oracle.topk_softmax(logits, k)
    for t in range(T):
        assert list(idx[t]) == _brute_rank_topk(logits[t], k), t
        assert len(set(idx[t])) == k


def test_gate_weight_invariants():
    rng = np.random.default_rng(7)
    T, N, k = 500, 32, 6
    logits = rng.normal(size=(T, N)) * 3
    idx, w = oracle.topk_softmax(logits, k)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-14)       # sum to 1
    assert np.all(np.diff(w, axis=1) <= 1e-15)                            # follow logit order
    assert np.all(w > 0)
    # shift invariance, and no overflow for huge logits
    idx2, w2 = oracle.topk_softmax(logits + 1000.0, k)
    assert np.array_equal(idx, idx2)
    np.testing.assert_allclose(w, w2, rtol=1e-12)
    # weights depend only on the selected logits: pushing every unselected
    # logit further down changes nothing
    low = logits.copy()
    mask = np.ones_like(low, dtype=bool)
    np.put_along_axis(mask, idx, False, axis=1)
    low[mask] -= 50.0
    idx3, w3 = oracle.topk_softmax(low, k)
    assert np.array_equal(idx, idx3)
    np.testing.assert_allclose(w, w3, rtol=1e-13)
    # k = 1 always has weight exactly 1
    _, w1 = oracle.topk_softmax(logits, 1)
    assert np.all(w1 == 1.0)


def test_page_toy_layer():
    """The toy single-token layer of the inference-learning-path page ("代码"):
    logits x @ router_W, top-k, softmax over the k, weighted sum of x @ W_e.
    Restated with numpy; the oracle's routing must give the same output."""
    N, d, k = 8, 16, 2
    for seed in range(20):
        x = rand_f32((1, d), seed)
        router_W = rand_f32((d, N), 1000 + seed)
        experts_W = rand_f32((N, d, d), 2000 + seed, 1.0 / d).double().numpy()
        xv = x.double().numpy()[0]
        gate = xv @ router_W.double().numpy()
        top = np.argsort(gate)[-k:]
        wt = np.exp(gate[top] - gate[top].max())
        wt /= wt.sum()
        y_toy = sum(wi * (xv @ experts_W[e]) for wi, e in zip(wt, top))
        _, idx, w = oracle.route(x, router_W, k)
        y = sum(w[0, j] * (xv @ experts_W[idx[0, j]]) for j in range(k))
        assert set(idx[0]) == set(top)
        np.testing.assert_allclose(y, y_toy, rtol=1e-12, atol=1e-14)


def test_router_logits_one_hot():
    """A one-hot router forces a known routing: logits are read straight off x."""
    d, N, k = 12, 8, 2
    Wg = torch.zeros(d, N)
    for e in range(N):
        Wg[e, e] = 10.0
    x = torch.zeros(N, d)
    for t in range(N):
        x[t, t] = 2.0
        x[t, (t + 3) % N] = 1.0
        x[t, N + (t % (d - N))] = 7.0     # dims with no router weight
    bias = torch.zeros(N)
    logits = oracle.router_logits(x, Wg, bias)
    for t in range(N):
        exp_l = np.zeros(N)
        exp_l[t] = 20.0
        exp_l[(t + 3) % N] = 10.0
        np.testing.assert_array_equal(logits[t], exp_l)
    idx, w = oracle.topk_softmax(logits, k)
    for t in range(N):
        assert list(idx[t]) == [t, (t + 3) % N]
        np.testing.assert_allclose(w[t], [1 / (1 + math.exp(-10)), 1 / (1 + math.exp(10))],
                                   rtol=1e-14)
    # the bias is added to every token's logits before selection
    b = torch.zeros(N)
    b[(0 + 5) % N] = 25.0
    l2 = oracle.router_logits(x[:1], Wg, b)
    assert l2[0, 5] == 25.0
    idx2, _ = oracle.topk_softmax(l2, k)
    assert list(idx2[0]) == [5, 0]


def test_router_logits_bf16_exact_widening():
    """bf16 inputs are widened exactly: powers of two give exact dot products."""
    d, N = 64, 4
    x = torch.tensor([[2.0 ** (i % 7 - 3) for i in range(d)]], dtype=torch.bfloat16)
    Wg = torch.zeros(d, N, dtype=torch.bfloat16)
    Wg[:, 1] = 1.0
    Wg[3, 2] = -0.5
    l = oracle.router_logits(x, Wg)
    assert l[0, 1] == sum(2.0 ** (i % 7 - 3) for i in range(d))
    assert l[0, 2] == -0.5 * 2.0 ** (3 % 7 - 3)
    assert l[0, 0] == 0.0 and l[0, 3] == 0.0


def test_near_tie_definition():
    l = np.array([[5.0, 4.99999, 1.0, 0.0],      # k=2: 2nd/3rd far apart -> no tie
                  [5.0, 1.0, 1.00001, 0.0],      # 1.0 vs 1.00001: rel gap 1e-5 < 1e-4
                  [5.0, 3.0, 2.0, 0.0]])
    m = oracle.near_tie_tokens(l, 2)
    assert list(m) == [False, True, False]


# ---------------------------------------------------------------- the FFN ---
@pytest.mark.parametrize("s", [1.0, -1.0])
def test_swiglu_closed_form(s):
    """Sparse weights on a non-square expert (d=3, f=2), every non-zero at a
    position no transposed reading reaches.  The output follows from
    SiLU(ln 3) = 0.75 ln 3 and SiLU(-ln 3) = -0.25 ln 3 (sigmoid(ln 3) = 3/4)."""
    d, f = 3, 2
    a32 = float(torch.tensor(math.log(3.0)))   # ln 3 as stored in fp32
    x = torch.tensor([[s, 1.0, 1.5]])
    Wg = torch.zeros(d, f); Wg[0, 0] = a32; Wg[1, 1] = a32     # g = [s ln3, ln3]
    Wu = torch.zeros(d, f); Wu[2, 0] = 2.0; Wu[0, 1] = 1.0     # u = [3, s]
    Wd = torch.zeros(f, d); Wd[0, 1] = -0.5; Wd[1, 2] = 4.0
    out = oracle.expert_rows(Wg, Wu, Wd, x)
    sig0 = 0.75 if s > 0 else 0.25
    h0 = s * a32 * sig0 * 3.0
    h1 = a32 * 0.75 * s
    expect = [0.0, -0.5 * h0, 4.0 * h1]
    assert out[0, 0] == 0.0
    np.testing.assert_allclose(out[0], expect, rtol=2e-7, atol=0)


def test_swiglu_homogeneity_and_zeros():
    d, f = 16, 24
    x = rand_f32((5, d), 3)
    Wg, Wu, Wd = rand_f32((d, f), 4), rand_f32((d, f), 5), rand_f32((f, d), 6)
    o = oracle.expert_rows(Wg, Wu, Wd, x)
    # linear in W_up and in W_down
    np.testing.assert_allclose(oracle.expert_rows(Wg, Wu * 2, Wd, x), 2 * o, rtol=1e-12)
    np.testing.assert_allclose(oracle.expert_rows(Wg, Wu, Wd * -4, x), -4 * o, rtol=1e-12)
    # a zero up or down projection gives zero
    assert np.all(oracle.expert_rows(Wg, Wu * 0, Wd, x) == 0)
    assert np.all(oracle.expert_rows(Wg, Wu, Wd * 0, x) == 0)
    # SiLU(0) = 0: a zero gate projection gives zero too
    assert np.all(oracle.expert_rows(Wg * 0, Wu, Wd, x) == 0)
    # a huge positive gate makes SiLU the identity: out = ((xWg) * (xWu)) Wd
    # on the rows where x Wg >> 0 -- checked through positivity of SiLU(z)/z -> 1
    big = oracle.expert_rows(Wg * 1e4, Wu, Wd, x)
    assert np.all(np.isfinite(big))


# ---------------------------------------------------------------- grouping --
def _random_topk(T, N, k, seed, skew=0.0):
    rng = np.random.default_rng(seed)
    p = np.exp(skew * rng.normal(size=N)); p /= p.sum()
    return np.stack([rng.choice(N, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,N,k,cap", [(64, 8, 2, 0), (257, 16, 3, 0), (300, 8, 2, 40),
                                       (1, 4, 4, 0), (100, 128, 8, 0), (90, 6, 2, 5)])
def test_group_brute_force(T, N, k, cap):
    idx = _random_topk(T, N, k, T + N + k + cap, skew=1.5)
    g = oracle.group(idx, N, cap)
    counts, offsets, inv = g["counts"], g["offsets"], g["inv_pos"]
    assert counts.sum() == T * k
    np.testing.assert_array_equal(counts, np.bincount(idx.ravel(), minlength=N))
    kept = np.minimum(counts, cap) if cap else counts
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(kept)]))
    A = offsets[-1]
    assert g["dropped"] == T * k - A
    # brute force: assignment (t,j) is kept iff fewer than cap earlier tokens chose its expert
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            earlier = int(np.sum(idx[:t] == e))
            if cap and earlier >= cap:
                assert inv[t, j] == -1
            else:
                assert inv[t, j] == offsets[e] + earlier
    # inv_pos is a bijection onto [0, A), consistent with perm_token / perm_slot
    pos = inv[inv >= 0]
    assert sorted(pos.tolist()) == list(range(A))
    for t in range(T):
        for j in range(k):
            p = inv[t, j]
            if p >= 0:
                assert g["perm_token"][p] == t and g["perm_slot"][p] == j
    # each expert's rows hold strictly ascending tokens
    for e in range(N):
        seg = g["perm_token"][offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)


def test_capacity_closed_form():
    gd = golden("capacity_example.json")
    assert oracle.capacity(gd["cf"], gd["T"], gd["k"], gd["N"]) == gd["capacity"]
    assert oracle.capacity(CAPACITY.cf, CAPACITY.T, CAPACITY.k, CAPACITY.N) == 80
    assert oracle.capacity(0.0, 100, 2, 8) == 0          # no limit
    assert oracle.capacity(1.0, 10, 1, 3) == 4           # ceil(10/3)


def test_group_out_of_range_ids_are_dropped():
    idx = np.array([[0, 1], [5, 0], [1, -1]], dtype=np.int32)
    g = oracle.group(idx, 2, 0)
    assert g["inv_pos"][1, 0] == -1 and g["inv_pos"][2, 1] == -1
    assert g["dropped"] == 2 and g["offsets"][-1] == 4


# ---------------------------------------------------------------- the layer -
def _small_layer(seed, T=40, d=16, f=24, N=6, k=2, fs=0, bias=True, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=g)
    L = dict(x=r(T, d).to(dtype), W_g=(r(d, N) / math.sqrt(d)).to(dtype),
             W_gate=(r(N, d, f) / math.sqrt(d)).to(dtype),
             W_up=(r(N, d, f) / math.sqrt(d)).to(dtype),
             W_down=(r(N, f, d) / math.sqrt(f)).to(dtype),
             bias=r(N) * 0.5 if bias else None)
    if fs:
        L.update(Ws_gate=(r(d, fs) / math.sqrt(d)).to(dtype),
                 Ws_up=(r(d, fs) / math.sqrt(d)).to(dtype),
                 Ws_down=(r(fs, d) / math.sqrt(fs)).to(dtype))
    return L


def _fw(L, k, cf=0.0):
    return oracle.moe_forward(L["x"], L["W_g"], L["W_gate"], L["W_up"], L["W_down"], k,
                              bias=L.get("bias"), Ws_gate=L.get("Ws_gate"),
                              Ws_up=L.get("Ws_up"), Ws_down=L.get("Ws_down"),
                              capacity_factor=cf)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_k_equals_N_is_dense_softmax_sum(dtype):
    """With k = N every expert is used: y = sum_e softmax(l)_e E_e(x), the dense
    softmax over all N router scores ("動態 token 路由", step 2) -- no top-k."""
    N, k = 5, 5
    L = _small_layer(11, N=N, dtype=dtype)
    r = _fw(L, k)
    l = oracle.router_logits(L["x"], L["W_g"], L["bias"])
    p = np.exp(l - l.max(1, keepdims=True)); p /= p.sum(1, keepdims=True)
    dense = sum(p[:, e:e + 1] * oracle.expert_rows(L["W_gate"][e], L["W_up"][e],
                                                   L["W_down"][e], L["x"])
                for e in range(N))
    np.testing.assert_allclose(r["y"], dense, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("fs", [0, 20])
def test_sparse_equals_dense_then_mask(fs):
    """Brute force: run every expert on every token, then keep only the top-k
    with their gate weights (unselected experts contribute nothing,
    "什麼是 MoE 模型")."""
    N, k = 6, 2
    L = _small_layer(12, N=N, fs=fs)
    r = _fw(L, k)
    allout = np.stack([oracle.expert_rows(L["W_gate"][e], L["W_up"][e], L["W_down"][e], L["x"])
                       for e in range(N)], axis=1)                  # [T, N, d]
    T = L["x"].shape[0]
    mask = np.zeros((T, N))
    np.put_along_axis(mask, r["topk_idx"], r["topk_w"], axis=1)
    expect = np.einsum("tn,tnd->td", mask, allout)
    if fs:
        expect += oracle.expert_rows(L["Ws_gate"], L["Ws_up"], L["Ws_down"], L["x"])
    np.testing.assert_allclose(r["y"], expect, rtol=1e-12, atol=1e-13)
    assert r["counts"].sum() == T * k


def test_token_order_equivariance():
    """Without capacity each token's output depends on that token only:
    y(P x) = P y(x)."""
    L = _small_layer(13, T=50, fs=12)
    r = _fw(L, 2)
    perm = torch.randperm(50, generator=torch.Generator().manual_seed(0))
    L2 = dict(L)
    L2["x"] = L["x"][perm]
    r2 = _fw(L2, 2)
    np.testing.assert_allclose(r2["y"], r["y"][perm.numpy()], rtol=1e-13, atol=1e-14)


def test_capacity_drops_by_token_order():
    """With capacity, dropped slots contribute zero and the kept weights are not
    renormalised; a token whose every slot is dropped gets y = 0."""
    L = _small_layer(14, T=60, N=4, k=2, bias=False)
    L["bias"] = torch.tensor([4.0, 3.0, -4.0, -4.0])   # push most tokens to experts 0,1
    cf = 0.5
    r = _fw(L, 2, cf)
    C = oracle.capacity(cf, 60, 2, 4)
    assert C == 15
    kept = np.minimum(r["counts"], C)
    assert r["offsets"][-1] == kept.sum() and r["dropped"] == 120 - kept.sum()
    assert r["dropped"] > 0
    full = _fw(L, 2, 0.0)
    allout = np.stack([oracle.expert_rows(L["W_gate"][e], L["W_up"][e], L["W_down"][e], L["x"])
                       for e in range(4)], axis=1)
    for t in range(60):
        acc = np.zeros(L["x"].shape[1])
        for j in range(2):
            if r["inv_pos"][t, j] >= 0:
                acc += r["topk_w"][t, j] * allout[t, r["topk_idx"][t, j]]
        np.testing.assert_allclose(r["y"][t], acc, rtol=1e-12, atol=1e-13)
        if np.all(r["inv_pos"][t] < 0):
            assert np.all(r["y"][t] == 0)
    # the routing itself is the same as without capacity
    assert np.array_equal(full["topk_idx"], r["topk_idx"])


def test_forward_rows_matches_whole_layer():
    """The per-expert-fetch path used for large layers gives the same rows."""
    L = _small_layer(15, T=30, N=5, k=3, fs=8)
    r = _fw(L, 3)
    rows = np.array([0, 7, 8, 29])
    y = oracle.forward_rows(L["x"][rows], r["topk_idx"][rows], r["topk_w"][rows],
                            r["inv_pos"][rows],
                            lambda e: (L["W_gate"][e], L["W_up"][e], L["W_down"][e]),
                            shared=(L["Ws_gate"], L["Ws_up"], L["Ws_down"]))
    np.testing.assert_allclose(y, r["y"][rows], rtol=1e-13, atol=1e-14)


def test_tiny_config_end_to_end_invariants():
    inp = make_inputs(TINY, device="cpu")
    r = oracle.moe_forward(inp.x, inp.W_g, inp.W_gate, inp.W_up, inp.W_down, TINY.k)
    assert r["counts"].sum() == TINY.T * TINY.k
    np.testing.assert_allclose(r["topk_w"].sum(1), 1.0, atol=1e-14)
    assert np.all(np.isfinite(r["y"]))


# ---------------------------------------------------------------- routing diagnostics

def test_routing_entropy_uniform_128_experts_is_7_bits():
    """[Sparse] 4.2: an even load over 128 experts has entropy log2(128) = 7 bits."""
    g = json.load(open(os.path.join(GOLDEN, "router_entropy.json")))
    r = oracle.routing_stats(np.full(g["N"], 11))
    assert r["entropy_bits"] == pytest.approx(g["uniform_entropy_bits"], abs=1e-12)
    assert r["entropy_max_bits"] == pytest.approx(g["uniform_entropy_bits"], abs=1e-12)
    assert r["freq_cv"] == pytest.approx(0.0, abs=1e-12)
    assert r["top3_share"] == pytest.approx(3 / 128, abs=1e-12)


def test_routing_stats_closed_forms():
    # every assignment to one expert: zero entropy, full share, std/mean = sqrt(N-1)
    r = oracle.routing_stats(np.array([0, 0, 0, 9, 0, 0, 0, 0]))
    assert r["entropy_bits"] == 0.0
    assert r["max_share"] == 1.0 and r["top3_share"] == 1.0
    assert r["top3"].tolist() == [3, 0, 1]          # then equal (zero) shares by lower id
    assert r["freq_cv"] == pytest.approx(np.sqrt(7.0), rel=1e-12)
    # two experts with the same load: one bit
    r = oracle.routing_stats(np.array([0, 5, 0, 5]))
    assert r["entropy_bits"] == pytest.approx(1.0, abs=1e-12)
    assert r["top3"].tolist() == [1, 3, 0]
    # shares 1/2, 1/4, 1/8, 1/8: 1.75 bits
    r = oracle.routing_stats(np.array([8, 4, 2, 2]))
    assert r["entropy_bits"] == pytest.approx(1.75, abs=1e-12)
    assert r["top3_share"] == pytest.approx(0.875, abs=1e-12)
    assert r["top3"].tolist() == [0, 1, 2]
    # fewer than three experts: the missing ids are -1
    r = oracle.routing_stats(np.array([3, 1]))
    assert r["top3"].tolist() == [0, 1, -1]
    # no assignments at all
    r = oracle.routing_stats(np.zeros(4, dtype=np.int32))
    assert r["entropy_bits"] == 0 and r["max_share"] == 0 and r["freq_cv"] == 0


def test_routing_balance_closed_forms():
    """[DSV4] balance statistic N * sum f_i p_i: 1 for an even load and even
    probabilities, N when load and probability sit on one expert."""
    N, T = 16, 32
    r = oracle.routing_stats(np.full(N, 4), np.zeros((T, N)))
    assert r["balance"] == pytest.approx(1.0, rel=1e-12)
    assert np.allclose(r["prob_mean"], 1.0 / N, rtol=0, atol=1e-15)
    lg = np.full((T, N), -1e4)
    lg[:, 5] = 0.0
    cnt = np.zeros(N, dtype=np.int32)
    cnt[5] = T
    r = oracle.routing_stats(cnt, lg)
    assert r["balance"] == pytest.approx(N, rel=1e-12)
    # half the load and half the probability on each of two experts: N/2
    lg = np.full((T, N), -1e4)
    lg[:, 2] = lg[:, 9] = 0.0
    cnt = np.zeros(N, dtype=np.int32)
    cnt[2] = cnt[9] = 7
    r = oracle.routing_stats(cnt, lg)
    assert r["balance"] == pytest.approx(N / 2, rel=1e-12)
    assert r["prob_mean"][2] == pytest.approx(0.5, rel=1e-12)
    # softmax probabilities: exp(ln 3) against 1 gives 3/4 and 1/4
    lg = np.full((1, 2), 0.0)
    lg[0, 0] = np.log(3.0)
    r = oracle.routing_stats(np.array([1, 0]), lg)
    assert r["prob_mean"].tolist() == pytest.approx([0.75, 0.25], rel=1e-12)
    assert r["balance"] == pytest.approx(2 * 0.75, rel=1e-12)
    assert np.isnan(oracle.routing_stats(np.array([1, 2]))["balance"])


def test_routing_stats_invariances():
    rng = np.random.default_rng(3)
    N, T = 12, 40
    lg = rng.normal(size=(T, N))
    cnt = rng.integers(0, 50, size=N).astype(np.int32)
    a = oracle.routing_stats(cnt, lg)
    # a per-token shift of the logits leaves the probabilities unchanged
    b = oracle.routing_stats(cnt, lg + rng.normal(size=(T, 1)) * 10)
    assert np.allclose(a["prob_mean"], b["prob_mean"], rtol=1e-12, atol=0)
    # relabelling the experts permutes the per-expert values, not the scalars
    perm = rng.permutation(N)
    c = oracle.routing_stats(cnt[perm], lg[:, perm])
    assert np.allclose(c["freq"], a["freq"][perm]) and np.allclose(c["prob_mean"], a["prob_mean"][perm])
    for key in ("entropy_bits", "top3_share", "max_share", "freq_cv", "balance"):
        assert c[key] == pytest.approx(a[key], rel=1e-12)
    assert a["prob_mean"].sum() == pytest.approx(1.0, rel=1e-12)
    assert a["freq"].sum() == pytest.approx(1.0, rel=1e-12)


# ---------------------------------------------------------------- overflow re-routing

def test_reroute_hand_examples():
    """[Sparse] 2.2: a token whose expert is full goes to its next-best expert."""
    cand = np.array([[0, 1]] * 4 + [[0, 2]] * 2, dtype=np.int32)
    r = oracle.reroute(cand, 1, 1, 3, 2)
    assert r["final_idx"].ravel().tolist() == [0, 0, 1, 1, 2, 2]
    assert r["rerouted"] == 4
    # capacity 1: token 1 takes expert 1, tokens 2 and 3 find it full, token 4 takes 2
    r = oracle.reroute(cand, 1, 1, 3, 1)
    assert r["final_idx"].ravel().tolist() == [0, 1, -1, -1, 2, -1]
    assert r["rerouted"] == 2
    # two rounds: the second untried candidate is used once the first was full
    cand = np.array([[0, 1, 2]] * 3, dtype=np.int32)
    r = oracle.reroute(cand, 1, 2, 3, 1)
    assert r["final_idx"].ravel().tolist() == [0, 1, 2]
    # a token's two overflowing slots propose different candidates
    cand = np.array([[0, 1, 2, 3], [0, 1, 2, 3]], dtype=np.int32)
    r = oracle.reroute(cand, 2, 2, 4, 1)
    assert r["final_idx"].tolist() == [[0, 1], [2, 3]]


def test_reroute_gate_weights_closed_form():
    """Weights are the softmax over the final experts' logits: with logits
    2, ln 3, 0 and expert 0 full, slot 0 moves to expert 2 -> 1/4 and 3/4."""
    lg = np.array([[2.0, np.log(3.0), 0.0], [2.0, np.log(3.0), 0.0]])
    cand = np.array([[0, 1, 2], [0, 1, 2]], dtype=np.int32)
    r = oracle.reroute(cand, 2, 1, 3, 1, logits=lg)
    assert r["final_idx"].tolist() == [[0, 1], [2, -1]]
    assert r["final_w"][1].tolist() == pytest.approx([0.25, 0.75], rel=1e-12)
    # token 0 kept its top-2: the plain softmax over the two
    _, w = oracle.topk_softmax(lg[:1], 2)
    assert r["final_w"][0].tolist() == pytest.approx(w[0].tolist(), rel=1e-12)


@pytest.mark.parametrize("T,N,k,R,cap,seed", [(300, 8, 2, 2, 40, 1), (500, 16, 3, 3, 60, 2),
                                              (64, 4, 1, 3, 5, 3), (200, 32, 2, 0, 9, 4)])
def test_reroute_invariants(T, N, k, R, cap, seed):
    rng = np.random.default_rng(seed)
    lg = rng.normal(size=(T, N)) + np.linspace(2, -2, N)      # skewed towards low ids
    cand, _ = oracle.topk_softmax(lg, k + R)
    r = oracle.reroute(cand, k, R, N, cap, logits=lg)
    fi, pl = r["final_idx"], r["placed"]
    # no expert over capacity; a token's final experts are distinct candidates of its own
    assert np.bincount(fi[pl], minlength=N).max() <= cap
    for t in range(T):
        got = fi[t][pl[t]]
        assert len(set(got.tolist())) == got.size
        assert set(got.tolist()) <= set(cand[t].tolist())
    # the first pass is the plain capacity rule
    g = oracle.group(cand[:, :k], N, cap)
    first = (g["inv_pos"] >= 0)
    assert (pl | ~first).all() and (r["final_cand"][first] < k).all()
    assert (r["final_cand"][first] == np.nonzero(first)[1]).all()
    # re-routed slots are exactly the placed slots beyond the first pass
    assert r["rerouted"] == int(pl.sum() - first.sum())
    if R == 0:
        assert r["rerouted"] == 0 and (pl == first).all()
    # unlimited capacity: nothing moves
    u = oracle.reroute(cand, k, R, N, T * k)
    assert u["rerouted"] == 0 and (u["final_idx"] == cand[:, :k]).all()
    # weights: a softmax over the k final experts
    assert np.allclose(r["final_w"].sum(1), 1.0)


# ---------------------------------------------------------------------------
# FP8 E4M3 expert weights and activations
# ---------------------------------------------------------------------------
def test_e4m3_decode_spec_values():
    """Values the OCP 8-bit floating-point definition fixes for E4M3 (bias 7,
    subnormals m/8 * 2^-6, largest finite 448, S.1111.111 = NaN)."""
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x3C: 1.5, 0x40: 2.0, 0x77: 240.0, 0x78: 256.0, 0x7E: 448.0, 0xFE: -448.0,
             0xB8: -1.0, 0x81: -(2.0 ** -9)}
    got = oracle.e4m3_decode(np.array(list(cases), dtype=np.uint8))
    assert got.tolist() == list(cases.values())
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_e4m3_decode_matches_torch_float8():
    """Every code against torch's own float8_e4m3fn type (a library routine)."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_e4m3_encode_matches_torch_rounding():
    """Round to nearest, ties to even, against torch's float32 -> float8_e4m3fn
    cast: random magnitudes over the whole finite range and every midpoint
    between neighbouring codes (the tie cases)."""
    rng = np.random.default_rng(7)
    mags = np.exp2(rng.uniform(-12, np.log2(448.0), 20000))
    v = (mags * rng.choice([-1.0, 1.0], mags.size)).astype(np.float32)
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids, np.float32([0.0, 448.0, -448.0])])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(v)
    np.testing.assert_array_equal(got, ref)
    # two ties by hand: 1.0625 lies between 1.0 (m=0) and 1.125 (m=1) -> 1.0;
    # 1.1875 between 1.125 (m=1) and 1.25 (m=2) -> 1.25
    assert oracle.e4m3_encode(np.float32([1.0625, 1.1875])).tolist() == [0x38, 0x3A]


def test_e4m3_encode_saturates():
    v = np.float32([449.0, 464.0, 1e6, -1e6, np.inf, -np.inf])
    assert oracle.e4m3_encode(v).tolist() == [0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0xFE]


def test_quantize_rows_e4m3_exact_and_bounded():
    rng = np.random.default_rng(3)
    # rows that are codes times a power of two come back exactly
    codes = rng.integers(0, 0x7E, size=(5, 96)).astype(np.uint8)
    codes[:, 7] = 0x7E                                    # each row's absmax is 448
    codes ^= rng.integers(0, 2, size=codes.shape).astype(np.uint8) << 7
    s = 2.0 ** rng.integers(-6, 4, size=5)
    x = torch.from_numpy(oracle.e4m3_decode(codes) * s[:, None]).to(torch.bfloat16)
    assert torch.equal(x.double(), torch.from_numpy(oracle.e4m3_decode(codes) * s[:, None]))
    q, sc = oracle.quantize_rows_e4m3(x)
    np.testing.assert_array_equal(q, codes)
    np.testing.assert_array_equal(sc, (448.0 * s / 448.0).astype(np.float32))
    # random rows: the absmax element takes +-448; every element within half a
    # step of E4M3 (relative 2^-4 in the normal range, 2^-10 absolute below it)
    x = (torch.randn(64, 300, generator=torch.Generator().manual_seed(5)) * 3).to(torch.bfloat16)
    q, sc = oracle.quantize_rows_e4m3(x)
    xv = x.double().numpy()
    am = np.abs(xv).argmax(1)
    assert (q[np.arange(64), am] & 0x7F == 0x7E).all()
    v = (x.float().numpy() * (np.float32(448.0) / np.abs(x.float().numpy()).max(1))[:, None])
    err = np.abs(oracle.e4m3_decode(q) - v)
    step = np.where(np.abs(v) >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(np.abs(v),
                                                                                 1e-30))) - 3),
                    2.0 ** -9)
    assert (err <= step / 2 + 1e-12).all()
    # an all-zero row: codes 0, scale 1
    q0, s0 = oracle.quantize_rows_e4m3(torch.zeros(2, 16))
    assert (q0 == 0).all() and (s0 == 1.0).all()


def test_quantize_weights_e4m3_per_output_channel():
    """W [N,d,f] -> codes [N,f,d]: output channel j of expert e is column j of
    W[e] over d, quantised with its own absmax."""
    rng = np.random.default_rng(11)
    N, d, f = 3, 40, 24
    codes = rng.integers(0, 0x7E, size=(N, f, d)).astype(np.uint8)
    codes[:, :, 5] = 0x7E
    s = 2.0 ** rng.integers(-8, 0, size=(N, f))
    W = np.transpose(oracle.e4m3_decode(codes) * s[..., None], (0, 2, 1))   # [N,d,f]
    q, sc = oracle.quantize_weights_e4m3(torch.from_numpy(W).to(torch.bfloat16))
    np.testing.assert_array_equal(q, codes)
    np.testing.assert_array_equal(sc, s.astype(np.float32))


def test_fp8_expert_equals_bf16_expert_on_representable_values():
    """When x and the gate/up weights are exactly E4M3 values times their
    scales, the FP8 expert is the bf16 expert: the dequantised operands, the
    scales' axes (per token row, per output channel) and the SwiGLU are fed
    through unchanged."""
    rng = np.random.default_rng(21)
    R, d, f = 9, 48, 32
    cx = rng.integers(0, 0x7E, size=(R, d)).astype(np.uint8) | \
        (rng.integers(0, 2, size=(R, d)).astype(np.uint8) << 7)
    cx[:, 0] = 0x7E
    sx = 2.0 ** rng.integers(-9, -6, size=R)
    x = torch.from_numpy(oracle.e4m3_decode(cx) * sx[:, None]).to(torch.bfloat16)
    Ws = []
    for _ in range(2):
        c = rng.integers(0, 0x7E, size=(f, d)).astype(np.uint8) | \
            (rng.integers(0, 2, size=(f, d)).astype(np.uint8) << 7)
        c[:, 3] = 0x7E
        s = 2.0 ** rng.integers(-12, -9, size=f)
        Ws.append(torch.from_numpy((oracle.e4m3_decode(c) * s[:, None]).T.copy()).to(torch.bfloat16))
    Wd = (torch.randn(f, d, generator=torch.Generator().manual_seed(2)) * 0.1).to(torch.bfloat16)
    ref = oracle.expert_rows(Ws[0], Ws[1], Wd, x)
    qx, sxq = oracle.quantize_rows_e4m3(x)
    qw = [oracle.quantize_weights_e4m3(W[None]) for W in Ws]
    got = oracle.expert_rows_fp8(qw[0][0][0], qw[0][1][0], qw[1][0][0], qw[1][1][0], Wd, qx, sxq)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_expert_hidden_is_the_first_half_of_the_expert():
    """h = SiLU(x W_gate) * (x W_up) from the hidden-activation function, times
    W_down, is the whole expert (pinned above by its closed forms)."""
    g = torch.Generator().manual_seed(9)
    d, f, R = 24, 40, 7
    Wg, Wu = torch.randn(d, f, generator=g), torch.randn(d, f, generator=g)
    Wd = torch.randn(f, d, generator=g)
    x = torch.randn(R, d, generator=g)
    h = oracle.expert_hidden(Wg, Wu, x)
    np.testing.assert_allclose(h @ Wd.double().numpy(), oracle.expert_rows(Wg, Wu, Wd, x),
                               rtol=1e-12, atol=1e-12)
    # closed form on one element: x = e_0, so g = Wg[0], u = Wu[0]
    e0 = torch.zeros(1, d)
    e0[0, 0] = 1
    gv, uv = Wg[0].double().numpy(), Wu[0].double().numpy()
    np.testing.assert_allclose(oracle.expert_hidden(Wg, Wu, e0)[0], gv / (1 + np.exp(-gv)) * uv,
                               rtol=1e-14)


def _codes(rng, shape, absmax_col=None):
    """Random finite E4M3 codes with random signs; column absmax_col (if given)
    holds +-448 so that every row's absmax is exactly 448."""
    c = rng.integers(0, 0x7E, size=shape).astype(np.uint8) | \
        (rng.integers(0, 2, size=shape).astype(np.uint8) << 7)
    if absmax_col is not None:
        c[..., absmax_col] = (c[..., absmax_col] & 0x80) | 0x7E
    return c


def test_fp8_down_rows_exact_on_representable_h():
    """Rows of h that are E4M3 codes times a per-row power of two (each row's
    absmax maps to 448) quantise exactly, and W_down channels that are codes
    times a per-channel power of two too: the E4M3 down projection is then the
    exact product h W_down.  Rows and channels get different scales and f != d,
    so a scale on the wrong axis or row, a dropped scale or a transposed W_down
    gives another result."""
    rng = np.random.default_rng(29)
    R, f, d = 7, 40, 24
    ch = _codes(rng, (R, f), absmax_col=3)
    hs = 2.0 ** rng.integers(-6, 6, size=R)
    h = oracle.e4m3_decode(ch) * hs[:, None]
    cd = _codes(rng, (d, f), absmax_col=11)
    sd = (2.0 ** rng.integers(-12, -4, size=d)).astype(np.float32)
    Wd = (oracle.e4m3_decode(cd) * sd[:, None]).T        # [f, d]: the matrix itself
    got = oracle.down_rows_e4m3(h, cd, sd)
    np.testing.assert_allclose(got, h @ Wd, rtol=1e-13, atol=1e-300)
    # one-hot rows (values 448 times a power of two: exact scales) read out
    # W_down's rows, scaled by the row's value
    eye = np.zeros((3, f))
    eye[0, 0], eye[1, 5], eye[2, f - 1] = 448.0, -448.0 * 2.0 ** -3, 448.0 * 2.0 ** -9
    np.testing.assert_allclose(oracle.down_rows_e4m3(eye, cd, sd),
                               eye[:, [0, 5, f - 1]].sum(1)[:, None] * Wd[[0, 5, f - 1]],
                               rtol=1e-14)


def test_fp8_down_quantises_the_unrounded_h():
    """h is quantised from its own values, not from a bf16-rounded copy:
    1.0625 + 2^-12 (above the tie between 1.0 and 1.125) becomes 1.125, while
    its bf16 rounding (1.0625, exactly the tie) would become 1.0 (ties to even)."""
    f, d = 16, 2
    h = np.zeros((1, f))
    h[0, 0], h[0, 1] = 1.0625 + 2.0 ** -12, 448.0            # absmax 448: scale 1
    cd = np.zeros((d, f), dtype=np.uint8)
    cd[0, 0] = 0x38                                          # W_down[0, 0] = 1.0
    cd[1, 1] = 0x38                                          # W_down[1, 1] = 1.0
    out = oracle.down_rows_e4m3(h, cd, np.ones(d, dtype=np.float32))
    assert out.tolist() == [[1.125, 448.0]]


def test_fp8_expert_down_is_hidden_then_down():
    """The E4M3 expert with an E4M3 down projection is its hidden activation
    (pinned through the bf16 expert above) followed by the E4M3 down
    projection (pinned above), row by row."""
    rng = np.random.default_rng(23)
    R, d, f = 6, 32, 48
    x = torch.from_numpy(rng.normal(size=(R, d))).to(torch.bfloat16)
    Wg = torch.from_numpy(rng.normal(size=(d, f)) / d ** 0.5).to(torch.bfloat16)
    Wu = torch.from_numpy(rng.normal(size=(d, f)) / d ** 0.5).to(torch.bfloat16)
    Wd = torch.from_numpy(rng.normal(size=(f, d)) / f ** 0.5).to(torch.bfloat16)
    qx, sx = oracle.quantize_rows_e4m3(x)
    (qg, sg), (qu, su) = oracle.quantize_weights_e4m3(Wg[None]), oracle.quantize_weights_e4m3(Wu[None])
    (qd, sdq) = oracle.quantize_weights_e4m3(Wd[None])
    got = oracle.expert_rows_fp8(qg[0], sg[0], qu[0], su[0], None, qx, sx, qd[0], sdq[0])
    h = oracle.expert_hidden(np.ascontiguousarray(oracle.dequantize_e4m3(qg[0], sg[0]).T),
                             np.ascontiguousarray(oracle.dequantize_e4m3(qu[0], su[0]).T),
                             oracle.dequantize_e4m3(qx, sx))
    np.testing.assert_allclose(got, oracle.down_rows_e4m3(h, qd[0], sdq[0]), rtol=1e-12,
                               atol=1e-14)
    # and the E4M3 down projection stays close to the exact one (a loose bound
    # that a lost or misplaced scale breaks)
    exact = h @ Wd.double().numpy()
    assert np.linalg.norm(got - exact) / np.linalg.norm(exact) < 0.1
