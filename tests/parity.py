"""Shared parity checks: the CUDA path (through the C ABI) against the oracle.

Every expected value comes from the oracle run on the test's inputs; nothing
the GPU produced is fed to the oracle.

Acceptance (the layer's stated tolerances):
  * expert indices bit-exact, except tokens whose oracle k-th and (k+1)-th
    logits differ by less than 1e-4 relative (near-ties: counted, reported);
    inside the top-k, two slots whose fp64 logits differ by less than the same
    relative gap may appear in either order (same set: counted);
  * counts / offsets / perm_token bit-exact against the oracle's grouping, and
    inv_pos bit-exact per (token, expert); when a near-tie token took the other
    valid expert set, the experts it touches are checked for validity instead
    (stable order, capacity ranks, a bijection) and exactness holds elsewhere;
  * gate weights within 1e-5 relative;
  * bf16 layer output within max-abs 2e-2 and relative Frobenius 5e-3;
    fp32 layer output within max-abs 1e-4 and relative Frobenius 2e-5 (fp32
    accumulation over at most a few hundred terms of size O(1/sqrt(n)), with a
    margin of ~10x over the rounding bound).
"""
from dataclasses import dataclass, field

import numpy as np
import torch

import oracle
from sparse_mixture_experts_63_b300 import binding as B

TIE_REL = 1e-4
W_REL = 1e-5
TOL = {"bf16": (2e-2, 5e-3), "f32": (1e-4, 2e-5)}


@dataclass
class RoutingReport:
    tokens: int
    near_tie: int = 0                 # k/k+1 near-ties in the oracle's logits
    set_mismatch: int = 0             # tokens whose selected set differs (must be near-ties)
    order_swaps: int = 0              # same set, different slot order (near-equal logits)
    unexplained: list = field(default_factory=list)
    w_max_rel: float = 0.0


def check_routing(logits_o, idx_g, w_g, k):
    """Compare GPU routing (idx_g, w_g: numpy) with the oracle's fp64 logits."""
    T, N = logits_o.shape
    idx_o, w_o = oracle.topk_softmax(logits_o, k)
    near = oracle.near_tie_tokens(logits_o, k, TIE_REL)
    rep = RoutingReport(tokens=T, near_tie=int(near.sum()))
    for t in np.nonzero((idx_o != idx_g).any(1))[0]:
        so, sg = set(idx_o[t].tolist()), set(idx_g[t].tolist())
        if so != sg:
            rep.set_mismatch += 1
            if not near[t]:
                rep.unexplained.append(("set", int(t), idx_o[t].tolist(), idx_g[t].tolist()))
            continue
        # same set, different order: every out-of-place pair must be a near-tie
        lo = logits_o[t]
        ok = True
        for j in range(k):
            if idx_o[t, j] != idx_g[t, j]:
                a, b = lo[idx_o[t, j]], lo[idx_g[t, j]]
                if abs(a - b) >= TIE_REL * max(abs(a), abs(b)):
                    ok = False
        rep.order_swaps += 1
        if not ok:
            rep.unexplained.append(("order", int(t), idx_o[t].tolist(), idx_g[t].tolist()))
    # weights: per expert id, on tokens whose sets agree
    same = np.array([set(idx_o[t].tolist()) == set(idx_g[t].tolist()) for t in range(T)])
    if same.any():
        wo = np.zeros((T, N))
        wg = np.zeros((T, N))
        np.put_along_axis(wo, idx_o, w_o, axis=1)
        np.put_along_axis(wg, idx_g, w_g.astype(np.float64), axis=1)
        rel = np.abs(wg[same] - wo[same]) / np.maximum(np.abs(wo[same]), 1e-30)
        rel[wo[same] == 0] = 0
        rep.w_max_rel = float(rel.max())
    return rep


def _by_expert(idx, inv):
    """Per token, (expert, position) pairs sorted by expert: slot order is
    free for near-equal logits, the position of each (token, expert) is not."""
    o = np.argsort(idx, axis=1, kind="stable")
    return np.take_along_axis(idx, o, 1), np.take_along_axis(inv, o, 1)


def check_grouping(out, idx_g, g_o, idx_o, N, C, flipped):
    """GPU grouping against the oracle's grouping of the oracle's routing.

    flipped: tokens whose GPU expert set is the other valid near-tie choice.
    Experts they touch (either choice) are checked for validity; every other
    expert's list and every other token's positions must match exactly."""
    counts_g = out["counts"].cpu().numpy()
    offsets_g = out["offsets"].cpu().numpy()
    inv_g = out["inv_pos"].cpu().numpy()
    A_g = int(offsets_g[-1])
    T, k = idx_g.shape
    # the GPU's per-expert token lists, read back through inv_pos (a bijection
    # of the kept (token, slot) pairs onto [0, A))
    kept = inv_g >= 0
    assert np.count_nonzero(kept) == A_g
    pos = inv_g[kept]
    assert pos.min(initial=0) >= 0 and pos.max(initial=-1) < A_g
    assert np.unique(pos).size == A_g, "inv_pos is not a bijection"
    perm_g = np.full(A_g, -1, dtype=np.int64)
    perm_g[pos] = np.nonzero(kept)[0]
    touched = np.zeros(N, dtype=bool)
    if flipped.size:
        touched[np.unique(np.concatenate([idx_g[flipped].ravel(), idx_o[flipped].ravel()]))] = True
    if not touched.any():
        np.testing.assert_array_equal(counts_g, g_o["counts"])
        np.testing.assert_array_equal(offsets_g, g_o["offsets"])
        np.testing.assert_array_equal(perm_g, g_o["perm_token"])
        assert int(out["dropped"].item()) == g_o["dropped"]
        eg, pg = _by_expert(idx_g, inv_g)
        eo, po = _by_expert(idx_o, g_o["inv_pos"])
        np.testing.assert_array_equal(eg, eo)
        np.testing.assert_array_equal(pg, po)
        return 0
    # offsets are the exclusive scan of the kept counts
    kept_g = np.diff(offsets_g)
    assert (kept_g == (np.minimum(counts_g, C) if C > 0 else counts_g)).all()
    kept_o = np.diff(g_o["offsets"])
    for e in range(N):
        lst = perm_g[offsets_g[e]:offsets_g[e + 1]]
        if not touched[e]:
            np.testing.assert_array_equal(lst, g_o["perm_token"][g_o["offsets"][e]:g_o["offsets"][e + 1]])
            assert counts_g[e] == g_o["counts"][e] and kept_g[e] == kept_o[e]
            continue
        # validity: the first kept_g[e] tokens (ascending) that chose e on the GPU
        chose = np.nonzero((idx_g == e).any(1))[0]
        assert counts_g[e] == chose.size
        np.testing.assert_array_equal(lst, chose[:kept_g[e]])
    # every kept (token, slot) sits inside its expert's range
    tt, jj = np.nonzero(kept)
    e_of = idx_g[tt, jj]
    assert ((offsets_g[e_of] <= inv_g[tt, jj]) & (inv_g[tt, jj] < offsets_g[e_of + 1])).all()
    return int(touched.sum())


def y_error(y_gpu, y_ref):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    diff = y_gpu - y_ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    fro = float(np.linalg.norm(diff) / max(np.linalg.norm(y_ref), 1e-30)) if diff.size else 0.0
    return max_abs, fro


def assert_y_close(y_gpu, y_ref, dtype):
    max_abs, fro = y_error(y_gpu, y_ref)
    tol_abs, tol_fro = TOL[dtype]
    assert max_abs <= tol_abs and fro <= tol_fro, (
        f"layer output off: max-abs {max_abs:.3e} (tol {tol_abs}), rel-fro {fro:.3e} (tol {tol_fro})")
    return max_abs, fro


def run_forward(inp, logits=True, y_dtype=torch.float32):
    """moe_forward through the C ABI; returns y and the routing outputs (on GPU)."""
    cfg = inp.cfg
    layer = B.MoELayer(inp.W_g, inp.W_gate, inp.W_up, inp.W_down, cfg.k, bias=inp.bias,
                       Ws_gate=inp.Ws_gate, Ws_up=inp.Ws_up, Ws_down=inp.Ws_down,
                       capacity_factor=cfg.cf, y_dtype=y_dtype)
    y = layer(inp.x, logits=logits)
    torch.cuda.synchronize()
    return y, layer.last


def fetcher(inp):
    cache = {}

    def fetch(e):
        if e not in cache:
            cache[e] = (inp.W_gate[e].cpu(), inp.W_up[e].cpu(), inp.W_down[e].cpu())
        return cache[e]
    return fetch


def check_layer(inp, rows=None, y_dtype=torch.float32, report=None):
    """End-to-end parity of moe_forward on one synthetic layer.

    The oracle routes, groups and evaluates the layer from the inputs alone.
    Routing is compared on all tokens and grouping on every expert; the layer
    output on `rows` (all if None), leaving out the tokens whose output may
    legitimately differ: near-tie tokens that took the other valid expert set
    and, with a capacity, tokens sharing an expert with one (their drop ranks
    may move).  Returns a dict of the measured errors and counts."""
    cfg = inp.cfg
    y, out = run_forward(inp, logits=True, y_dtype=y_dtype)
    status = int(out["device_status"].item())
    assert status == 0, f"device_status {status:#x}"
    x_c = inp.x.cpu()
    logits_o = oracle.router_logits(x_c, inp.W_g.cpu(), None if inp.bias is None else inp.bias.cpu())
    idx_o, w_o = oracle.topk_softmax(logits_o, cfg.k)
    idx_g = out["topk_idx"].cpu().numpy()
    w_g = out["topk_w"].cpu().numpy()
    # GPU logits against fp64 (fp32 accumulation)
    lg = out["logits"].cpu().double().numpy()
    rep = check_routing(logits_o, idx_g, w_g, cfg.k)
    assert not rep.unexplained, f"routing mismatches not explained by near-ties: {rep.unexplained[:5]}"
    assert rep.w_max_rel <= W_REL, f"gate weights off by {rep.w_max_rel:.3e} relative"
    flipped = np.nonzero(np.sort(idx_g, 1) != np.sort(idx_o, 1))[0]
    flipped = np.unique(flipped)
    # grouping
    C = oracle.capacity(cfg.cf, cfg.T, cfg.k, cfg.N)
    g_o = oracle.group(idx_o, cfg.N, C)
    touched = check_grouping(out, idx_g, g_o, idx_o, cfg.N, C, flipped)
    # layer output: the oracle's own routing and grouping
    sel = np.arange(cfg.T) if rows is None else np.asarray(rows)
    skip = np.zeros(cfg.T, dtype=bool)
    skip[flipped] = True
    if C > 0 and flipped.size:
        ex = np.unique(np.concatenate([idx_g[flipped].ravel(), idx_o[flipped].ravel()]))
        skip |= np.isin(idx_o, ex).any(1)
    excluded = int(skip[sel].sum())
    assert excluded <= max(2, len(sel) // 100), f"{excluded} of {len(sel)} rows left out"
    sel = sel[~skip[sel]]
    shared = None
    if cfg.fs:
        shared = (inp.Ws_gate.cpu(), inp.Ws_up.cpu(), inp.Ws_down.cpu())
    y_o = oracle.forward_rows(x_c[torch.as_tensor(sel)], idx_o[sel], w_o[sel], g_o["inv_pos"][sel],
                              fetcher(inp), shared=shared)
    y_g = y[torch.as_tensor(sel, device=y.device)].float().cpu().numpy()
    max_abs, fro = assert_y_close(y_g, y_o, cfg.dtype)
    res = dict(max_abs=max_abs, rel_fro=fro, near_tie=rep.near_tie, set_mismatch=rep.set_mismatch,
               order_swaps=rep.order_swaps, dropped=g_o["dropped"], w_max_rel=rep.w_max_rel,
               logits_max_abs=float(np.abs(lg - logits_o).max()), rows=len(sel),
               rows_left_out=excluded, experts_validity_checked=touched)
    if report is not None:
        report.append((cfg.name, res))
    return res


def _fp8_fetch(inp, qw):
    (qg, sg), (qu, su) = qw[:2]
    qd = qw[2] if len(qw) > 2 else None

    def fetch(e):
        w = (qg[e], sg[e], qu[e], su[e], inp.W_down[e].cpu())
        return w if qd is None else w + (qd[0][e], qd[1][e])
    return fetch


_QCACHE = {}


def oracle_codes(cfg, name, W):
    """The oracle's E4M3 codes and channel scales of one weight tensor of a
    seeded layer, computed once per (layer, tensor) in this process (the
    inputs of a config and seed are always the same tensors)."""
    key = (cfg, name)
    if key not in _QCACHE:
        _QCACHE[key] = oracle.quantize_weights_e4m3(W.cpu())
    return _QCACHE[key]


def check_layer_fp8(cfg, inp, rows=None, down=False):
    """moe_forward with E4M3 gate/up (and down, with `down`) against the
    oracle's fp64 layer on its own E4M3 codes of x and of the weights; the
    layer's codes must equal the oracle's byte for byte.  Routing as in
    check_layer (near-tie rows left out).  Returns the measured errors."""
    layer = B.MoELayer(inp.W_g, inp.W_gate, inp.W_up, inp.W_down, cfg.k, bias=inp.bias,
                       Ws_gate=inp.Ws_gate, Ws_up=inp.Ws_up, Ws_down=inp.Ws_down,
                       capacity_factor=cfg.cf, fp8=True, fp8_down=down)
    y = layer(inp.x)
    torch.cuda.synchronize()
    out = layer.last
    assert int(out["device_status"].item()) == 0
    # the layer's quantised weights are the oracle's, byte for byte
    qw = [oracle_codes(cfg, "W_gate", inp.W_gate), oracle_codes(cfg, "W_up", inp.W_up)]
    if down:
        qw.append(oracle_codes(cfg, "W_down", inp.W_down))
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
    max_abs, fro = assert_y_close(y_g, y_o, "bf16")
    # how far E4M3 moves the layer from its bf16 definition (reported; a
    # loose bound catches a lost or misplaced scale)
    y_b = oracle.forward_rows(x_c[torch.as_tensor(sel)], idx_o[sel], w_o[sel],
                              g_o["inv_pos"][sel], fetcher(inp), shared=shared)
    q_err = float(np.linalg.norm(y_g - y_b) / max(np.linalg.norm(y_b), 1e-30))
    assert q_err < (0.15 if down else 0.1), f"FP8 layer {q_err:.3f} (rel-fro) away from the bf16 layer"
    return dict(max_abs=max_abs, rel_fro=fro, fp8_vs_bf16_rel_fro=q_err, rows=len(sel))
