"""Shared parity checks: the CUDA path (through the C ABI) against the oracle.

Acceptance (the layer's stated tolerances):
  * expert indices bit-exact, except tokens whose oracle k-th and (k+1)-th
    logits differ by less than 1e-4 relative (near-ties: counted, reported);
    inside the top-k, two slots whose fp64 logits differ by less than the same
    relative gap may appear in either order (same set: counted);
  * counts / offsets / inv_pos / perm_token bit-exact given the same indices;
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


def masked_oracle_routing(logits_o, idx_g, k):
    """The oracle's routing restricted to the GPU-selected expert sets: the
    oracle's top-k/softmax over fp64 logits with every other expert at -inf.
    Isolates the FFN/combine comparison from near-tie routing flips."""
    m = np.full_like(logits_o, -np.inf)
    np.put_along_axis(m, idx_g.astype(np.int64), np.take_along_axis(logits_o, idx_g.astype(np.int64), 1), 1)
    return oracle.topk_softmax(m, k)


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

    Routing is compared on all tokens; the layer output on `rows` (all if None)
    against the oracle run with the GPU-selected expert sets.  Returns a dict of
    the measured errors and counts."""
    cfg = inp.cfg
    y, out = run_forward(inp, logits=True, y_dtype=y_dtype)
    status = int(out["device_status"].item())
    assert status == 0, f"device_status {status:#x}"
    x_c = inp.x.cpu()
    logits_o = oracle.router_logits(x_c, inp.W_g.cpu(), None if inp.bias is None else inp.bias.cpu())
    idx_g = out["topk_idx"].cpu().numpy()
    w_g = out["topk_w"].cpu().numpy()
    # GPU logits against fp64 (fp32 accumulation)
    lg = out["logits"].cpu().double().numpy()
    rep = check_routing(logits_o, idx_g, w_g, cfg.k)
    assert not rep.unexplained, f"routing mismatches not explained by near-ties: {rep.unexplained[:5]}"
    assert rep.w_max_rel <= W_REL, f"gate weights off by {rep.w_max_rel:.3e} relative"
    # grouping, given the GPU's indices
    C = oracle.capacity(cfg.cf, cfg.T, cfg.k, cfg.N)
    g = oracle.group(idx_g, cfg.N, C)
    np.testing.assert_array_equal(out["counts"].cpu().numpy(), g["counts"])
    np.testing.assert_array_equal(out["offsets"].cpu().numpy(), g["offsets"])
    np.testing.assert_array_equal(out["inv_pos"].cpu().numpy(), g["inv_pos"])
    assert int(out["dropped"].item()) == g["dropped"]
    # layer output
    idx_m, w_m = masked_oracle_routing(logits_o, idx_g, cfg.k)
    gm = oracle.group(idx_m, cfg.N, C)
    sel = np.arange(cfg.T) if rows is None else np.asarray(rows)
    shared = None
    if cfg.fs:
        shared = (inp.Ws_gate.cpu(), inp.Ws_up.cpu(), inp.Ws_down.cpu())
    y_o = oracle.forward_rows(x_c[torch.as_tensor(sel)], idx_m[sel], w_m[sel], gm["inv_pos"][sel],
                              fetcher(inp), shared=shared)
    y_g = y[torch.as_tensor(sel, device=y.device)].float().cpu().numpy()
    max_abs, fro = assert_y_close(y_g, y_o, cfg.dtype)
    res = dict(max_abs=max_abs, rel_fro=fro, near_tie=rep.near_tie, set_mismatch=rep.set_mismatch,
               order_swaps=rep.order_swaps, dropped=g["dropped"], w_max_rel=rep.w_max_rel,
               logits_max_abs=float(np.abs(lg - logits_o).max()), rows=len(sel))
    if report is not None:
        report.append((cfg.name, res))
    return res
