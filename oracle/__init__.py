"""fp64 CPU oracle for one sparse MoE layer forward -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it and
shares no code with it.

This module is argument marshalling around ``moe_oracle.c`` (ctypes); all the
arithmetic of the layer is in that C file, written as the plain definition in
double precision (``dequantize_e4m3``, the decoded codes times their scales,
is a convenience for the tests).  Inputs are torch CPU tensors (float32 or bfloat16) or numpy
arrays; outputs are numpy arrays (float64 for values, int32 for indices).
"""
import ctypes
import math
import os

import numpy as np
import torch

from . import build as _build

_lib = None

F32, BF16, F64 = 0, 1, 2


def _load(path=None):
    """Load liboracle.so (building it first if needed).  ``path`` loads another
    build of the same source instead (used by the mutation tests)."""
    global _lib
    if _lib is None or path is not None:
        path = path or _build.build()
        lib = ctypes.CDLL(path)
        vp, i32p, f64p, f32p = (ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_void_p)
        ci, cd = ctypes.c_int, ctypes.c_double
        lib.oracle_router_logits.argtypes = [ci, ci, ci, ci, vp, vp, f32p, f64p, ci]
        lib.oracle_topk_softmax.argtypes = [ci, ci, ci, f64p, i32p, f64p]
        lib.oracle_capacity.argtypes = [cd, ci, ci, ci]
        lib.oracle_group.argtypes = [ci, ci, ci, ci, i32p, i32p, i32p, i32p, i32p,
                                     i32p, i32p]
        lib.oracle_expert_rows.argtypes = [ci, ci, ci, vp, vp, vp, ci, vp, ci, f64p, ci]
        lib.oracle_combine_rows.argtypes = [ci, ci, ci, i32p, f64p, f64p, f64p, f64p]
        lib.oracle_routing_stats.argtypes = [ci, ci, f64p, i32p, f64p, i32p, f64p, f64p]
        lib.oracle_reroute.argtypes = [ci, ci, ci, ci, ci, i32p, f64p, i32p, i32p, i32p, f64p]
        lib.oracle_expert_hidden.argtypes = [ci, ci, ci, vp, vp, ci, vp, ci, f64p, ci]
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_long, vp, f64p]
        lib.oracle_e4m3_decode.restype = None
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_long, f32p, vp]
        lib.oracle_e4m3_encode.restype = None
        lib.oracle_quantize_rows_e4m3.argtypes = [ci, ci, ci, vp, vp, f32p]
        lib.oracle_quantize_weights_e4m3.argtypes = [ci, ci, ci, ci, vp, vp, f32p, ci]
        lib.oracle_down_rows_e4m3.argtypes = [ci, ci, ci, f64p, vp, f32p, f64p, ci]
        lib.oracle_expert_rows_e4m3.argtypes = [ci, ci, vp, f32p, vp, f32p, ci, vp, f32p, ci,
                                                vp, vp, f32p, f64p, ci]
        lib.oracle_moe_forward.argtypes = (
            [ci] * 6 + [vp, vp, f32p, vp, vp, vp, ci, vp, vp, vp, cd, f64p, f64p,
                        i32p, f64p, i32p, i32p, i32p, i32p, ci])
        for name in ("oracle_router_logits", "oracle_topk_softmax", "oracle_capacity",
                     "oracle_group", "oracle_expert_rows", "oracle_combine_rows",
                     "oracle_moe_forward", "oracle_routing_stats", "oracle_reroute",
                     "oracle_down_rows_e4m3", "oracle_expert_rows_e4m3"):
            getattr(lib, name).restype = ci
        _lib = lib
    return _lib


def default_threads() -> int:
    return os.cpu_count() or 1


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------
class _Buf:
    """Keeps a contiguous CPU buffer alive and exposes its address + dtype code."""

    def __init__(self, a):
        if isinstance(a, torch.Tensor):
            a = a.detach()
            if a.device.type != "cpu":
                a = a.cpu()
            a = a.contiguous()
            if a.dtype == torch.bfloat16:
                self.dtype = BF16
            elif a.dtype == torch.float32:
                self.dtype = F32
            elif a.dtype == torch.float64:
                self.dtype = F64
            else:
                self.dtype = None
            self.keep = a
            self.ptr = a.data_ptr()
        else:
            a = np.ascontiguousarray(a)
            self.dtype = {np.dtype(np.float32): F32, np.dtype(np.float64): F64}.get(a.dtype)
            self.keep = a
            self.ptr = a.ctypes.data


def _f32_or_none(b):
    if b is None:
        return None, None
    if isinstance(b, torch.Tensor):
        b = b.detach().cpu().float().contiguous().numpy()
    b = np.ascontiguousarray(b, dtype=np.float32)
    return b, b.ctypes.data


def _i32(a):
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a):
    return None if a is None else a.ctypes.data


def _check(rc, name):
    if rc != 0:
        raise RuntimeError(f"{name} failed with code {rc}")


# --------------------------------------------------------------------------
# stage functions
# --------------------------------------------------------------------------
def router_logits(x, W_g, bias=None, nthreads=None):
    """logits[T,N] (fp64) = x[T,d] @ W_g[d,N] + bias[N]."""
    lib = _load()
    bx, bw = _Buf(x), _Buf(W_g)
    assert bx.dtype is not None and bx.dtype == bw.dtype
    T, d = bx.keep.shape
    N = bw.keep.shape[1]
    bb, pb = _f32_or_none(bias)
    out = np.empty((T, N), dtype=np.float64)
    _check(lib.oracle_router_logits(T, d, N, bx.dtype, bx.ptr, bw.ptr, pb, out.ctypes.data,
                                    nthreads or default_threads()), "oracle_router_logits")
    return out


def topk_softmax(logits, k):
    """(topk_idx[T,k] int32, topk_w[T,k] fp64) from fp64 logits[T,N]."""
    lib = _load()
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    T, N = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    _check(lib.oracle_topk_softmax(T, N, k, logits.ctypes.data, idx.ctypes.data,
                                   w.ctypes.data), "oracle_topk_softmax")
    return idx, w


def route(x, W_g, k, bias=None, nthreads=None):
    logits = router_logits(x, W_g, bias, nthreads)
    idx, w = topk_softmax(logits, k)
    return logits, idx, w


def capacity(cf, T, k, N) -> int:
    return int(_load().oracle_capacity(float(cf), T, k, N))


def group(topk_idx, N, capacity_rows=0):
    """Grouping by expert.  Returns dict of counts, offsets, perm_token,
    perm_slot, inv_pos, dropped (see moe_oracle.c, oracle_group)."""
    lib = _load()
    idx = _i32(topk_idx)
    T, k = idx.shape
    counts = np.empty(N, dtype=np.int32)
    offsets = np.empty(N + 1, dtype=np.int32)
    perm_token = np.full(T * k, -1, dtype=np.int32)
    perm_slot = np.full(T * k, -1, dtype=np.int32)
    inv_pos = np.empty((T, k), dtype=np.int32)
    dropped = np.zeros(1, dtype=np.int32)
    _check(lib.oracle_group(T, N, k, int(capacity_rows), idx.ctypes.data, counts.ctypes.data,
                            offsets.ctypes.data, perm_token.ctypes.data,
                            perm_slot.ctypes.data, inv_pos.ctypes.data,
                            dropped.ctypes.data), "oracle_group")
    A = int(offsets[N])
    return dict(counts=counts, offsets=offsets, perm_token=perm_token[:A],
                perm_slot=perm_slot[:A], inv_pos=inv_pos, dropped=int(dropped[0]))


def expert_rows(W_gate_e, W_up_e, W_down_e, xrows, nthreads=None):
    """out[R,d] (fp64) = SwiGLU expert (W_gate_e [d,f], W_up_e [d,f], W_down_e [f,d])
    applied to each row of xrows [R,d]."""
    lib = _load()
    bg, bu, bd, bx = _Buf(W_gate_e), _Buf(W_up_e), _Buf(W_down_e), _Buf(xrows)
    assert bg.dtype is not None and bg.dtype == bu.dtype == bd.dtype
    d, f = bg.keep.shape
    R = bx.keep.shape[0]
    out = np.empty((R, d), dtype=np.float64)
    _check(lib.oracle_expert_rows(d, f, bg.dtype, bg.ptr, bu.ptr, bd.ptr, R, bx.ptr,
                                  bx.dtype, out.ctypes.data, nthreads or default_threads()),
           "oracle_expert_rows")
    return out


def combine_rows(inv_pos_rows, topk_w_rows, expert_out, shared=None):
    """y[R,d] = sum_j kept w[r,j] * expert_out[r,j,:] (+ shared[r,:])."""
    lib = _load()
    inv = _i32(inv_pos_rows)
    w = np.ascontiguousarray(topk_w_rows, dtype=np.float64)
    o = np.ascontiguousarray(expert_out, dtype=np.float64)
    R, k, d = o.shape
    sh = None if shared is None else np.ascontiguousarray(shared, dtype=np.float64)
    y = np.empty((R, d), dtype=np.float64)
    _check(lib.oracle_combine_rows(R, k, d, inv.ctypes.data, w.ctypes.data, o.ctypes.data,
                                   _p(sh), y.ctypes.data), "oracle_combine_rows")
    return y


def moe_forward(x, W_g, W_gate, W_up, W_down, k, bias=None, Ws_gate=None, Ws_up=None,
                Ws_down=None, capacity_factor=0.0, nthreads=None):
    """Whole layer on all tokens with every weight in host memory (small cases).

    Returns dict: y [T,d] fp64, logits, topk_idx, topk_w, counts, offsets,
    inv_pos, dropped.
    """
    lib = _load()
    bx, bg = _Buf(x), _Buf(W_g)
    bwg, bwu, bwd = _Buf(W_gate), _Buf(W_up), _Buf(W_down)
    dt = bx.dtype
    assert dt is not None and all(b.dtype == dt for b in (bg, bwg, bwu, bwd))
    T, d = bx.keep.shape
    N, _, f = bwg.keep.shape
    fs = 0
    ps = (None, None, None)
    keep = []
    if Ws_gate is not None:
        bsg, bsu, bsd = _Buf(Ws_gate), _Buf(Ws_up), _Buf(Ws_down)
        assert bsg.dtype == dt == bsu.dtype == bsd.dtype
        fs = bsg.keep.shape[1]
        ps = (bsg.ptr, bsu.ptr, bsd.ptr)
        keep += [bsg, bsu, bsd]
    bb, pb = _f32_or_none(bias)
    y = np.empty((T, d), dtype=np.float64)
    logits = np.empty((T, N), dtype=np.float64)
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    counts = np.empty(N, dtype=np.int32)
    offsets = np.empty(N + 1, dtype=np.int32)
    inv = np.empty((T, k), dtype=np.int32)
    dropped = np.zeros(1, dtype=np.int32)
    _check(lib.oracle_moe_forward(
        T, d, f, N, k, dt, bx.ptr, bg.ptr, pb, bwg.ptr, bwu.ptr, bwd.ptr, fs, *ps,
        float(capacity_factor), y.ctypes.data, logits.ctypes.data, idx.ctypes.data,
        w.ctypes.data, counts.ctypes.data, offsets.ctypes.data, inv.ctypes.data,
        dropped.ctypes.data, nthreads or default_threads()), "oracle_moe_forward")
    return dict(y=y, logits=logits, topk_idx=idx, topk_w=w, counts=counts,
                offsets=offsets, inv_pos=inv, dropped=int(dropped[0]))


def forward_rows(x_rows, topk_idx_rows, topk_w_rows, inv_pos_rows, fetch_expert,
                 shared=None, nthreads=None):
    """Layer output for a subset of tokens, fetching one expert's weights at a time.

    x_rows [R,d] (CPU tensor), topk_idx/topk_w/inv_pos rows [R,k] for those
    tokens (routing and grouping already computed over ALL tokens, because
    capacity drops depend on every earlier token), fetch_expert(e) -> (W_gate_e,
    W_up_e, W_down_e) CPU tensors, shared = None or (Ws_gate, Ws_up, Ws_down).
    Experts are evaluated concurrently (each call releases the GIL).
    Returns y [R,d] fp64.
    """
    import concurrent.futures as cf
    idx = _i32(topk_idx_rows)
    inv = _i32(inv_pos_rows)
    R, k = idx.shape
    d = x_rows.shape[1]
    out = np.zeros((R, k, d), dtype=np.float64)
    experts = sorted(set(int(v) for v in idx[inv >= 0].ravel()))
    cores = nthreads or default_threads()
    workers = max(1, min(cores, len(experts)))
    per_call = max(1, cores // workers)

    def run(e):
        rows, slots = np.nonzero((idx == e) & (inv >= 0))
        wg, wu, wd = fetch_expert(e)
        o = expert_rows(wg, wu, wd, x_rows[torch.as_tensor(rows, dtype=torch.long)], per_call)
        return rows, slots, o

    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        for rows, slots, o in ex.map(run, experts):
            out[rows, slots] = o
    sh = None
    if shared is not None:
        sh = expert_rows(shared[0], shared[1], shared[2], x_rows, cores)
    return combine_rows(inv, topk_w_rows, out, sh)


def routing_stats(counts, logits=None):
    """Routing diagnostics from per-expert assignment counts [N] and, when
    given, the router logits [T,N] (fp64).  Returns a dict: freq [N],
    prob_mean [N] (None without logits), entropy_bits, entropy_max_bits,
    top3 (ids), top3_share, max_share, freq_cv, balance (NaN without logits)."""
    lib = _load()
    c = _i32(counts)
    N = c.shape[0]
    lg = None
    T = 0
    if logits is not None:
        lg = np.ascontiguousarray(logits, dtype=np.float64)
        T = lg.shape[0]
        assert lg.shape[1] == N
    stats = np.empty(6, dtype=np.float64)
    top3 = np.empty(3, dtype=np.int32)
    freq = np.empty(N, dtype=np.float64)
    prob = np.empty(N, dtype=np.float64) if lg is not None else None
    _check(lib.oracle_routing_stats(T, N, _p(lg), c.ctypes.data, stats.ctypes.data,
                                    top3.ctypes.data, freq.ctypes.data, _p(prob)),
           "oracle_routing_stats")
    return dict(freq=freq, prob_mean=prob, entropy_bits=stats[0], entropy_max_bits=stats[1],
                top3=top3, top3_share=stats[2], max_share=stats[3], freq_cv=stats[4],
                balance=stats[5])


def reroute(cand, k, R, N, capacity_rows, logits=None):
    """Capacity overflow re-routed to the next-best expert (see moe_oracle.c,
    oracle_reroute).  cand [T, k+R] the tokens' experts by rank; logits [T,N]
    (fp64) for the final gate weights.  Returns dict final_cand [T,k]
    (candidate index per slot), placed [T,k] bool, final_idx [T,k] (the slot's
    expert; -1 when dropped), rerouted, final_w [T,k] (None without logits)."""
    lib = _load()
    c = _i32(cand)
    T = c.shape[0]
    assert c.shape[1] == k + R
    lg = None if logits is None else np.ascontiguousarray(logits, dtype=np.float64)
    fc = np.empty((T, k), dtype=np.int32)
    pl = np.empty((T, k), dtype=np.int32)
    rr = np.zeros(1, dtype=np.int32)
    fw = np.empty((T, k), dtype=np.float64) if lg is not None else None
    _check(lib.oracle_reroute(T, N, k, R, int(capacity_rows), c.ctypes.data, _p(lg),
                              fc.ctypes.data, pl.ctypes.data, rr.ctypes.data, _p(fw)),
           "oracle_reroute")
    fi = np.take_along_axis(c, fc.astype(np.int64), 1)
    fi[pl == 0] = -1
    return dict(final_cand=fc, placed=pl.astype(bool), final_idx=fi, rerouted=int(rr[0]),
                final_w=fw)


def near_tie_tokens(logits, k, rel=1e-4):
    """Boolean mask of tokens whose k-th and (k+1)-th largest logits differ by
    less than rel * max(|l_k|, |l_k+1|) (the routing near-tie reading)."""
    logits = np.asarray(logits, dtype=np.float64)
    T, N = logits.shape
    if k >= N:
        return np.zeros(T, dtype=bool)
    s = -np.sort(-np.where(np.isnan(logits), -np.inf, logits), axis=1)
    a, b = s[:, k - 1], s[:, k]
    scale = np.maximum(np.abs(a), np.abs(b))
    return np.abs(a - b) < rel * scale




# --------------------------------------------------------------------------
# FP8 E4M3 expert weights and activations (absmax scales; see moe_oracle.c)
# --------------------------------------------------------------------------
def e4m3_decode(codes):
    """Values (fp64) of E4M3 codes (uint8 array of any shape)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_e4m3_decode(c.size, c.ctypes.data, out.ctypes.data)
    return out


def e4m3_encode(values):
    """Nearest E4M3 codes (ties to even, saturating at 448) of fp32 values."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode(v.size, v.ctypes.data, out.ctypes.data)
    return out


def quantize_rows_e4m3(x):
    """Per-row absmax E4M3: x [R,C] -> (codes uint8 [R,C], scales float32 [R])."""
    b = _Buf(x)
    assert b.dtype in (F32, BF16)
    R, C = b.keep.shape
    q = np.empty((R, C), dtype=np.uint8)
    sc = np.empty(R, dtype=np.float32)
    _check(_load().oracle_quantize_rows_e4m3(R, C, b.dtype, b.ptr, q.ctypes.data,
                                             sc.ctypes.data), "oracle_quantize_rows_e4m3")
    return q, sc


def quantize_weights_e4m3(W, nthreads=None):
    """Per-output-channel absmax E4M3 of gate/up weights W [N,d,f]:
    (codes uint8 [N,f,d], scales float32 [N,f])."""
    b = _Buf(W)
    assert b.dtype in (F32, BF16)
    N, d, f = b.keep.shape
    q = np.empty((N, f, d), dtype=np.uint8)
    sc = np.empty((N, f), dtype=np.float32)
    _check(_load().oracle_quantize_weights_e4m3(N, d, f, b.dtype, b.ptr, q.ctypes.data,
                                                sc.ctypes.data, nthreads or default_threads()),
           "oracle_quantize_weights_e4m3")
    return q, sc


def dequantize_e4m3(codes, scales):
    """decode(codes) * scale, one scale per leading-axis row (exact in fp64)."""
    return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[..., None]


def expert_hidden(W_gate_e, W_up_e, xrows, nthreads=None):
    """h[R,f] (fp64) = SiLU(x W_gate_e) * (x W_up_e) for each row of xrows."""
    lib = _load()
    bg, bu, bx = _Buf(W_gate_e), _Buf(W_up_e), _Buf(xrows)
    assert bg.dtype is not None and bg.dtype == bu.dtype
    d, f = bg.keep.shape
    R = bx.keep.shape[0]
    h = np.empty((R, f), dtype=np.float64)
    _check(lib.oracle_expert_hidden(d, f, bg.dtype, bg.ptr, bu.ptr, R, bx.ptr, bx.dtype,
                                    h.ctypes.data, nthreads or default_threads()),
           "oracle_expert_hidden")
    return h


def _u8(a):
    return np.ascontiguousarray(np.asarray(a), dtype=np.uint8)


def _f32(a):
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.float32)


def down_rows_e4m3(h, qd_e, sd_e, nthreads=None):
    """E4M3 down projection of hidden rows h [R,f] (fp64): each row quantised
    per row from its exact values (narrowed to fp32, as the quantiser takes
    them), times W_down's E4M3 channels (codes [d,f], scales [d]).  Returns
    out [R,d] fp64 (see moe_oracle.c)."""
    hh = np.ascontiguousarray(h, dtype=np.float64)
    R, f = hh.shape
    qd, sd = _u8(qd_e), _f32(sd_e)
    d = qd.shape[0]
    assert qd.shape == (d, f) and sd.shape == (d,)
    out = np.empty((R, d), dtype=np.float64)
    _check(_load().oracle_down_rows_e4m3(R, f, d, hh.ctypes.data, qd.ctypes.data,
                                         sd.ctypes.data, out.ctypes.data,
                                         nthreads or default_threads()), "oracle_down_rows_e4m3")
    return out


def expert_rows_fp8(qg_e, sg_e, qu_e, su_e, W_down_e, xq_rows, sx_rows, qd_e=None, sd_e=None,
                    nthreads=None):
    """SwiGLU expert with E4M3 gate/up weights (codes [f,d], scales [f]) on E4M3
    token rows (codes [R,d], scales [R]).  Down projection: W_down_e [f,d] as
    given, or, with qd_e (codes [d,f]) and sd_e (scales [d]), E4M3 too: the
    exact hidden row h is quantised per row like a token row before it.
    Every operand is its exact dequantised value; fp64 throughout, in
    moe_oracle.c."""
    qg, qu, qx = _u8(qg_e), _u8(qu_e), _u8(xq_rows)
    sg, su, sx = _f32(sg_e), _f32(su_e), _f32(sx_rows)
    f, d = qg.shape
    R = qx.shape[0]
    assert qu.shape == (f, d) and qx.shape[1] == d and sx.shape == (R,)
    out = np.empty((R, d), dtype=np.float64)
    wd = qd = sd = None
    wd_dtype, wd_ptr = F32, None
    if qd_e is None:
        wd = _Buf(W_down_e)
        assert wd.keep.shape == (f, d)
        wd_dtype, wd_ptr = wd.dtype, wd.ptr
    else:
        qd, sd = _u8(qd_e), _f32(sd_e)
        assert qd.shape == (d, f) and sd.shape == (d,)
    _check(_load().oracle_expert_rows_e4m3(
        d, f, qg.ctypes.data, sg.ctypes.data, qu.ctypes.data, su.ctypes.data, R,
        qx.ctypes.data, sx.ctypes.data, wd_dtype, wd_ptr,
        None if qd is None else qd.ctypes.data, None if sd is None else sd.ctypes.data,
        out.ctypes.data, nthreads or default_threads()), "oracle_expert_rows_e4m3")
    return out


def forward_rows_fp8(xq_rows, sx_rows, topk_idx_rows, topk_w_rows, inv_pos_rows,
                     fetch_expert_fp8, shared=None, x_rows=None, nthreads=None):
    """Layer output for a subset of tokens with E4M3 gate/up weights and token
    rows: fetch_expert_fp8(e) -> (qg [f,d], sg [f], qu [f,d], su [f], W_down [f,d])
    or the same plus (qd [d,f], sd [d]) for an E4M3 down projection.
    Experts one at a time (each dequantised expert is held in fp64).  The
    shared expert (Ws_gate, Ws_up, Ws_down), when given, runs in the layer's
    own precision on x_rows.  Returns y [R,d] fp64."""
    idx = _i32(topk_idx_rows)
    inv = _i32(inv_pos_rows)
    R, k = idx.shape
    d = xq_rows.shape[1]
    out = np.zeros((R, k, d), dtype=np.float64)
    for e in sorted(set(int(v) for v in idx[inv >= 0].ravel())):
        rows, slots = np.nonzero((idx == e) & (inv >= 0))
        w = fetch_expert_fp8(e)          # qg, sg, qu, su, W_down (, qd, sd)
        out[rows, slots] = expert_rows_fp8(*w[:5], xq_rows[rows], sx_rows[rows],
                                           *(w[5:7] if len(w) > 5 else (None, None)),
                                           nthreads=nthreads)
    sh = None
    if shared is not None:
        sh = expert_rows(shared[0], shared[1], shared[2], x_rows, nthreads)
    return combine_rows(inv, topk_w_rows, out, sh)
