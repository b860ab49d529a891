"""ctypes binding to libmoe.so -- argument marshalling only.

Every function here has the name of the C entry point it calls (see
include/moe.h), takes torch CUDA tensors, passes their device addresses and
sizes, and enqueues on torch's current CUDA stream.  No step of the layer runs
in Python or on the CPU: if libmoe.so is missing or the device is not a
B300, the calls raise.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_F32, MOE_BF16 = 0, 1
MOE_DEV_BAD_EXPERT_ID, MOE_DEV_NAN_LOGIT, MOE_DEV_TIMEOUT, MOE_DEV_BAD_TILE = 1, 2, 4, 8
MOE_DEV_BAD_COUNTS, MOE_DEV_BAD_ROW = 16, 32
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
          3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE"}

# Every symbol the header declares.
EXPORTS = ("moe_status_string", "moe_last_error", "moe_version", "moe_launch_counter",
           "moe_capacity",
           "moe_router_topk", "moe_permute_workspace_size", "moe_permute",
           "moe_permute_noalloc",
           "moe_expert_ffn_workspace_size", "moe_expert_ffn", "moe_expert_ffn_to_rows",
           "moe_combine",
           "moe_forward_workspace_size", "moe_forward", "moe_forward_host_io",
           "moe_forward_overlap_chunks", "moe_forward_host_io_overlapped",
           "moe_routing_stats_workspace_size", "moe_routing_stats",
           "moe_permute_reroute_workspace_size", "moe_permute_reroute",
           "moe_quantize_weights_e4m3", "moe_quantize_rows_e4m3",
           "moe_expert_ffn_fp8_workspace_size", "moe_expert_ffn_fp8",
           "moe_ep_regroup", "moe_ep_return")


class MoEError(RuntimeError):
    def __init__(self, name, code, msg):
        super().__init__(f"{name} -> {STATUS.get(code, code)}: {msg}")
        self.code = code


class moe_forward_args(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("d", ctypes.c_int), ("f", ctypes.c_int),
                ("N", ctypes.c_int), ("k", ctypes.c_int), ("dtype", ctypes.c_int),
                ("x", ctypes.c_void_p), ("W_g", ctypes.c_void_p),
                ("router_bias", ctypes.c_void_p), ("W_gate", ctypes.c_void_p),
                ("W_up", ctypes.c_void_p), ("W_down", ctypes.c_void_p),
                ("fs", ctypes.c_int), ("Ws_gate", ctypes.c_void_p),
                ("Ws_up", ctypes.c_void_p), ("Ws_down", ctypes.c_void_p),
                ("capacity_factor", ctypes.c_float), ("y", ctypes.c_void_p),
                ("y_dtype", ctypes.c_int), ("logits", ctypes.c_void_p),
                ("topk_idx", ctypes.c_void_p), ("topk_w", ctypes.c_void_p),
                ("counts", ctypes.c_void_p), ("offsets", ctypes.c_void_p),
                ("inv_pos", ctypes.c_void_p), ("dropped", ctypes.c_void_p),
                ("device_status", ctypes.c_void_p), ("reroute_rounds", ctypes.c_int),
                ("rerouted", ctypes.c_void_p), ("Wq_gate", ctypes.c_void_p),
                ("wscale_gate", ctypes.c_void_p), ("Wq_up", ctypes.c_void_p),
                ("wscale_up", ctypes.c_void_p), ("Wq_down", ctypes.c_void_p),
                ("wscale_down", ctypes.c_void_p), ("ffn_event_begin", ctypes.c_void_p),
                ("ffn_event_end", ctypes.c_void_p)]


_lib = None


def lib():
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmoe.so not built ({LIB_PATH}); run "
                               "python -m sparse_mixture_experts_63_b300.build")
        L = ctypes.CDLL(LIB_PATH)
        vp, ci, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [ci]
        L.moe_last_error.restype = ctypes.c_char_p
        L.moe_version.restype = ctypes.c_char_p
        L.moe_launch_counter.restype = ctypes.c_uint64
        L.moe_capacity.argtypes = [ctypes.c_float, ci, ci, ci]
        L.moe_capacity.restype = ci
        L.moe_router_topk.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, vp, vp, vp, vp, vp]
        L.moe_permute_workspace_size.argtypes = [ci, ci, ci]
        L.moe_permute_workspace_size.restype = sz
        L.moe_permute.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, ci, vp, vp, vp, vp, vp, vp,
                                  vp, vp, vp, sz, vp]
        L.moe_permute_noalloc.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, ci, vp, vp, vp, vp, vp,
                                          vp, vp, vp, vp]
        L.moe_expert_ffn_workspace_size.argtypes = [ci, ci, ci, ci, ci]
        L.moe_expert_ffn_workspace_size.restype = sz
        L.moe_expert_ffn.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, vp, vp, vp, vp, vp, vp,
                                     sz, vp]
        L.moe_expert_ffn_to_rows.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, vp, vp, vp, vp,
                                             ci, vp, vp, sz, vp]
        L.moe_combine.argtypes = [vp, ci, vp, ci, ci, ci, vp, vp, ci, vp]
        L.moe_forward_workspace_size.argtypes = [ctypes.POINTER(moe_forward_args)]
        L.moe_forward_workspace_size.restype = sz
        L.moe_forward.argtypes = [ctypes.POINTER(moe_forward_args), vp, sz, vp]
        L.moe_forward_host_io.argtypes = [ctypes.POINTER(moe_forward_args), vp, vp, vp, sz, vp]
        L.moe_forward_overlap_chunks.argtypes = [ctypes.POINTER(moe_forward_args)]
        L.moe_forward_overlap_chunks.restype = ci
        L.moe_forward_host_io_overlapped.argtypes = [ctypes.POINTER(moe_forward_args), vp, vp,
                                                     vp, sz, ci, vp, vp, vp]
        L.moe_routing_stats_workspace_size.argtypes = [ci, ci]
        L.moe_routing_stats_workspace_size.restype = sz
        L.moe_routing_stats.argtypes = [vp, vp, ci, ci, vp, vp, vp, vp, sz, vp]
        L.moe_permute_reroute_workspace_size.argtypes = [ci, ci, ci, ci]
        L.moe_permute_reroute_workspace_size.restype = sz
        L.moe_permute_reroute.argtypes = ([vp, vp, vp, ci, ci, ci, ci, ci, ci, ci] + [vp] * 13 +
                                          [sz, vp])
        L.moe_quantize_weights_e4m3.argtypes = [vp, ci, ci, ci, vp, vp, vp]
        L.moe_quantize_rows_e4m3.argtypes = [vp, ci, ci, vp, vp, vp]
        L.moe_expert_ffn_fp8_workspace_size.argtypes = [ci, ci, ci, ci, ci]
        L.moe_expert_ffn_fp8_workspace_size.restype = sz
        L.moe_expert_ffn_fp8.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, vp, vp, vp, vp, vp,
                                         vp, vp, vp, vp, vp, sz, vp]
        L.moe_ep_regroup.argtypes = [vp, ci, ci, vp, vp, ci, ci, ci, vp, vp, vp, vp, vp, vp, vp]
        L.moe_ep_return.argtypes = [vp, vp, ci, ci, ci, vp, vp]
        for n in ("moe_router_topk", "moe_permute", "moe_permute_noalloc", "moe_expert_ffn",
                  "moe_ep_regroup", "moe_ep_return",
                  "moe_quantize_weights_e4m3", "moe_quantize_rows_e4m3", "moe_expert_ffn_fp8",
                  "moe_combine", "moe_routing_stats", "moe_permute_reroute",
                  "moe_forward", "moe_forward_host_io", "moe_forward_host_io_overlapped"):
            getattr(L, n).restype = ci
        _lib = L
    return _lib


def _check(name, code):
    if code != 0:
        raise MoEError(name, code, lib().moe_last_error().decode())


def _p(t):
    return None if t is None else t.data_ptr()


def _dt(t):
    if t.dtype == torch.bfloat16:
        return MOE_BF16
    if t.dtype == torch.float32:
        return MOE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


# ---------------------------------------------------------------------------
def moe_version() -> str:
    return lib().moe_version().decode()


def moe_launch_counter() -> int:
    return int(lib().moe_launch_counter())


def moe_capacity(capacity_factor, T, k, N) -> int:
    return int(lib().moe_capacity(float(capacity_factor), T, k, N))


def moe_router_topk(x, W_g, k, bias=None, logits=None, topk_idx=None, topk_w=None,
                    device_status=None, stream=None):
    """Returns (topk_idx [T,k] int32, topk_w [T,k] fp32); fills logits if given."""
    _cuda(x, W_g, bias, logits)
    T, d = x.shape
    N = W_g.shape[1]
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=x.device)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=x.device)
    _check("moe_router_topk", lib().moe_router_topk(
        _p(x), _p(W_g), _p(bias), _dt(x), T, d, N, k, _p(logits), _p(topk_idx), _p(topk_w),
        _p(device_status), _stream(stream)))
    return topk_idx, topk_w


def moe_permute(topk_idx, N, x=None, topk_w=None, capacity=0, gather=True,
                device_status=None, stream=None, A_max=None):
    """Returns dict counts, offsets, perm_token, row_scale, inv_pos, x_perm, dropped."""
    _cuda(topk_idx, x, topk_w)
    T, k = topk_idx.shape
    dev = topk_idx.device
    d = x.shape[1] if x is not None else 0
    A = T * k if A_max is None else A_max
    out = dict(counts=torch.empty(N, dtype=torch.int32, device=dev),
               offsets=torch.empty(N + 1, dtype=torch.int32, device=dev),
               perm_token=torch.empty(max(T * k, 1), dtype=torch.int32, device=dev),
               row_scale=(torch.empty(max(T * k, 1), dtype=torch.float32, device=dev)
                          if topk_w is not None else None),
               inv_pos=torch.empty((T, k), dtype=torch.int32, device=dev),
               x_perm=(torch.empty((max(A, 1), d), dtype=x.dtype, device=dev)
                       if (gather and x is not None) else None),
               dropped=torch.zeros(1, dtype=torch.int32, device=dev))
    ws_bytes = lib().moe_permute_workspace_size(T, N, k)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    _check("moe_permute", lib().moe_permute(
        _p(topk_idx), _p(topk_w), _p(x), _dt(x) if x is not None else MOE_BF16, T, d, N, k,
        int(capacity), _p(out["counts"]), _p(out["offsets"]), _p(out["perm_token"]),
        _p(out["row_scale"]), _p(out["inv_pos"]), _p(out["x_perm"]), _p(out["dropped"]),
        _p(device_status), _p(ws), ws_bytes, _stream(stream)))
    return out


def moe_permute_noalloc(topk_idx, N, x=None, topk_w=None, capacity=0, gather=True,
                        device_status=None, stream=None, A_max=None):
    """moe_permute without a workspace: the library's fixed scratch is used
    instead (see include/moe.h for its size limit and sharing rules)."""
    _cuda(topk_idx, x, topk_w)
    T, k = topk_idx.shape
    dev = topk_idx.device
    d = x.shape[1] if x is not None else 0
    A = T * k if A_max is None else A_max
    out = dict(counts=torch.empty(N, dtype=torch.int32, device=dev),
               offsets=torch.empty(N + 1, dtype=torch.int32, device=dev),
               perm_token=torch.empty(max(T * k, 1), dtype=torch.int32, device=dev),
               row_scale=(torch.empty(max(T * k, 1), dtype=torch.float32, device=dev)
                          if topk_w is not None else None),
               inv_pos=torch.empty((T, k), dtype=torch.int32, device=dev),
               x_perm=(torch.empty((max(A, 1), d), dtype=x.dtype, device=dev)
                       if (gather and x is not None) else None),
               dropped=torch.zeros(1, dtype=torch.int32, device=dev))
    _check("moe_permute_noalloc", lib().moe_permute_noalloc(
        _p(topk_idx), _p(topk_w), _p(x), _dt(x) if x is not None else MOE_BF16, T, d, N, k,
        int(capacity), _p(out["counts"]), _p(out["offsets"]), _p(out["perm_token"]),
        _p(out["row_scale"]), _p(out["inv_pos"]), _p(out["x_perm"]), _p(out["dropped"]),
        _p(device_status), _stream(stream)))
    return out


def moe_expert_ffn(x_perm, offsets, W_gate, W_up, W_down, row_scale=None, y_perm=None,
                   device_status=None, stream=None, A_max=None, out_row=None, rows_out=None):
    """y_perm [A_max,d] = row_scale * SwiGLU_e(x_perm) for each expert's rows.
    With out_row (int32 [A_max]): moe_expert_ffn_to_rows, row p stored at
    y_perm row out_row[p] of rows_out rows."""
    _cuda(x_perm, offsets, W_gate, W_up, W_down, row_scale, y_perm, out_row)
    A = x_perm.shape[0] if A_max is None else A_max
    d = x_perm.shape[1]
    N, _, f = W_gate.shape
    rows = A if out_row is None else (A if rows_out is None else rows_out)
    if y_perm is None:
        y_perm = torch.empty((max(rows, 1), d), dtype=x_perm.dtype, device=x_perm.device)
    ws_bytes = lib().moe_expert_ffn_workspace_size(A, d, f, N, _dt(x_perm))
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=x_perm.device)
    if out_row is not None:
        _check("moe_expert_ffn_to_rows", lib().moe_expert_ffn_to_rows(
            _p(x_perm), _p(offsets), _p(row_scale), _p(out_row), A, d, f, N, _dt(x_perm),
            _p(W_gate), _p(W_up), _p(W_down), _p(y_perm), rows, _p(device_status), _p(ws),
            ws_bytes, _stream(stream)))
        return y_perm
    _check("moe_expert_ffn", lib().moe_expert_ffn(
        _p(x_perm), _p(offsets), _p(row_scale), A, d, f, N, _dt(x_perm), _p(W_gate),
        _p(W_up), _p(W_down), _p(y_perm), _p(device_status), _p(ws), ws_bytes,
        _stream(stream)))
    return y_perm


def quantize_weights_e4m3(W, stream=None):
    """Weights W [N,K,M] bf16 (K the reduction dim: gate/up [N,d,f], down
    [N,f,d]) -> (codes uint8 [N,M,K], scales fp32 [N,M]), E4M3 with one absmax
    scale per output channel."""
    _cuda(W)
    N, d, f = W.shape
    q = torch.empty((N, f, d), dtype=torch.uint8, device=W.device)
    sc = torch.empty((N, f), dtype=torch.float32, device=W.device)
    _check("moe_quantize_weights_e4m3", lib().moe_quantize_weights_e4m3(
        _p(W), N, d, f, _p(q), _p(sc), _stream(stream)))
    return q, sc


def quantize_rows_e4m3(x, stream=None):
    """Rows x [R,C] bf16 -> (codes uint8 [R,C], scales fp32 [R]), E4M3 per row."""
    _cuda(x)
    R, C = x.shape
    q = torch.empty((R, C), dtype=torch.uint8, device=x.device)
    sc = torch.empty(max(R, 1), dtype=torch.float32, device=x.device)
    _check("moe_quantize_rows_e4m3", lib().moe_quantize_rows_e4m3(
        _p(x), R, C, _p(q), _p(sc), _stream(stream)))
    return q, sc[:R]


def moe_expert_ffn_fp8(xq_perm, x_scale, perm_token, offsets, Wq_gate, wscale_gate, Wq_up,
                       wscale_up, W_down=None, Wq_down=None, wscale_down=None, row_scale=None,
                       y_perm=None, device_status=None, stream=None, A_max=None):
    """moe_expert_ffn with E4M3 gate/up (codes [N,f,d] + channel scales [N,f]) on
    E4M3 permuted token rows xq_perm [A_max,d] (row p's scale x_scale[perm_token[p]]);
    the down projection from W_down (bf16) or, given Wq_down [N,d,f] and
    wscale_down [N,d], in E4M3 on h quantised per row."""
    _cuda(xq_perm, x_scale, perm_token, offsets, Wq_gate, wscale_gate, Wq_up, wscale_up, W_down,
          Wq_down, wscale_down, row_scale, y_perm)
    A = xq_perm.shape[0] if A_max is None else A_max
    d = xq_perm.shape[1]
    N, f, _ = Wq_gate.shape
    if y_perm is None:
        y_perm = torch.empty((max(A, 1), d), dtype=torch.bfloat16, device=xq_perm.device)
    ws_bytes = lib().moe_expert_ffn_fp8_workspace_size(A, d, f, N, int(Wq_down is not None))
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=xq_perm.device)
    _check("moe_expert_ffn_fp8", lib().moe_expert_ffn_fp8(
        _p(xq_perm), _p(x_scale), _p(perm_token), _p(offsets), _p(row_scale), A, d, f, N,
        _p(Wq_gate), _p(wscale_gate), _p(Wq_up), _p(wscale_up), _p(W_down), _p(Wq_down),
        _p(wscale_down), _p(y_perm), _p(device_status), _p(ws), ws_bytes, _stream(stream)))
    return y_perm


class moe_routing_stats_t(ctypes.Structure):
    _fields_ = [("entropy_bits", ctypes.c_float), ("entropy_max_bits", ctypes.c_float),
                ("top3_share", ctypes.c_float), ("max_share", ctypes.c_float),
                ("freq_cv", ctypes.c_float), ("balance", ctypes.c_float),
                ("top3", ctypes.c_int32 * 3), ("assignments", ctypes.c_int32)]


def moe_routing_stats(counts, logits=None, stream=None):
    """Routing diagnostics on the device.  counts [N] int32 (before capacity),
    logits [T,N] fp32 or None.  Returns (stats, freq, prob_mean): stats a uint8
    device tensor holding one moe_routing_stats_t (read it with
    routing_stats_dict after a sync), freq [N] and prob_mean [N] (None without
    logits) fp32 device tensors."""
    _cuda(counts, logits)
    N = counts.shape[0]
    T = logits.shape[0] if logits is not None else 0
    dev = counts.device
    stats = torch.empty(ctypes.sizeof(moe_routing_stats_t), dtype=torch.uint8, device=dev)
    freq = torch.empty(N, dtype=torch.float32, device=dev)
    prob = torch.empty(N, dtype=torch.float32, device=dev) if logits is not None else None
    ws_bytes = lib().moe_routing_stats_workspace_size(T, N) if logits is not None else 0
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    _check("moe_routing_stats", lib().moe_routing_stats(
        _p(logits), _p(counts), T, N, _p(stats), _p(freq), _p(prob), _p(ws), ws_bytes,
        _stream(stream)))
    return stats, freq, prob


def routing_stats_dict(stats):
    """moe_routing_stats_t from the device buffer returned by moe_routing_stats."""
    raw = bytes(stats.cpu().numpy().tobytes())
    st = moe_routing_stats_t.from_buffer_copy(raw)
    return dict(entropy_bits=st.entropy_bits, entropy_max_bits=st.entropy_max_bits,
                top3_share=st.top3_share, max_share=st.max_share, freq_cv=st.freq_cv,
                balance=st.balance, top3=list(st.top3), assignments=st.assignments)


def moe_permute_reroute(cand_idx, cand_w, N, k, capacity, x=None, demand=False,
                        device_status=None, stream=None):
    """Dispatch with capacity overflow re-routed (cand_idx/cand_w [T, k+R] from
    moe_router_topk with k+R).  Returns dict final_idx, final_w, counts,
    offsets, perm_token, row_scale, inv_pos, x_perm (if x), dropped, rerouted,
    demand (if asked)."""
    _cuda(cand_idx, cand_w, x)
    T, kr = cand_idx.shape
    R = kr - k
    dev = cand_idx.device
    d = x.shape[1] if x is not None else 0
    A = T * k
    out = dict(final_idx=torch.empty((T, k), dtype=torch.int32, device=dev),
               final_w=torch.empty((T, k), dtype=torch.float32, device=dev),
               counts=torch.empty(N, dtype=torch.int32, device=dev),
               offsets=torch.empty(N + 1, dtype=torch.int32, device=dev),
               perm_token=torch.empty(max(A, 1), dtype=torch.int32, device=dev),
               row_scale=torch.empty(max(A, 1), dtype=torch.float32, device=dev),
               inv_pos=torch.empty((T, k), dtype=torch.int32, device=dev),
               dropped=torch.zeros(1, dtype=torch.int32, device=dev),
               rerouted=torch.zeros(1, dtype=torch.int32, device=dev))
    if demand:
        out["demand"] = torch.empty(N, dtype=torch.int32, device=dev)
    if x is not None:
        out["x_perm"] = torch.empty((max(A, 1), d), dtype=x.dtype, device=dev)
    ws_bytes = lib().moe_permute_reroute_workspace_size(T, N, k, R)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    _check("moe_permute_reroute", lib().moe_permute_reroute(
        _p(cand_idx), _p(cand_w), _p(x), _dt(x) if x is not None else 1, T, d, N, k, R,
        int(capacity), _p(out["final_idx"]), _p(out["final_w"]), _p(out.get("demand")),
        _p(out["counts"]), _p(out["offsets"]), _p(out["perm_token"]), _p(out["row_scale"]),
        _p(out["inv_pos"]), _p(out.get("x_perm")), _p(out["dropped"]), _p(out["rerouted"]),
        _p(device_status), _p(ws), ws_bytes, _stream(stream)))
    return out


def moe_combine(y_perm, inv_pos, shared_y=None, y=None, y_dtype=torch.float32, stream=None):
    _cuda(y_perm, inv_pos, shared_y, y)
    T, k = inv_pos.shape
    d = y_perm.shape[1]
    if y is None:
        y = torch.empty((T, d), dtype=y_dtype, device=y_perm.device)
    _check("moe_combine", lib().moe_combine(
        _p(y_perm), _dt(y_perm), _p(inv_pos), T, k, d, _p(shared_y), _p(y), _dt(y),
        _stream(stream)))
    return y


def moe_ep_regroup(recv_counts, Ne, x_recv, row_scale_recv=None, device_status=None,
                   stream=None):
    """Rows received from G source ranks (block (s, e) = recv_counts[s*Ne + e]
    rows, in (s, e) order) regrouped by local expert.  Returns dict x_local,
    row_scale_local (or None), offsets_local [Ne+1], dest [R] (where received
    row i went) and src [R] (its inverse: the received row of local row p)."""
    _cuda(recv_counts, x_recv, row_scale_recv)
    G = recv_counts.numel() // Ne
    R, d = x_recv.shape
    dev = x_recv.device
    out = dict(x_local=torch.empty((max(R, 1), d), dtype=x_recv.dtype, device=dev),
               row_scale_local=(torch.empty(max(R, 1), dtype=torch.float32, device=dev)
                                if row_scale_recv is not None else None),
               offsets_local=torch.empty(Ne + 1, dtype=torch.int32, device=dev),
               dest=torch.empty(max(R, 1), dtype=torch.int32, device=dev),
               src=torch.empty(max(R, 1), dtype=torch.int32, device=dev))
    _check("moe_ep_regroup", lib().moe_ep_regroup(
        _p(recv_counts), G, Ne, _p(x_recv), _p(row_scale_recv), R, d, _dt(x_recv),
        _p(out["x_local"]), _p(out["row_scale_local"]), _p(out["offsets_local"]),
        _p(out["dest"]), _p(out["src"]), _p(device_status), _stream(stream)))
    return out


def moe_ep_return(y_local, dest, R, y_back=None, stream=None):
    """y_back[i] = y_local[dest[i]] for the R received rows."""
    _cuda(y_local, dest, y_back)
    d = y_local.shape[1]
    if y_back is None:
        y_back = torch.empty((max(R, 1), d), dtype=y_local.dtype, device=y_local.device)
    _check("moe_ep_return", lib().moe_ep_return(
        _p(y_local), _p(dest), R, d, _dt(y_local), _p(y_back), _stream(stream)))
    return y_back


def make_forward_args(x, W_g, W_gate, W_up, W_down, k, y, bias=None, Ws_gate=None,
                      Ws_up=None, Ws_down=None, capacity_factor=0.0, outputs=None,
                      device_status=None, reroute_rounds=0, fp8_gate_up=None):
    _cuda(x, W_g, W_gate, W_up, W_down, y, bias, Ws_gate, Ws_up, Ws_down)
    T, d = x.shape
    N, _, f = W_gate.shape
    o = outputs or {}
    a = moe_forward_args()
    a.T, a.d, a.f, a.N, a.k, a.dtype = T, d, f, N, k, _dt(x)
    a.x, a.W_g, a.router_bias = _p(x), _p(W_g), _p(bias)
    a.W_gate, a.W_up, a.W_down = _p(W_gate), _p(W_up), _p(W_down)
    a.fs = 0 if Ws_gate is None else Ws_gate.shape[1]
    a.Ws_gate, a.Ws_up, a.Ws_down = _p(Ws_gate), _p(Ws_up), _p(Ws_down)
    a.capacity_factor = float(capacity_factor)
    a.y, a.y_dtype = _p(y), _dt(y)
    for key in ("logits", "topk_idx", "topk_w", "counts", "offsets", "inv_pos", "dropped"):
        setattr(a, key, _p(o.get(key)))
    a.device_status = _p(device_status)
    a.reroute_rounds = int(reroute_rounds)
    a.rerouted = _p(o.get("rerouted"))
    if fp8_gate_up is not None:   # (Wq_gate, wscale_gate, Wq_up, wscale_up[, Wq_down, wscale_down])
        _cuda(*fp8_gate_up)
        a.Wq_gate, a.wscale_gate, a.Wq_up, a.wscale_up = (_p(t) for t in fp8_gate_up[:4])
        if len(fp8_gate_up) > 4:
            a.Wq_down, a.wscale_down = _p(fp8_gate_up[4]), _p(fp8_gate_up[5])
    return a


def moe_forward_workspace_size(args) -> int:
    n = lib().moe_forward_workspace_size(ctypes.byref(args))
    if n == 0:
        raise MoEError("moe_forward_workspace_size", 1, lib().moe_last_error().decode())
    return n


def moe_forward(args, workspace, stream=None):
    _check("moe_forward", lib().moe_forward(ctypes.byref(args), _p(workspace),
                                            workspace.numel(), _stream(stream)))


def moe_forward_host_io(args, x_host, y_host, workspace, stream=None):
    if x_host.is_cuda or y_host.is_cuda:
        raise ValueError("x_host / y_host must be host tensors")
    _check("moe_forward_host_io", lib().moe_forward_host_io(
        ctypes.byref(args), _p(x_host), _p(y_host), _p(workspace), workspace.numel(),
        _stream(stream)))


_copy_streams = {}


def moe_forward_host_io_overlapped(args, x_host, y_host, workspace, chunks=0, stream=None):
    """moe_forward_host_io with the copies overlapped with the layer (token
    chunks; see include/moe.h).  The two copy streams are the binding's own,
    one pair per device."""
    if x_host.is_cuda or y_host.is_cuda:
        raise ValueError("x_host / y_host must be host tensors")
    dev = torch.cuda.current_device()
    if dev not in _copy_streams:
        _copy_streams[dev] = (torch.cuda.Stream(), torch.cuda.Stream())
    h2d, d2h = _copy_streams[dev]
    _check("moe_forward_host_io_overlapped", lib().moe_forward_host_io_overlapped(
        ctypes.byref(args), _p(x_host), _p(y_host), _p(workspace), workspace.numel(), int(chunks),
        _stream(stream), _stream(h2d), _stream(d2h)))


def moe_forward_overlap_chunks(args) -> int:
    return int(lib().moe_forward_overlap_chunks(ctypes.byref(args)))


class MoELayer:
    """Convenience holder: the layer's weights plus a reusable workspace.

    ``layer(x)`` returns y [T,d] (fp32 by default) and keeps the routing
    outputs of the last call in ``layer.last``.  ``fp8=True`` quantises the
    routed experts' gate/up weights to E4M3 once (per-channel scales) and runs
    those projections in FP8 (x quantised per token on the fly);
    ``fp8_down=True`` does the same for the down projection (h quantised per
    row on the fly).
    """

    def __init__(self, W_g, W_gate, W_up, W_down, k, bias=None, Ws_gate=None, Ws_up=None,
                 Ws_down=None, capacity_factor=0.0, y_dtype=torch.float32, reroute_rounds=0,
                 fp8=False, fp8_down=False):
        self.reroute_rounds = reroute_rounds
        self.fp8 = None
        if fp8 or fp8_down:
            qg, sg = quantize_weights_e4m3(W_gate)
            qu, su = quantize_weights_e4m3(W_up)
            self.fp8 = (qg, sg, qu, su)
            if fp8_down:   # W_down [N,f,d] read as [N, K=f, M=d]
                self.fp8 += quantize_weights_e4m3(W_down)
        self.W_g, self.W_gate, self.W_up, self.W_down = W_g, W_gate, W_up, W_down
        self.k, self.bias, self.cf, self.y_dtype = k, bias, capacity_factor, y_dtype
        self.Ws_gate, self.Ws_up, self.Ws_down = Ws_gate, Ws_up, Ws_down
        self._ws = None
        self.last = None

    def outputs_for(self, T, device, logits=False):
        N = self.W_gate.shape[0]
        k = self.k
        o = dict(topk_idx=torch.empty((T, k), dtype=torch.int32, device=device),
                 topk_w=torch.empty((T, k), dtype=torch.float32, device=device),
                 counts=torch.empty(N, dtype=torch.int32, device=device),
                 offsets=torch.empty(N + 1, dtype=torch.int32, device=device),
                 inv_pos=torch.empty((T, k), dtype=torch.int32, device=device),
                 dropped=torch.zeros(1, dtype=torch.int32, device=device),
                 rerouted=torch.zeros(1, dtype=torch.int32, device=device),
                 device_status=torch.zeros(1, dtype=torch.int32, device=device))
        if logits:
            o["logits"] = torch.empty((T, N), dtype=torch.float32, device=device)
        return o

    def args(self, x, y, outputs):
        return make_forward_args(x, self.W_g, self.W_gate, self.W_up, self.W_down, self.k, y,
                                 bias=self.bias, Ws_gate=self.Ws_gate, Ws_up=self.Ws_up,
                                 Ws_down=self.Ws_down, capacity_factor=self.cf,
                                 outputs=outputs, device_status=outputs.get("device_status"),
                                 reroute_rounds=self.reroute_rounds, fp8_gate_up=self.fp8)

    def workspace(self, args, device):
        n = moe_forward_workspace_size(args)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(n, dtype=torch.uint8, device=device)
        return self._ws

    def __call__(self, x, logits=False, stream=None):
        T, d = x.shape
        y = torch.empty((T, d), dtype=self.y_dtype, device=x.device)
        o = self.outputs_for(T, x.device, logits)
        a = self.args(x, y, o)
        moe_forward(a, self.workspace(a, x.device), stream)
        self.last = o
        return y
