"""Expert-parallel MoE layer: the experts split over G ranks, two all-to-all
exchanges per layer.

Source: "MoE 分片：混合專家模型的平行化策略", sections 專家平行化詳解 (each of G
GPUs holds N/G experts) and 動態 token 路由 steps 3-5 (dispatch all-to-all,
expert compute, combine all-to-all); "MoE稀疏激活原理与工程实践", 2.2.

Rank r holds experts [r*Ne, (r+1)*Ne), Ne = N/G, and its own batch of tokens.
One forward, per rank:
  1. router, top-k and dispatch over all N experts (moe_router_topk,
     moe_permute): x_perm is ordered by expert, so the rows bound for rank q
     are one contiguous range of it;
  2. exchange of the kept counts per expert (G*Ne int32: Ne to each rank);
  3. exchange of the rows and their gate weights (row_scale);
  4. regroup by local expert (moe_ep_regroup), then the local grouped SwiGLU
     FFN (gate weight applied in its epilogue) storing each output row at its
     received position (moe_expert_ffn_to_rows with the regroup's inverse
     map), ready for the return exchange;
  5. the reverse exchange of the output rows, which land in the source rank's
     own x_perm order;
  6. combine (moe_combine) into y, with the optional always-on shared expert
     (replicated: each rank runs it on its own tokens with moe_expert_ffn).
Every step on the device is a libmoe kernel; this module only computes the
split sizes and calls the exchange.  The exchange is an object with one
method, all_to_all(out, inp, out_splits, in_splits), with the semantics of
torch.distributed.all_to_all_single (TorchDistExchange: NCCL between GPUs,
gloo on CPU).  Rows go to the receiver's own memory before any kernel reads
them; no multicast and no peer operand is used.  The split sizes need the
counts on the host: two device-to-host reads of a few hundred integers per
forward (offsets before the row exchange, received counts after the counts
exchange).
"""
from dataclasses import dataclass
from typing import List, Optional

import torch

from . import binding as B


class TorchDistExchange:
    """all_to_all through torch.distributed (the process group's backend)."""

    def __init__(self, group=None):
        self.group = group

    def all_to_all(self, out, inp, out_splits, in_splits):
        import torch.distributed as dist
        dist.all_to_all_single(out, inp, out_splits, in_splits, group=self.group)


def plan_from_offsets(offsets, G: int, Ne: int):
    """From moe_permute's offsets [N+1] (host): the kept rows per expert
    (int32 [G*Ne], the counts to exchange) and the rows per destination rank."""
    off = [int(v) for v in offsets]
    assert len(off) == G * Ne + 1
    counts = torch.tensor([off[e + 1] - off[e] for e in range(G * Ne)], dtype=torch.int32)
    send_rows = [off[(q + 1) * Ne] - off[q * Ne] for q in range(G)]
    return counts, send_rows


def recv_rows_from_counts(recv_counts, G: int, Ne: int) -> List[int]:
    """Rows arriving from each source rank: the sum of its block of Ne counts."""
    c = [int(v) for v in recv_counts]
    return [sum(c[s * Ne:(s + 1) * Ne]) for s in range(G)]


def exchange_counts(exchange, counts, G: int, Ne: int):
    """Each rank sends Ne counts to every rank; rank r receives [s][e] = the
    rows source s sends for r's local expert e."""
    out = torch.empty_like(counts)
    exchange.all_to_all(out, counts.contiguous(), [Ne] * G, [Ne] * G)
    return out


def exchange_rows(exchange, send, send_rows: List[int], recv_rows: List[int]):
    """Variable-size all-to-all of rows (first dimension) of `send`."""
    out = torch.empty((max(sum(recv_rows), 1),) + tuple(send.shape[1:]), dtype=send.dtype,
                      device=send.device)
    exchange.all_to_all(out[:sum(recv_rows)], send[:sum(send_rows)].contiguous(), recv_rows,
                        send_rows)
    return out


@dataclass
class EPState:
    """What one rank keeps between the steps of a forward."""
    T: int
    A: int                      # kept rows of this rank's tokens
    perm: dict                  # moe_permute outputs (inv_pos, x_perm, row_scale, ...)
    counts: torch.Tensor        # kept rows per expert [G*Ne] (host)
    send_rows: List[int]
    recv_counts: Optional[torch.Tensor] = None   # [G*Ne] on the device
    recv_rows: Optional[List[int]] = None
    shared_y: Optional[torch.Tensor] = None      # [T,d] shared expert output, if any


class ExpertParallelMoE:
    """One rank's part of an expert-parallel layer.

    W_g [d,N], bias [N] and the shared expert (Ws_gate, Ws_up [d,fs], Ws_down
    [fs,d], optional) are replicated; W_gate_local / W_up_local [Ne,d,f] and
    W_down_local [Ne,f,d] are this rank's experts [rank*Ne, (rank+1)*Ne).
    `forward(x)` runs the whole layer with `exchange`; the step methods
    (dispatch, post_counts, experts, combine) let a caller drive several ranks
    in one process with its own exchange."""

    def __init__(self, W_g, W_gate_local, W_up_local, W_down_local, k, rank, world, exchange=None,
                 bias=None, capacity_factor=0.0, y_dtype=torch.float32, Ws_gate=None, Ws_up=None,
                 Ws_down=None):
        self.W_g, self.bias, self.k = W_g, bias, k
        self.Wg, self.Wu, self.Wd = W_gate_local, W_up_local, W_down_local
        self.rank, self.G = rank, world
        self.Ne = W_gate_local.shape[0]
        self.N = W_g.shape[1]
        assert self.N == self.G * self.Ne, "N must equal world * local experts"
        self.cf, self.y_dtype = capacity_factor, y_dtype
        self.Ws = None if Ws_gate is None else (Ws_gate, Ws_up, Ws_down)
        self.exchange = exchange if exchange is not None else TorchDistExchange()
        self.status = torch.zeros(1, dtype=torch.int32, device=W_g.device)

    # step 1: routing and dispatch over all N experts
    def dispatch(self, x) -> EPState:
        T = x.shape[0]
        cap = B.moe_capacity(self.cf, T, self.k, self.N)
        idx, w = B.moe_router_topk(x, self.W_g, self.k, bias=self.bias,
                                   device_status=self.status)
        perm = B.moe_permute(idx, self.N, x=x, topk_w=w, capacity=cap,
                             device_status=self.status)
        counts, send_rows = plan_from_offsets(perm["offsets"].cpu(), self.G, self.Ne)
        st = EPState(T=T, A=sum(send_rows), perm=perm, counts=counts, send_rows=send_rows)
        if self.Ws is not None:   # the shared expert on this rank's own tokens, weight 1
            off = torch.tensor([0, T], dtype=torch.int32, device=x.device)
            st.shared_y = B.moe_expert_ffn(x, off, self.Ws[0][None], self.Ws[1][None],
                                           self.Ws[2][None], device_status=self.status)
        return st

    # after the counts exchange: the received counts (device) and row splits
    def post_counts(self, st: EPState, recv_counts):
        st.recv_counts = recv_counts.to(self.W_g.device, torch.int32).contiguous()
        st.recv_rows = recv_rows_from_counts(recv_counts.cpu(), self.G, self.Ne)

    # step 4: the local experts on the received rows; returns the output rows in
    # received order, for the return exchange
    def experts(self, st: EPState, x_recv, rs_recv):
        R = sum(st.recv_rows)
        g = B.moe_ep_regroup(st.recv_counts, self.Ne, x_recv[:R], rs_recv[:R],
                             device_status=self.status)
        return B.moe_expert_ffn(g["x_local"], g["offsets_local"], self.Wg, self.Wu, self.Wd,
                                row_scale=g["row_scale_local"], device_status=self.status,
                                A_max=R, out_row=g["src"], rows_out=R)

    # step 6: the output rows, back in this rank's x_perm order, combined
    def combine(self, st: EPState, y_perm):
        return B.moe_combine(y_perm, st.perm["inv_pos"], shared_y=st.shared_y,
                             y_dtype=self.y_dtype)

    def forward(self, x):
        ex = self.exchange
        st = self.dispatch(x)
        self.post_counts(st, exchange_counts(ex, st.counts.to(x.device), self.G, self.Ne))
        x_recv = exchange_rows(ex, st.perm["x_perm"], st.send_rows, st.recv_rows)
        rs_recv = exchange_rows(ex, st.perm["row_scale"], st.send_rows, st.recv_rows)
        y_back = self.experts(st, x_recv, rs_recv)
        y_perm = exchange_rows(ex, y_back, st.recv_rows, st.send_rows)
        return self.combine(st, y_perm)

    __call__ = forward


def _split(t, sizes):
    out, p = [], 0
    for n in sizes:
        out.append(t[p:p + n])
        p += n
    return out


def _loopback(parts):
    """out[r] = the parts every source s sends to r, in source order."""
    G = len(parts)
    return [torch.cat([parts[s][r] for s in range(G)]) for r in range(G)]


def run_ranks_in_one_process(layers, xs):
    """Drives G ranks' layers (rank r's ExpertParallelMoE and its tokens xs[r])
    in one process on one device, doing each exchange as plain device copies:
    the data movement an all-to-all performs, with no kernel waiting on another
    rank's.  For checking the expert-parallel path on a single GPU.  Returns
    each rank's y."""
    G = len(layers)
    Ne = layers[0].Ne
    sts = [layers[r].dispatch(xs[r]) for r in range(G)]
    recv = _loopback([list(torch.split(st.counts.to(xs[0].device), Ne)) for st in sts])
    for r in range(G):
        layers[r].post_counts(sts[r], recv[r])
    x_recv = _loopback([_split(st.perm["x_perm"], st.send_rows) for st in sts])
    s_recv = _loopback([_split(st.perm["row_scale"], st.send_rows) for st in sts])
    y_back = [layers[r].experts(sts[r], x_recv[r], s_recv[r]) for r in range(G)]
    y_perm = _loopback([_split(y_back[r], sts[r].recv_rows) for r in range(G)])
    return [layers[r].combine(sts[r], y_perm[r]) for r in range(G)]
