"""Expert parallelism on CPU: the split-size bookkeeping, and the three
exchanges of a forward run by two (and three) gloo ranks.

Rows are tagged with (source rank, global expert, index within the expert),
so every received block can be checked against what the layout rule says it
must hold; the round trip (regroup by a plain reference of the documented
layout, identity expert, return exchange) must give every rank its own rows
back in its own order.  The device steps (router, dispatch, regroup, experts,
combine) are libmoe kernels, covered by tests/test_gpu_expert_parallel.py.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from conftest import ROOT  # noqa: F401  (puts the repository on sys.path)
from sparse_mixture_experts_63_b300 import expert_parallel as EP


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _counts(rank, G, Ne, seed):
    rng = np.random.default_rng(seed * 100 + rank)
    c = rng.integers(0, 7, size=G * Ne)
    c[rng.integers(0, G * Ne)] = 0          # at least one empty expert
    return c


def _x_perm(rank, counts):
    """Rows of width 4: (source, expert, index in expert, marker)."""
    rows = []
    for e, n in enumerate(counts):
        for j in range(n):
            rows.append([rank, e, j, 7.0])
    return torch.tensor(rows, dtype=torch.float32).reshape(-1, 4)


def test_plan_from_offsets_closed_form():
    G, Ne = 3, 2
    counts = [2, 0, 5, 1, 0, 3]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    c, send = EP.plan_from_offsets(torch.tensor(offsets), G, Ne)
    assert c.tolist() == counts
    assert send == [2, 6, 3]
    assert EP.recv_rows_from_counts(torch.tensor([1, 2, 0, 0, 4, 4]), G, Ne) == [3, 0, 8]


def _regroup_reference(recv, recv_counts, G, Ne):
    """Block (s, e) moved behind the blocks of sources < s inside expert e's range."""
    c = recv_counts.view(G, Ne)
    starts = torch.zeros(G * Ne, dtype=torch.long)
    acc = 0
    for b in range(G * Ne):
        starts[b] = acc
        acc += int(recv_counts[b])
    out, dest = [], torch.empty(acc, dtype=torch.long)
    pos = 0
    for e in range(Ne):
        for s in range(G):
            b = s * Ne + e
            n = int(c[s, e])
            out.append(recv[starts[b]:starts[b] + n])
            dest[starts[b]:starts[b] + n] = torch.arange(pos, pos + n)
            pos += n
    return torch.cat(out) if out else recv[:0], dest


def _rank_main(rank, G, Ne, port, seed, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=G)
    ex = EP.TorchDistExchange()
    try:
        counts = _counts(rank, G, Ne, seed)
        x_perm = _x_perm(rank, counts)
        offsets = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32)
        c, send_rows = EP.plan_from_offsets(offsets, G, Ne)
        recv_counts = EP.exchange_counts(ex, c, G, Ne)
        # what every source sent for this rank's experts
        expect = np.stack([_counts(s, G, Ne, seed)[rank * Ne:(rank + 1) * Ne] for s in range(G)])
        assert recv_counts.view(G, Ne).tolist() == expect.tolist()
        recv_rows = EP.recv_rows_from_counts(recv_counts, G, Ne)
        x_recv = EP.exchange_rows(ex, x_perm, send_rows, recv_rows)[:sum(recv_rows)]
        scale = x_perm[:, 2] + 0.5 * rank        # a per-row value travelling with the row
        s_recv = EP.exchange_rows(ex, scale, send_rows, recv_rows)[:sum(recv_rows)]
        # received blocks: source-major, then local expert, each in its source's order
        p = 0
        for s in range(G):
            for e in range(Ne):
                n = int(expect[s, e])
                blk = x_recv[p:p + n]
                assert (blk[:, 0] == s).all() and (blk[:, 1] == rank * Ne + e).all()
                assert blk[:, 2].tolist() == list(range(n))
                assert torch.equal(s_recv[p:p + n], blk[:, 2] + 0.5 * s)
                p += n
        # regroup, identity expert, return: each rank gets its own rows back
        x_loc, dest = _regroup_reference(x_recv, recv_counts, G, Ne)
        assert (x_loc[1:, 1] >= x_loc[:-1, 1]).all()          # grouped by expert
        y_back = x_loc[dest]
        y_perm = EP.exchange_rows(ex, y_back, recv_rows, send_rows)[:sum(send_rows)]
        assert torch.equal(y_perm, x_perm)
        q.put((rank, "ok"))
    except Exception as exc:   # noqa: BLE001 -- reported to the parent
        q.put((rank, repr(exc)))
    finally:
        dist.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="the gloo leg is the CPU path")
@pytest.mark.parametrize("G,Ne,seed", [(2, 3, 1), (3, 2, 2), (2, 1, 3)])
def test_exchange_round_trip_gloo(G, Ne, seed):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, G, Ne, port, seed, q)) for r in range(G)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(G))
    assert [r[1] for r in res] == ["ok"] * G, res
