"""Expert parallelism on one GPU: the regroup and return kernels against the
layout they document, and a whole expert-parallel layer with G ranks emulated
in one process.

The emulation runs each rank's steps (dispatch, experts, combine) through the
C ABI and performs the exchanges between them as plain device copies -- the
data movement an all-to-all does; no kernel waits on another rank's.  Each
rank's output is compared with the oracle's layer on that rank's tokens (all
N experts), within the layer tolerance, and with the single-GPU layer on the
same tokens, bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
from sparse_mixture_experts_63_b300 import binding as B
from sparse_mixture_experts_63_b300 import expert_parallel as EP
from sparse_mixture_experts_63_b300.configs import MoEConfig
from sparse_mixture_experts_63_b300.inputs import make_inputs, make_x

pytestmark = pytest.mark.gpu


def _regroup_reference(recv, rs, counts, G, Ne):
    starts, acc = [], 0
    for b in range(G * Ne):
        starts.append(acc)
        acc += int(counts[b])
    order, offsets = [], [0]
    for e in range(Ne):
        for s in range(G):
            b = s * Ne + e
            order.extend(range(starts[b], starts[b] + int(counts[b])))
        offsets.append(len(order))
    order = torch.tensor(order, dtype=torch.long)
    dest = torch.empty(acc, dtype=torch.long)
    dest[order] = torch.arange(acc)
    return recv[order], (rs[order] if rs is not None else None), offsets, dest


@pytest.mark.parametrize("G,Ne,dtype,seed", [(2, 4, torch.bfloat16, 1), (4, 3, torch.float32, 2),
                                             (1, 8, torch.bfloat16, 3), (8, 32, torch.bfloat16, 4),
                                             (3, 1, torch.float32, 5)])
def test_regroup_and_return_bit_exact(G, Ne, dtype, seed):
    rng = np.random.default_rng(seed)
    counts = rng.integers(0, 9, size=G * Ne)
    counts[rng.integers(0, G * Ne, size=max(1, G * Ne // 4))] = 0     # empty blocks
    R, d = int(counts.sum()), 64
    x = torch.randn((max(R, 1), d), generator=torch.Generator().manual_seed(seed)).to(dtype)[:R]
    rs = torch.rand(R, generator=torch.Generator().manual_seed(seed + 1))
    cd = torch.from_numpy(counts.astype(np.int32)).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = B.moe_ep_regroup(cd, Ne, x.cuda(), rs.cuda(), device_status=st)
    y = B.moe_ep_return(out["x_local"], out["dest"], R)
    torch.cuda.synchronize()
    xr, rsr, off, dest = _regroup_reference(x, rs, counts, G, Ne)
    assert int(st.item()) == 0
    assert out["offsets_local"].cpu().tolist() == off
    assert torch.equal(out["dest"][:R].cpu().long(), dest)
    src = out["src"][:R].cpu().long()                  # the inverse map: src[dest[i]] = i
    assert torch.equal(src[dest], torch.arange(R))
    assert torch.equal(out["x_local"][:R].cpu(), xr)
    assert torch.equal(out["row_scale_local"][:R].cpu(), rsr)
    assert torch.equal(y[:R].cpu(), x)                   # the return undoes the regroup


@pytest.mark.parametrize("counts,dtype", [
    pytest.param([0, 1, 160, 161, 300, 7], torch.bfloat16, id="bf16-256-row-tiles"),
    pytest.param([257, 290, 203, 313], torch.bfloat16, id="bf16-wide-tiles"),
    pytest.param([5, 0, 40, 13], torch.float32, id="fp32")])
def test_expert_ffn_to_rows_equals_ffn_then_scatter(counts, dtype):
    """moe_expert_ffn_to_rows = moe_expert_ffn followed by y[out_row[p]] = y_perm[p],
    bit for bit (bf16 on the tensor cores, one-sub-tile and wide tiles; fp32 on the
    CUDA cores); rows no p maps to keep their contents; an out-of-range row stores
    nothing and sets MOE_DEV_BAD_ROW."""
    g = torch.Generator().manual_seed(sum(counts) + len(counts))
    N, d, f = len(counts), 128, 256
    A = sum(counts)
    x = torch.randn((A, d), generator=g).to(dtype).cuda()
    Wg = (torch.randn((N, d, f), generator=g) / d ** 0.5).to(dtype).cuda()
    Wu = (torch.randn((N, d, f), generator=g) / d ** 0.5).to(dtype).cuda()
    Wd = (torch.randn((N, f, d), generator=g) / f ** 0.5).to(dtype).cuda()
    rs = torch.rand(A, generator=g).cuda()
    off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32).cuda()
    rows_out = A + 5
    perm = torch.randperm(rows_out, generator=g)[:A]
    out_row = perm.to(torch.int32).cuda()
    y_ref = B.moe_expert_ffn(x, off, Wg, Wu, Wd, row_scale=rs)
    y = torch.full((rows_out, d), 7.0, dtype=dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_expert_ffn(x, off, Wg, Wu, Wd, row_scale=rs, out_row=out_row, rows_out=rows_out,
                     y_perm=y, device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(y[perm.cuda()], y_ref[:A])
    untouched = torch.ones(rows_out, dtype=torch.bool)
    untouched[perm] = False
    assert bool((y[untouched.cuda()] == 7.0).all())
    bad = out_row.clone()
    bad[A // 2] = rows_out                                    # outside the output
    y2 = torch.full((rows_out, d), 7.0, dtype=dtype, device="cuda")
    B.moe_expert_ffn(x, off, Wg, Wu, Wd, row_scale=rs, out_row=bad, rows_out=rows_out,
                     y_perm=y2, device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & B.MOE_DEV_BAD_ROW
    keep = torch.arange(A) != A // 2
    assert torch.equal(y2[perm[keep].cuda()], y_ref[:A][keep.cuda()])


def test_regroup_flags_counts_that_do_not_add_up():
    cd = torch.tensor([3, 2], dtype=torch.int32, device="cuda")
    x = torch.randn((4, 64), device="cuda").to(torch.bfloat16)    # 4 rows, counts say 5
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_ep_regroup(cd, 1, x, None, device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & B.MOE_DEV_BAD_COUNTS


def _emulated_ep(cfg, G, seeds):
    inp = make_inputs(cfg, device=torch.device("cuda"))
    Ne = cfg.N // G
    layers = [EP.ExpertParallelMoE(inp.W_g, inp.W_gate[r * Ne:(r + 1) * Ne],
                                   inp.W_up[r * Ne:(r + 1) * Ne], inp.W_down[r * Ne:(r + 1) * Ne],
                                   cfg.k, r, G, bias=inp.bias, capacity_factor=cfg.cf,
                                   Ws_gate=inp.Ws_gate, Ws_up=inp.Ws_up, Ws_down=inp.Ws_down)
              for r in range(G)]
    xs = [make_x(cfg, device=torch.device("cuda"), seed=s) for s in seeds]
    ys = EP.run_ranks_in_one_process(layers, xs)
    torch.cuda.synchronize()
    for L in layers:
        assert int(L.status.item()) == 0
    return inp, xs, ys


@pytest.mark.parametrize("G", [2, 4])
@pytest.mark.parametrize("cfg", [
    MoEConfig("ep_fine", T=300, d=256, f=256, N=16, k=4, seed=81),
    MoEConfig("ep_capacity", T=512, d=256, f=192, N=32, k=2, cf=1.25, bias_std=1.0, seed=82),
    MoEConfig("ep_f32", T=100, d=64, f=96, N=8, k=2, dtype="f32", seed=83),
    MoEConfig("ep_shared", T=200, d=256, f=256, N=32, k=8, fs=256, seed=84),
], ids=lambda c: c.name)
def test_expert_parallel_layer_emulated_ranks(cfg, G):
    seeds = [cfg.seed * 10 + r for r in range(G)]
    inp, xs, ys = _emulated_ep(cfg, G, seeds)
    single = B.MoELayer(inp.W_g, inp.W_gate, inp.W_up, inp.W_down, cfg.k, bias=inp.bias,
                        capacity_factor=cfg.cf, Ws_gate=inp.Ws_gate, Ws_up=inp.Ws_up,
                        Ws_down=inp.Ws_down)
    shared = None if not cfg.fs else (inp.Ws_gate.cpu(), inp.Ws_up.cpu(), inp.Ws_down.cpu())
    for r in range(G):
        x = xs[r]
        # the single-GPU layer on the same tokens: same kernels, same per-row math
        y1 = single(x)
        torch.cuda.synchronize()
        d_single = float((ys[r] - y1).abs().max())
        # the oracle's layer on this rank's tokens, with all N experts
        xc = x.cpu()
        lo = oracle.router_logits(xc, inp.W_g.cpu(), None if inp.bias is None else inp.bias.cpu())
        idx_o, w_o = oracle.topk_softmax(lo, cfg.k)
        C = oracle.capacity(cfg.cf, cfg.T, cfg.k, cfg.N)
        g_o = oracle.group(idx_o, cfg.N, C)
        near = oracle.near_tie_tokens(lo, cfg.k, parity.TIE_REL)
        keep = ~near if C == 0 else ~(near | np.isin(idx_o, idx_o[near]).any(1))
        sel = np.nonzero(keep)[0]
        y_o = oracle.forward_rows(xc[torch.as_tensor(sel)], idx_o[sel], w_o[sel],
                                  g_o["inv_pos"][sel], parity.fetcher(inp), shared=shared)
        max_abs, fro = parity.assert_y_close(ys[r][torch.as_tensor(sel, device="cuda")].float()
                                             .cpu().numpy(), y_o, cfg.dtype)
        # each row meets the same MMAs in the same K order on either path, so the
        # expert-parallel output is the single-GPU layer's bit for bit
        assert torch.equal(ys[r], y1), f"rank {r}: {d_single} from the single-GPU layer"
        print(cfg.name, G, r, "oracle", max_abs, fro, "single-GPU max diff", d_single,
              "rows", len(sel))


def test_regroup_with_no_rows():
    cd = torch.zeros(6, dtype=torch.int32, device="cuda")
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    out = B.moe_ep_regroup(cd, 3, x, None)
    y = B.moe_ep_return(out["x_local"], out["dest"], 0)
    torch.cuda.synchronize()
    assert out["offsets_local"].cpu().tolist() == [0, 0, 0, 0]
    assert y.shape[1] == 64
