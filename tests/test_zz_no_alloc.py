"""moe_permute_noalloc: the dispatch step for callers that cannot allocate
device memory.  Its output must match moe_permute (which takes a caller
workspace) exactly -- every output is integer, index or a copied value -- on
two calls in a row, since the calls share the library's fixed scratch array.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from sparse_mixture_experts_63_b300 import binding as B
from sparse_mixture_experts_63_b300 import build as build_mod


def _case(T, N, k, seed, skew=1.0):
    rng = np.random.default_rng(seed)
    p = np.exp(skew * rng.normal(size=N))
    p /= p.sum()
    idx = np.stack([rng.choice(N, size=k, replace=False, p=p) for _ in range(T)])
    return torch.from_numpy(idx.astype(np.int32))


@pytest.mark.gpu
@pytest.mark.parametrize("T,N,k,cap", [(4096, 128, 2, 80), (8192, 256, 8, 0), (777, 32, 3, 50)])
def test_noalloc_matches_workspace_version_twice(T, N, k, cap):
    idx = _case(T, N, k, T + N).cuda()
    x = torch.randn((T, 64), device="cuda").to(torch.bfloat16)
    w = torch.rand((T, k), device="cuda")
    ref = B.moe_permute(idx, N, x=x, topk_w=w, capacity=cap)
    for _ in range(2):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        got = B.moe_permute_noalloc(idx, N, x=x, topk_w=w, capacity=cap, device_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        A = int(ref["offsets"][-1].item())
        for key in ("counts", "offsets", "inv_pos", "dropped"):
            assert torch.equal(got[key], ref[key]), key
        assert torch.equal(got["perm_token"][:A], ref["perm_token"][:A])
        assert torch.equal(got["row_scale"][:A], ref["row_scale"][:A])
        assert torch.equal(got["x_perm"][:A], ref["x_perm"][:A])


@pytest.mark.gpu
def test_noalloc_different_sizes_in_a_row():
    """A smaller call after a larger one reads none of the larger call's leftovers."""
    big = _case(8192, 256, 8, 1).cuda()
    small = _case(300, 16, 2, 2).cuda()
    B.moe_permute_noalloc(big, 256)
    got = B.moe_permute_noalloc(small, 16)
    ref = B.moe_permute(small, 16)
    torch.cuda.synchronize()
    for key in ("counts", "offsets", "inv_pos"):
        assert torch.equal(got[key], ref[key]), key


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """Sizes over the fixed scratch are refused on the host, before any launch."""
    build_mod.build()
    L = B.lib()
    T, N, k = 65536 + 256, 256, 8            # ceil(T/256) * N = 65792 > 65536
    fake = ctypes.c_void_p(4096)
    rc = L.moe_permute_noalloc(fake, None, None, 1, T, 64, N, k, 0, fake, fake, fake, None, fake,
                               None, None, None, None)
    assert rc == 2
    assert "65536" in L.moe_last_error().decode()
    # a token count near INT_MAX: the entry count is formed without overflow
    rc = L.moe_permute_noalloc(fake, None, None, 1, 2 ** 31 - 100, 64, 1, 1, 0, fake, fake, fake,
                               None, fake, None, None, None, None)
    assert rc == 2
    assert "65536" in L.moe_last_error().decode()
