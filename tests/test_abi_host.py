"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/moe.h declares, and rejects bad arguments on the
host with the documented status codes before touching any device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT
from sparse_mixture_experts_63_b300 import binding as B
from sparse_mixture_experts_63_b300 import build as build_mod
import oracle


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_what_binding_lists():
    assert header_functions() == sorted(B.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_version(lib):
    assert "sm_103a" in B.moe_version()


def test_capacity_matches_oracle(lib):
    for cf, T, k, N in [(1.25, 4096, 2, 128), (1.0, 10, 1, 3), (0.0, 5, 2, 4),
                        (-1.0, 5, 2, 4), (1.1, 1000, 2, 7), (2.0, 1, 1, 1)]:
        assert B.moe_capacity(cf, T, k, N) == oracle.capacity(cf, T, k, N)


def _args(**kw):
    a = B.moe_forward_args()
    a.T, a.d, a.f, a.N, a.k, a.dtype = 16, 64, 128, 8, 2, B.MOE_BF16
    for n in ("x", "W_g", "W_gate", "W_up", "W_down", "y"):
        setattr(a, n, 4096)          # a fake, aligned address: never dereferenced
    a.y_dtype = B.MOE_F32
    for key, v in kw.items():
        setattr(a, key, v)
    return a


@pytest.mark.parametrize("bad", [dict(k=0), dict(k=9), dict(T=0), dict(d=60), dict(f=100),
                                 dict(N=0), dict(x=None), dict(W_down=None), dict(y=None),
                                 dict(x=4100), dict(dtype=7), dict(fs=16)])
def test_forward_rejects_bad_arguments(lib, bad):
    a = _args(**bad)
    assert lib.moe_forward_workspace_size(ctypes.byref(a)) == 0
    rc = lib.moe_forward(ctypes.byref(a), ctypes.c_void_p(4096), 1 << 40, None)
    assert rc == 1, lib.moe_last_error()


def test_forward_unsupported_sizes(lib):
    a = _args(N=300, k=2)
    assert lib.moe_forward(ctypes.byref(a), ctypes.c_void_p(4096), 1 << 40, None) == 2


def test_forward_workspace_too_small(lib):
    a = _args()
    need = lib.moe_forward_workspace_size(ctypes.byref(a))
    assert need > 0
    assert lib.moe_forward(ctypes.byref(a), ctypes.c_void_p(4096), need - 1, None) == 3
    assert lib.moe_forward(ctypes.byref(a), None, need, None) == 3


def test_workspace_size_grows_with_shared_expert(lib):
    a = _args()
    b = _args(fs=64, Ws_gate=4096, Ws_up=4096, Ws_down=4096)
    assert lib.moe_forward_workspace_size(ctypes.byref(b)) > lib.moe_forward_workspace_size(
        ctypes.byref(a))


def test_stage_entry_points_reject_bad_arguments(lib):
    # router: k > N, misaligned x
    assert lib.moe_router_topk(4096, 4096, None, 1, 4, 64, 8, 9, None, 4096, 4096, None,
                               None) == 1
    assert lib.moe_router_topk(4098, 4096, None, 1, 4, 64, 8, 2, None, 4096, 4096, None,
                               None) == 1
    assert lib.moe_router_topk(4096, 4096, None, 1, 4, 64, 300, 2, None, 4096, 4096, None,
                               None) == 2
    # permute: negative capacity, workspace too small
    assert lib.moe_permute(4096, None, None, 1, 4, 64, 8, 2, -1, 4096, 4096, 4096, None, 4096,
                           None, None, None, 4096, 1 << 20, None) == 1
    assert lib.moe_permute(4096, None, None, 1, 4, 64, 8, 2, 0, 4096, 4096, 4096, None, 4096,
                           None, None, None, None, 0, None) == 3
    # expert ffn: f not a multiple of 8
    assert lib.moe_expert_ffn(4096, 4096, None, 8, 64, 100, 8, 1, 4096, 4096, 4096, 4096, None,
                              4096, 1 << 30, None) == 1
    # FP8: d not a multiple of 16, missing scales, workspace too small
    assert lib.moe_quantize_weights_e4m3(4096, 2, 40, 64, 4096, 4096, None) == 1
    assert lib.moe_quantize_rows_e4m3(4096, 4, 40, 4096, 4096, None) == 1
    assert lib.moe_quantize_rows_e4m3(4096, 4, 64, 4096, None, None) == 1
    p = 4096
    assert lib.moe_expert_ffn_fp8(p, p, p, p, None, 8, 64, 64, 2, p, None, p, p, p, None, None,
                                  p, None, p, 1 << 30, None) == 1
    assert lib.moe_expert_ffn_fp8(p, p, p, p, None, 8, 64, 64, 2, p, p, p, p, p, None, None, p,
                                  None, p, 16, None) == 3
    # E4M3 down projection: scales missing; f not a multiple of 16
    assert lib.moe_expert_ffn_fp8(p, p, p, p, None, 8, 64, 64, 2, p, p, p, p, None, p, None, p,
                                  None, p, 1 << 30, None) == 1
    assert lib.moe_expert_ffn_fp8(p, p, p, p, None, 8, 64, 72, 2, p, p, p, p, None, p, p, p,
                                  None, p, 1 << 30, None) == 1
    assert (lib.moe_expert_ffn_fp8_workspace_size(100, 64, 64, 4, 1) >
            lib.moe_expert_ffn_fp8_workspace_size(100, 64, 64, 4, 0))
    # combine: d not a multiple of 8
    assert lib.moe_combine(4096, 1, 4096, 4, 2, 60, None, 4096, 0, None) == 1
    assert "d=60" in B.lib().moe_last_error().decode()


def test_routing_stats_rejects_bad_arguments(lib):
    # N above 1024, missing counts or stats, workspace too small for the logits pass
    assert lib.moe_routing_stats(None, 4096, 16, 2048, 4096, None, None, None, 0, None) == 1
    assert lib.moe_routing_stats(None, None, 16, 8, 4096, None, None, None, 0, None) == 1
    assert lib.moe_routing_stats(None, 4096, 16, 8, None, None, None, None, 0, None) == 1
    need = lib.moe_routing_stats_workspace_size(1000, 64)
    assert need >= 4 * 64 * 4            # ceil(1000 / 256) chunks x 64 experts, fp32
    assert lib.moe_routing_stats(4096, 4096, 1000, 64, 4096, None, None, None, need - 1,
                                 None) == 3


def test_permute_reroute_rejects_bad_arguments(lib):
    p = 4096
    # capacity 0 (re-routing needs one), k + R > N, workspace too small
    assert lib.moe_permute_reroute(p, p, None, 1, 16, 64, 8, 2, 1, 0, p, p, None, p, p, p, p, p,
                                   None, None, None, None, p, 1 << 20, None) == 1
    assert lib.moe_permute_reroute(p, p, None, 1, 16, 64, 8, 2, 7, 5, p, p, None, p, p, p, p, p,
                                   None, None, None, None, p, 1 << 20, None) == 1
    need = lib.moe_permute_reroute_workspace_size(16, 8, 2, 2)
    assert need > 0
    assert lib.moe_permute_reroute(p, p, None, 1, 16, 64, 8, 2, 2, 5, p, p, None, p, p, p, p, p,
                                   None, None, None, None, p, need - 1, None) == 3


def test_forward_reroute_needs_capacity(lib):
    a = B.moe_forward_args()
    a.T, a.d, a.f, a.N, a.k, a.dtype, a.y_dtype = 16, 64, 64, 8, 2, 1, 0
    a.x = a.W_g = a.W_gate = a.W_up = a.W_down = a.y = 4096
    a.reroute_rounds = 2
    assert lib.moe_forward_workspace_size(ctypes.byref(a)) == 0      # no capacity factor
    a.capacity_factor = 1.0
    assert lib.moe_forward_workspace_size(ctypes.byref(a)) > 0
    a.reroute_rounds = 7                                             # k + R > N
    assert lib.moe_forward_workspace_size(ctypes.byref(a)) == 0


def test_overlapped_host_io_rejects_bad_arguments(lib):
    a = _args()
    h = ctypes.c_void_p(4096)
    # routing outputs set (the call returns y only); a stream used twice; no host buffer
    b = _args(topk_idx=4096)
    assert lib.moe_forward_host_io_overlapped(ctypes.byref(b), h, h, h, 1 << 40, 2, 8, 16,
                                              24) == 1
    assert lib.moe_forward_host_io_overlapped(ctypes.byref(a), h, h, h, 1 << 40, 2, 8, 8,
                                              24) == 1
    assert lib.moe_forward_host_io_overlapped(ctypes.byref(a), None, h, h, 1 << 40, 2, 8, 16,
                                              24) == 1
    need = lib.moe_forward_workspace_size(ctypes.byref(a))
    assert lib.moe_forward_host_io_overlapped(ctypes.byref(a), h, h, h, need - 1, 2, 8, 16,
                                              24) == 3


def test_overlap_chunks_rule(lib):
    """Chunks keep each batch's tensor work at least four times its weight
    streaming, at most one per 2048 tokens: a prefill-shaped layer (16384
    tokens, 8 experts of 4096 x 14336: 1.15e13 flop against 2.8 GB of weights,
    3.7 times the four-fold bound) gets 3; a DeepSeek-shaped one (weights near
    the ridge) and a 32-token decode batch get 1."""
    pre = _args(T=16384, d=4096, f=14336, N=8, k=2)
    ds = _args(T=8192, d=7168, f=2048, N=256, k=8, fs=2048, Ws_gate=4096, Ws_up=4096,
               Ws_down=4096)
    dec = _args(T=32, d=4096, f=14336, N=8, k=2)
    assert lib.moe_forward_overlap_chunks(ctypes.byref(pre)) == 3
    assert lib.moe_forward_overlap_chunks(ctypes.byref(ds)) == 1
    assert lib.moe_forward_overlap_chunks(ctypes.byref(dec)) == 1


def test_forward_args_layout_matches_header(tmp_path):
    """The binding's ctypes mirror of moe_forward_args has the C struct's
    field offsets and size (a C program compiled against include/moe.h
    prints them)."""
    fields = [f[0] for f in B.moe_forward_args._fields_]
    prog = ["#include <stdio.h>", "#include <stddef.h>", '#include "moe.h"', "int main(void) {",
            '  printf("%zu\\n", sizeof(moe_forward_args));']
    prog += [f'  printf("%zu\\n", offsetof(moe_forward_args, {n}));' for n in fields]
    prog += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(prog) + "\n")
    exe = tmp_path / "layout"
    import subprocess
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)],
                   check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    assert got[0] == ctypes.sizeof(B.moe_forward_args)
    assert got[1:] == [getattr(B.moe_forward_args, n).offset for n in fields]


def test_ep_argument_errors(lib):
    """moe_ep_regroup / moe_ep_return reject bad sizes on the host, before any launch."""
    fake = ctypes.c_void_p(4096)
    # G * Ne beyond the supported 4096 blocks
    assert lib.moe_ep_regroup(fake, 64, 65, fake, None, 10, 64, B.MOE_BF16, fake, None, fake, fake,
                              None, None, None) == 2
    # rows that are not a multiple of 16 bytes (bf16, d = 4)
    assert lib.moe_ep_regroup(fake, 2, 2, fake, None, 10, 4, B.MOE_BF16, fake, None, fake, fake,
                              None, None, None) == 1
    # missing destination map
    assert lib.moe_ep_regroup(fake, 2, 2, fake, None, 10, 64, B.MOE_BF16, fake, None, fake, None,
                              None, None, None) == 1
    # a row scale in without one out
    assert lib.moe_ep_regroup(fake, 2, 2, fake, fake, 10, 64, B.MOE_BF16, fake, None, fake, fake,
                              None, None, None) == 1
    assert lib.moe_ep_return(fake, None, 10, 64, B.MOE_BF16, fake, None) == 1
    # the FFN with an output-row map: the map is required, rows_out >= 0
    ws = ctypes.c_void_p(4096)
    assert lib.moe_expert_ffn_to_rows(fake, fake, None, None, 10, 64, 64, 2, B.MOE_BF16, fake,
                                      fake, fake, fake, 10, None, ws, 1 << 30, None) == 1
    assert lib.moe_expert_ffn_to_rows(fake, fake, None, fake, 10, 64, 64, 2, B.MOE_BF16, fake,
                                      fake, fake, fake, -1, None, ws, 1 << 30, None) == 1
    assert lib.moe_ep_return(fake, fake, -1, 64, B.MOE_BF16, fake, None) == 1
