"""flint_moe_route_noalloc (routing in the library's fixed static scratch)
against flint_moe_route (caller workspace) on the GPU.

The file name sorts last so that the static-scratch entry point also runs
after every other GPU test in the same process; it passes alone as well.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import nvfp4_w4a16_mixture_gb300 as fm
from nvfp4_w4a16_mixture_gb300 import synth

pytestmark = pytest.mark.gpu


def _route_ws(x, w, k):
    M, H = x.shape
    ws = fm.alloc_workspace(M, H, w.shape[0], k, 128, 0)
    ids = torch.empty(M, k, dtype=torch.int32, device="cuda")
    tw = torch.empty(M, k, dtype=torch.float32, device="cuda")
    fm.flint_moe_route(x, w, k, ids, tw, ws)
    return ids, tw


def _route_static(x, w, k):
    M = x.shape[0]
    ids = torch.full((M, k), -7, dtype=torch.int32, device="cuda")
    tw = torch.full((M, k), float("nan"), dtype=torch.float32, device="cuda")
    fm.flint_moe_route_noalloc(x, w, k, ids, tw)
    return ids, tw


@pytest.mark.parametrize("M,H,E,k", [(1, 2048, 128, 8), (37, 2048, 128, 8), (300, 384, 96, 6)])
def test_two_calls_in_a_row_match_workspace_entry_point(M, H, E, k):
    gen = torch.Generator(device="cuda").manual_seed(M + E)
    outs = []
    for call in range(2):
        x = synth.make_x(M, H, gen, "cuda")
        w = (torch.randn(E, H, generator=gen, device="cuda") * H ** -0.5).to(torch.bfloat16)
        ref = _route_ws(x, w, k)
        got = _route_static(x, w, k)
        torch.cuda.synchronize()
        assert torch.equal(got[0], ref[0]), f"ids differ on call {call}"
        # same kernel, same fixed summation order: the weights agree exactly,
        # well inside the block's BF16 tolerance
        assert torch.equal(got[1], ref[1]), f"tw differ on call {call}"
        outs.append(got[0].cpu().numpy())
    if M > 1:
        assert not np.array_equal(outs[0], outs[1])  # the second call really recomputed


def test_largest_shape_that_fits_and_oversize_rejected():
    H, E, k = 256, 128, 8
    cap = fm.flint_moe_route_noalloc_capacity()
    M = 6543
    assert fm.flint_moe_route_noalloc_bytes(M, H, E, k) <= cap
    gen = torch.Generator(device="cuda").manual_seed(5)
    x = synth.make_x(M, H, gen, "cuda")
    w = (torch.randn(E, H, generator=gen, device="cuda") * H ** -0.5).to(torch.bfloat16)
    ref = _route_ws(x, w, k)
    got = _route_static(x, w, k)
    torch.cuda.synchronize()
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
    x2 = synth.make_x(M + 1, H, gen, "cuda")
    ids = torch.empty(M + 1, k, dtype=torch.int32, device="cuda")
    tw = torch.empty(M + 1, k, dtype=torch.float32, device="cuda")
    with pytest.raises(fm.FlintMoEError) as ei:
        fm.flint_moe_route_noalloc(x2, w, k, ids, tw)
    assert ei.value.code == fm.FLINT_ERR_SCRATCH
