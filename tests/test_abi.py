"""The C-ABI library builds, loads and exports every symbol include/*.h
declares; argument validation answers synchronously (no GPU work)."""
from __future__ import annotations

import ctypes
import glob
import os
import re

import pytest

import nvfp4_w4a16_mixture_gb300 as fm
from nvfp4_w4a16_mixture_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions() -> set[str]:
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(flint_\w+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_header_declares_binding_names():
    assert declared_functions() == set(fm.EXPORTED)


def test_library_exports_every_declared_symbol():
    lib = fm.load()
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_workspace_bytes_valid_and_invalid_shapes():
    ok = fm.flint_moe_workspace_bytes(1, 2048, 128, 8, 768, 768)
    assert ok > 0 and ok % 256 == 0
    big = fm.flint_moe_workspace_bytes(4096, 2048, 128, 8, 768, 768)
    assert big > ok
    assert fm.flint_moe_workspace_bytes(0, 2048, 128, 8, 768, 768) > 0  # empty batch
    for bad in [(-1, 2048, 128, 8, 768, 768), (1, 2000, 128, 8, 768, 768),
                (1, 2048, 257, 8, 768, 768), (1, 2048, 8, 9, 768, 768),
                (1, 2048, 128, 0, 768, 768), (1, 2048, 128, 33, 768, 768),
                (1, 2048, 128, 8, 700, 768), (1, 2048, 128, 8, 768, 100),
                (1, 2048, 128, 8, 768, -128)]:
        assert fm.flint_moe_workspace_bytes(*bad) == 0, bad
    assert fm.flint_moe_workspace_bytes(3, 256, 8, 2, 128, 0) > 0  # no shared expert


def test_strerror_covers_codes():
    for code in (fm.FLINT_OK, fm.FLINT_ERR_INVALID_ARG, fm.FLINT_ERR_UNSUPPORTED,
                 fm.FLINT_ERR_WORKSPACE, fm.FLINT_ERR_CUDA, fm.FLINT_ERR_TIMEOUT,
                 fm.FLINT_ERR_SCRATCH):
        assert fm.flint_moe_strerror(code) not in ("", "unknown error")
    assert fm.flint_moe_strerror(12345) == "unknown error"


def _call_forward(ptrs, shape, ws_bytes):
    lib = fm.load()
    s = _lib.flint_moe_shape(*shape)
    return lib.flint_moe_forward(*ptrs[:10], ctypes.byref(s), ptrs[10], None, None, ptrs[11],
                                 ws_bytes, None)


def test_fault_hook_accepts_only_known_sites():
    """The failure-path test hook is a host-side switch (no CUDA call)."""
    lib = fm.load()
    assert lib.flint_moe_debug_fault(fm.FLINT_FAULT_DOWN_HANDOVER) == fm.FLINT_OK
    assert lib.flint_moe_debug_fault(fm.FLINT_FAULT_NONE) == fm.FLINT_OK
    for bad in (1, -1, 9999):
        assert lib.flint_moe_debug_fault(bad) == fm.FLINT_ERR_INVALID_ARG


def test_empty_batch_is_a_no_op():
    """M = 0: the shape is checked and every entry point returns FLINT_OK
    before any CUDA call, even with NULL buffers and no workspace (so this
    runs without a GPU); a bad shape with M = 0 is still rejected."""
    lib = fm.load()
    s = _lib.flint_moe_shape(0, 2048, 128, 8, 768, 768)
    assert lib.flint_moe_forward(*([None] * 10), ctypes.byref(s), None, None, None, None, 0,
                                 None) == fm.FLINT_OK
    assert lib.flint_moe_route(None, None, ctypes.byref(s), None, None, None, 0, None) == fm.FLINT_OK
    assert lib.flint_moe_route_noalloc(None, None, ctypes.byref(s), None, None, None) == fm.FLINT_OK
    bad = _lib.flint_moe_shape(0, 2000, 128, 8, 768, 768)
    assert lib.flint_moe_forward(*([None] * 10), ctypes.byref(bad), None, None, None, None, 0,
                                 None) == fm.FLINT_ERR_INVALID_ARG


def test_validation_is_synchronous_and_touches_no_memory():
    """Null, misaligned and undersized arguments are rejected before any CUDA
    call (fake, never-dereferenced addresses)."""
    shape = (2, 256, 8, 2, 128, 128)
    need = fm.flint_moe_workspace_bytes(*shape)
    good = [0x10000 * (i + 1) for i in range(12)]
    assert _call_forward([None] + good[1:], shape, need) == fm.FLINT_ERR_INVALID_ARG
    mis = list(good)
    mis[2] += 8  # w13 not 16-byte aligned
    assert _call_forward(mis, shape, need) == fm.FLINT_ERR_INVALID_ARG
    assert _call_forward(good, shape, need - 1) == fm.FLINT_ERR_WORKSPACE
    ws_mis = list(good)
    ws_mis[11] += 16
    assert _call_forward(ws_mis, shape, need) == fm.FLINT_ERR_WORKSPACE
    assert _call_forward(good, (2, 256, 8, 3, 128, 100), need) == fm.FLINT_ERR_INVALID_ARG
    noshared = list(good)
    noshared[8] = None
    assert _call_forward(noshared, shape, need) == fm.FLINT_ERR_INVALID_ARG
    lib = fm.load()
    s = _lib.flint_moe_shape(*shape)
    assert lib.flint_moe_route(None, good[1], ctypes.byref(s), good[2], good[3], good[4], need,
                               None) == fm.FLINT_ERR_INVALID_ARG


def test_route_noalloc_size_limit_is_checked_before_any_cuda_call():
    """The static-scratch router rejects oversize and invalid shapes
    synchronously (fake, never-dereferenced addresses; no GPU here)."""
    cap = fm.flint_moe_route_noalloc_capacity()
    assert cap == 2 << 20
    need = fm.flint_moe_route_noalloc_bytes(6543, 2048, 128, 8)
    assert 0 < need <= cap
    assert fm.flint_moe_route_noalloc_bytes(6544, 2048, 128, 8) > cap
    assert fm.flint_moe_route_noalloc_bytes(1, 2048, 128, 33) == 0
    lib = fm.load()
    fake = [0x10000 * (i + 1) for i in range(4)]
    big = _lib.flint_moe_shape(6544, 2048, 128, 8, 128, 0)
    assert lib.flint_moe_route_noalloc(fake[0], fake[1], ctypes.byref(big), fake[2], fake[3],
                                       None) == fm.FLINT_ERR_SCRATCH
    ok = _lib.flint_moe_shape(4, 2048, 128, 8, 128, 0)
    assert lib.flint_moe_route_noalloc(None, fake[1], ctypes.byref(ok), fake[2], fake[3],
                                       None) == fm.FLINT_ERR_INVALID_ARG
    assert lib.flint_moe_route_noalloc(fake[0] + 8, fake[1], ctypes.byref(ok), fake[2], fake[3],
                                       None) == fm.FLINT_ERR_INVALID_ARG


def test_product_path_does_not_import_oracle():
    """The package never imports the oracle (the oracle is test-only)."""
    pkg = os.path.join(ROOT, "nvfp4_w4a16_mixture_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*.py"), recursive=True):
        src = open(path).read()
        assert not re.search(r"^\s*(import|from)\s+oracle", src, re.M), path
    for path in glob.glob(os.path.join(pkg, "csrc", "*")):
        assert "oracle" not in open(path).read().lower(), path


@pytest.mark.parametrize("shape", [(1, 2048, 128, 8, 768, 768), (64, 2048, 128, 8, 768, 768),
                                   (4096, 2048, 128, 8, 768, 768)])
def test_workspace_fits_expected_regions(shape):
    M, H, E, k, I, SI = shape
    need = fm.flint_moe_workspace_bytes(*shape)
    floor = 2 * M * k * (I + H) + 2 * M * (SI + H) + 2 * M * H  # act, y, sact, ys, xn
    if M > 64:
        floor += 2 * M * k * H  # token rows in sorted pair order (grouped path)
    assert floor <= need <= floor + 4 * 1024 * 1024 + 16 * M * k + 2 * M * E + 272 * E


def test_multiples_of_64_are_valid_but_unsupported():
    """H, I and SI are valid in multiples of 64; the kernels run 128-wide K
    slices, so an odd multiple of 64 is refused as unsupported (not as a bad
    argument), synchronously and before any CUDA call."""
    lib = fm.load()
    fake = [0x10000 * (i + 1) for i in range(12)]
    for shape in [(3, 192, 8, 2, 128, 128), (3, 256, 8, 2, 192, 128), (3, 256, 8, 2, 128, 64),
                  (3, 64, 8, 2, 64, 64)]:
        assert fm.flint_moe_workspace_bytes(*shape) == 0, shape
        assert _call_forward(fake, shape, 1 << 30) == fm.FLINT_ERR_UNSUPPORTED, shape
        s = _lib.flint_moe_shape(*shape)
        assert lib.flint_moe_route(fake[0], fake[1], ctypes.byref(s), fake[2], fake[3], fake[4],
                                   1 << 30, None) == fm.FLINT_ERR_UNSUPPORTED, shape
        assert lib.flint_moe_plan(ctypes.byref(s)) == fm.FLINT_ERR_UNSUPPORTED, shape
        with pytest.raises(fm.FlintMoEError) as ei:
            fm.flint_moe_plan(*shape)
        assert ei.value.code == fm.FLINT_ERR_UNSUPPORTED
        with pytest.raises(fm.FlintMoEError) as ei:
            fm.alloc_workspace(*shape, device="cpu")
        assert ei.value.code == fm.FLINT_ERR_UNSUPPORTED
    s = _lib.flint_moe_shape(3, 192, 8, 2, 128, 0)
    assert lib.flint_moe_route_noalloc(fake[0], fake[1], ctypes.byref(s), fake[2], fake[3],
                                       None) == fm.FLINT_ERR_UNSUPPORTED
    assert fm.flint_moe_route_noalloc_bytes(3, 192, 8, 2) == 0
    # not a multiple of 64: a malformed shape
    assert _call_forward(fake, (3, 160, 8, 2, 128, 128), 1 << 30) == fm.FLINT_ERR_INVALID_ARG


def test_plan_is_a_host_query():
    """flint_moe_plan answers an empty batch and a bad shape without a GPU."""
    assert fm.flint_moe_plan(0, 2048, 128, 8, 768, 768) == fm.FLINT_PATH_NONE
    with pytest.raises(fm.FlintMoEError) as ei:
        fm.flint_moe_plan(1, 2048, 128, 0, 768, 768)
    assert ei.value.code == fm.FLINT_ERR_INVALID_ARG


def test_forward_add_norm_validation_is_synchronous():
    """The add-RMSNorm entry point checks its extra arguments before any CUDA
    call (fake, never-dereferenced addresses)."""
    lib = fm.load()
    shape = (2, 256, 8, 2, 128, 128)
    need = fm.flint_moe_workspace_bytes(*shape)
    f = [0x10000 * (i + 1) for i in range(20)]
    s = _lib.flint_moe_shape(*shape)

    def call(attn=f[0], resid=f[1], lnw=f[2], eps=1e-6, res_out=f[14], xn_out=None, ws=f[17], shp=s):
        return lib.flint_moe_forward_add_norm(attn, resid, lnw, eps, *f[3:12], ctypes.byref(shp), f[13],
                                              res_out, xn_out, None, None, ws, need, None)

    assert call(res_out=None) == fm.FLINT_ERR_INVALID_ARG
    assert call(resid=None) == fm.FLINT_ERR_INVALID_ARG
    assert call(lnw=f[2] + 8) == fm.FLINT_ERR_INVALID_ARG
    assert call(eps=float("nan")) == fm.FLINT_ERR_INVALID_ARG
    assert call(eps=-1.0) == fm.FLINT_ERR_INVALID_ARG
    assert call(xn_out=f[15] + 4) == fm.FLINT_ERR_INVALID_ARG
    assert call(ws=None) == fm.FLINT_ERR_WORKSPACE
    odd = _lib.flint_moe_shape(2, 192, 8, 2, 128, 128)
    assert call(shp=odd) == fm.FLINT_ERR_UNSUPPORTED
    empty = _lib.flint_moe_shape(0, 256, 8, 2, 128, 128)
    assert lib.flint_moe_forward_add_norm(*([None] * 3), 1e-6, *([None] * 9), ctypes.byref(empty),
                                          *([None] * 6), 0, None) == fm.FLINT_OK


def test_forward_bf16_validation_is_synchronous():
    """The BF16-experts entry point refuses a shared intermediate size (the
    shared output comes in as a tensor), more than 64 tokens and odd
    multiples of 64, before any CUDA call."""
    lib = fm.load()
    f = [0x10000 * (i + 1) for i in range(12)]

    def call(shape, ws_bytes=1 << 30, x=f[0]):
        s = _lib.flint_moe_shape(*shape)
        return lib.flint_moe_forward_bf16(x, f[1], f[2], f[3], None, ctypes.byref(s), f[4], None, None,
                                          f[5], ws_bytes, None)

    assert call((2, 256, 8, 2, 128, 128)) == fm.FLINT_ERR_INVALID_ARG
    assert call((65, 256, 8, 2, 128, 0)) == fm.FLINT_ERR_UNSUPPORTED
    assert call((2, 192, 8, 2, 128, 0)) == fm.FLINT_ERR_UNSUPPORTED
    assert call((2, 256, 8, 2, 128, 0), x=None) == fm.FLINT_ERR_INVALID_ARG
    assert call((2, 256, 8, 2, 128, 0), ws_bytes=16) == fm.FLINT_ERR_WORKSPACE
    assert call((0, 256, 8, 2, 128, 0), x=None) == fm.FLINT_OK


def test_qkv_fused_validation_is_synchronous():
    """The fused qkv entry point sizes its workspace, refuses bad shapes,
    odd multiples of 64, missing pointers and a short workspace, and treats
    M = 0 as a no-op, before any CUDA call."""
    lib = fm.load()
    M, H, nq, nkv = 2, 256, 2, 1
    need = fm.flint_qkv_workspace_bytes(M, H, nq, nkv)
    N = (nq + 2 * nkv) * 128
    assert need >= 256 + M * H * 2 + M * N * 2
    assert fm.flint_qkv_workspace_bytes(M, 192, nq, nkv) == 0
    assert fm.flint_qkv_workspace_bytes(M, H, 0, nkv) == 0
    f = [0x10000 * (i + 1) for i in range(16)]

    def call(M=M, H=H, nq=nq, nkv=nkv, x=f[0], weight=f[2], ws=f[10], ws_bytes=need, slots=f[8], n_slots=M,
             k_cache=f[6], q_out=f[9], block_size=16):
        return lib.flint_qkv_fused(x, None, f[1], 1e-6, weight, None, None, f[3], f[4], 1e-6, None, 0, None,
                                   k_cache, f[7], 1024, 256, 128, block_size, 4, slots, n_slots, M, H, nq, nkv,
                                   q_out, None, ws, ws_bytes, None)

    assert call(H=250) == fm.FLINT_ERR_INVALID_ARG
    assert call(H=192) == fm.FLINT_ERR_UNSUPPORTED
    assert call(nq=0) == fm.FLINT_ERR_INVALID_ARG
    assert call(x=None) == fm.FLINT_ERR_INVALID_ARG
    assert call(weight=f[2] + 8) == fm.FLINT_ERR_INVALID_ARG  # not 16-byte aligned
    assert call(q_out=None) == fm.FLINT_ERR_INVALID_ARG
    assert call(k_cache=None) == fm.FLINT_ERR_INVALID_ARG
    assert call(block_size=0) == fm.FLINT_ERR_INVALID_ARG
    assert call(ws_bytes=need - 1) == fm.FLINT_ERR_WORKSPACE
    assert call(ws=None) == fm.FLINT_ERR_WORKSPACE
    assert call(M=0, x=None, ws=None) == fm.FLINT_OK
