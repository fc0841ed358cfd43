"""ctypes binding of libflint_moe (include/flint_moe.h), same names as the C ABI.

Argument marshalling only: every step of the MoE block runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors (torch provides device memory
and streams); their device pointers are passed straight through.  If the
library cannot be built or loaded this module raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import threading

import torch

from . import build as _build

FLINT_OK = 0
FLINT_ERR_INVALID_ARG = -1
FLINT_ERR_UNSUPPORTED = -2
FLINT_ERR_WORKSPACE = -3
FLINT_ERR_CUDA = -4
FLINT_ERR_TIMEOUT = -5
FLINT_ERR_SCRATCH = -6
FLINT_FAULT_NONE = 0
FLINT_FAULT_DOWN_HANDOVER = 17
FLINT_PATH_NONE = 0
FLINT_PATH_SINGLE_LAUNCH = 1
FLINT_PATH_DECODE = 2
FLINT_PATH_DECODE_FALLBACK = 3
FLINT_PATH_GROUPED = 4

# Every C symbol the header declares (checked by tests/test_abi.py).
EXPORTED = ("flint_moe_workspace_bytes", "flint_moe_route", "flint_moe_forward",
            "flint_moe_route_noalloc", "flint_moe_route_noalloc_bytes",
            "flint_moe_route_noalloc_capacity", "flint_moe_status", "flint_moe_strerror",
            "flint_moe_debug_fault", "flint_moe_plan", "flint_moe_prefer_path",
            "flint_moe_forward_add_norm", "flint_moe_record_spans", "flint_moe_forward_bf16",
            "flint_moe_forward_nvfp4_shared", "flint_qkv_workspace_bytes", "flint_qkv_fused")


class FlintMoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {flint_moe_strerror(code)} (code {code})")
        self.code = code


class flint_moe_shape(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int), ("H", ctypes.c_int), ("E", ctypes.c_int),
                ("top_k", ctypes.c_int), ("I", ctypes.c_int), ("SI", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Build (if stale) and load libflint_moe.so; raises on failure."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            lib = ctypes.CDLL(path)
            P, S = ctypes.c_void_p, ctypes.POINTER(flint_moe_shape)
            lib.flint_moe_workspace_bytes.restype = ctypes.c_size_t
            lib.flint_moe_workspace_bytes.argtypes = [S]
            lib.flint_moe_route.restype = ctypes.c_int
            lib.flint_moe_route.argtypes = [P, P, S, P, P, P, ctypes.c_size_t, P]
            lib.flint_moe_forward.restype = ctypes.c_int
            lib.flint_moe_forward.argtypes = [P] * 10 + [S, P, P, P, P, ctypes.c_size_t, P]
            lib.flint_moe_forward_add_norm.restype = ctypes.c_int
            lib.flint_moe_forward_add_norm.argtypes = ([P, P, P, ctypes.c_float] + [P] * 9 +
                                                       [S, P, P, P, P, P, P, ctypes.c_size_t, P])
            lib.flint_moe_route_noalloc.restype = ctypes.c_int
            lib.flint_moe_route_noalloc.argtypes = [P, P, S, P, P, P]
            lib.flint_moe_route_noalloc_bytes.restype = ctypes.c_size_t
            lib.flint_moe_route_noalloc_bytes.argtypes = [S]
            lib.flint_moe_route_noalloc_capacity.restype = ctypes.c_size_t
            lib.flint_moe_route_noalloc_capacity.argtypes = []
            lib.flint_moe_status.restype = ctypes.c_int
            lib.flint_moe_status.argtypes = [P, P]
            lib.flint_moe_strerror.restype = ctypes.c_char_p
            lib.flint_moe_strerror.argtypes = [ctypes.c_int]
            lib.flint_moe_debug_fault.restype = ctypes.c_int
            lib.flint_moe_debug_fault.argtypes = [ctypes.c_int]
            lib.flint_moe_plan.restype = ctypes.c_int
            lib.flint_moe_plan.argtypes = [S]
            lib.flint_moe_prefer_path.restype = ctypes.c_int
            lib.flint_moe_prefer_path.argtypes = [ctypes.c_int]
            lib.flint_moe_forward_nvfp4_shared.restype = ctypes.c_int
            lib.flint_moe_forward_nvfp4_shared.argtypes = [P] * 14 + [S, P, P, P, P, ctypes.c_size_t, P]
            lib.flint_moe_forward_bf16.restype = ctypes.c_int
            lib.flint_moe_forward_bf16.argtypes = [P] * 5 + [S, P, P, P, P, ctypes.c_size_t, P]
            lib.flint_moe_record_spans.restype = ctypes.c_int
            lib.flint_moe_record_spans.argtypes = [P]
            I, LL, F = ctypes.c_int, ctypes.c_longlong, ctypes.c_float
            lib.flint_qkv_workspace_bytes.restype = ctypes.c_size_t
            lib.flint_qkv_workspace_bytes.argtypes = [I, I, I, I]
            lib.flint_qkv_fused.restype = ctypes.c_int
            lib.flint_qkv_fused.argtypes = ([P, P, P, F, P, P, P, P, P, F, P, LL, P, P, P, LL, LL, LL, I, LL, P,
                                             I, I, I, I, I, P, P, P, ctypes.c_size_t, P])
            _lib = lib
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream or None
    return int(stream) or None


def _shape(M, H, E, top_k, I, SI) -> flint_moe_shape:
    return flint_moe_shape(int(M), int(H), int(E), int(top_k), int(I), int(SI))


def flint_moe_strerror(code: int) -> str:
    return load().flint_moe_strerror(int(code)).decode()


def flint_moe_workspace_bytes(M: int, H: int, E: int, top_k: int, I: int, SI: int) -> int:
    """Workspace bytes for the shape (0 if the shape is invalid or unsupported)."""
    s = _shape(M, H, E, top_k, I, SI)
    return int(load().flint_moe_workspace_bytes(ctypes.byref(s)))


def flint_moe_route(x, router_w, top_k: int, ids, tw, workspace, *, I: int = 128, SI: int = 0,
                    stream=None) -> None:
    """ids (int32 [M, k]) and tw (fp32 [M, k]) of x (bf16 [M, H]) under
    router_w (bf16 [E, H]).  `workspace` is a uint8 CUDA tensor sized by
    flint_moe_workspace_bytes for the same (M, H, E, top_k, I, SI)."""
    M, H = x.shape
    E = router_w.shape[0]
    s = _shape(M, H, E, top_k, I, SI)
    rc = load().flint_moe_route(_ptr(x), _ptr(router_w), ctypes.byref(s), _ptr(ids), _ptr(tw),
                                _ptr(workspace), workspace.numel(), _stream(stream))
    if rc != FLINT_OK:
        raise FlintMoEError(rc, "flint_moe_route")


def flint_moe_forward(x, router_w, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs, shared_gu, shared_down,
                      top_k: int, out, workspace, ids_out=None, tw_out=None, stream=None) -> None:
    """out (bf16 [M, H]) = MoE block of x; see include/flint_moe.h for the
    layouts.  shared_gu / shared_down may be None (no shared expert)."""
    M, H = x.shape
    E = router_w.shape[0]
    I = w2.shape[2] * 2
    SI = 0 if shared_down is None else shared_down.shape[1]
    s = _shape(M, H, E, top_k, I, SI)
    rc = load().flint_moe_forward(
        _ptr(x), _ptr(router_w), _ptr(w13), _ptr(w13_sf), _ptr(w13_gs), _ptr(w2), _ptr(w2_sf),
        _ptr(w2_gs), _ptr(shared_gu), _ptr(shared_down), ctypes.byref(s), _ptr(out), _ptr(ids_out),
        _ptr(tw_out), _ptr(workspace), workspace.numel(), _stream(stream))
    if rc != FLINT_OK:
        raise FlintMoEError(rc, "flint_moe_forward")


def flint_moe_forward_nvfp4_shared(x, router_w, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs, sgu, sgu_sf, sgu_gs,
                                   sdown, sdown_sf, sdown_gs, top_k: int, out, workspace, ids_out=None,
                                   tw_out=None, stream=None) -> None:
    """The block with an NVFP4 shared expert (codes, e4m3 scale bytes and a
    one-element fp32 global scale for its gate/up and its down)."""
    M, H = x.shape
    E = router_w.shape[0]
    I = w2.shape[2] * 2
    SI = sgu.shape[0] // 2
    s = _shape(M, H, E, top_k, I, SI)
    rc = load().flint_moe_forward_nvfp4_shared(
        _ptr(x), _ptr(router_w), _ptr(w13), _ptr(w13_sf), _ptr(w13_gs), _ptr(w2), _ptr(w2_sf), _ptr(w2_gs),
        _ptr(sgu), _ptr(sgu_sf), _ptr(sgu_gs), _ptr(sdown), _ptr(sdown_sf), _ptr(sdown_gs), ctypes.byref(s),
        _ptr(out), _ptr(ids_out), _ptr(tw_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream))
    if rc != FLINT_OK:
        raise FlintMoEError(rc, "flint_moe_forward_nvfp4_shared")


def flint_moe_forward_bf16(x, router_w, w13, w2, top_k: int, out, workspace, shared_out=None,
                           ids_out=None, tw_out=None, stream=None) -> None:
    """The block on BF16 routed experts (flint_moe_bf16_decode): w13 bf16
    [E, 2I, H], w2 bf16 [E, H, I], shared_out bf16 [M, H] or None."""
    M, H = x.shape
    E, I2, _ = w13.shape
    s = _shape(M, H, E, top_k, I2 // 2, 0)
    rc = load().flint_moe_forward_bf16(_ptr(x), _ptr(router_w), _ptr(w13), _ptr(w2), _ptr(shared_out),
                                       ctypes.byref(s), _ptr(out), _ptr(ids_out), _ptr(tw_out),
                                       _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream(stream))
    if rc != FLINT_OK:
        raise FlintMoEError(rc, "flint_moe_forward_bf16")


def flint_moe_forward_add_norm(attn_out, residual, ln_weight, eps: float, router_w, w13, w13_sf,
                               w13_gs, w2, w2_sf, w2_gs, shared_gu, shared_down, top_k: int, out,
                               residual_out, workspace, xn_out=None, ids_out=None, tw_out=None,
                               *, I: int, SI: int, stream=None) -> None:
    """The MoE block with its add-RMSNorm prologue (flint_moe_ll): writes out
    and residual_out (and xn_out when given)."""
    M, H = attn_out.shape
    E = router_w.shape[0]
    s = _shape(M, H, E, top_k, I, SI)
    rc = load().flint_moe_forward_add_norm(
        _ptr(attn_out), _ptr(residual), _ptr(ln_weight), float(eps), _ptr(router_w), _ptr(w13),
        _ptr(w13_sf), _ptr(w13_gs), _ptr(w2), _ptr(w2_sf), _ptr(w2_gs), _ptr(shared_gu),
        _ptr(shared_down), ctypes.byref(s), _ptr(out), _ptr(residual_out), _ptr(xn_out),
        _ptr(ids_out), _ptr(tw_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream))
    if rc != FLINT_OK:
        raise FlintMoEError(rc, "flint_moe_forward_add_norm")


def flint_moe_route_noalloc(x, router_w, top_k: int, ids, tw, stream=None) -> None:
    """flint_moe_route without a caller workspace: the library's fixed
    static scratch holds the intermediates (see include/flint_moe.h for the
    size limit and the rule that calls sharing a device must be ordered)."""
    M, H = x.shape
    E = router_w.shape[0]
    s = _shape(M, H, E, top_k, 128, 0)
    rc = load().flint_moe_route_noalloc(_ptr(x), _ptr(router_w), ctypes.byref(s), _ptr(ids),
                                        _ptr(tw), _stream(stream))
    if rc != FLINT_OK:
        raise FlintMoEError(rc, "flint_moe_route_noalloc")


def flint_moe_route_noalloc_bytes(M: int, H: int, E: int, top_k: int) -> int:
    s = _shape(M, H, E, top_k, 128, 0)
    return int(load().flint_moe_route_noalloc_bytes(ctypes.byref(s)))


def flint_moe_route_noalloc_capacity() -> int:
    return int(load().flint_moe_route_noalloc_capacity())


def flint_moe_plan(M: int, H: int, E: int, top_k: int, I: int, SI: int) -> int:
    """The FLINT_PATH_* flint_moe_forward takes for the shape on the current
    device; raises FlintMoEError for an invalid or unsupported shape."""
    s = _shape(M, H, E, top_k, I, SI)
    rc = int(load().flint_moe_plan(ctypes.byref(s)))
    if rc < 0:
        raise FlintMoEError(rc, "flint_moe_plan")
    return rc


def flint_moe_prefer_path(path: int) -> None:
    """Process-wide path preference (FLINT_PATH_NONE or FLINT_PATH_SINGLE_LAUNCH)."""
    rc = load().flint_moe_prefer_path(int(path))
    if rc != FLINT_OK:
        raise FlintMoEError(rc, "flint_moe_prefer_path")


SPAN_NAMES = ("route", "gate_up", "down", "single_launch", "group_count", "group_scan",
              "group_scatter", "plan", "gather", "gemm1", "gemm2", "combine", "add_norm",
              "shared_gate_up", "shared_down", "shared_add", "qkv_gemv", "qkv_heads")
SPAN_KERNELS = 18
SPAN_CTAS = 1024


def flint_moe_record_spans(buf) -> None:
    """Record kernel spans into `buf` (a zeroed int64 CUDA tensor of
    SPAN_KERNELS * SPAN_CTAS * 2 words), or stop recording (None)."""
    if buf is not None:
        assert buf.numel() * buf.element_size() >= SPAN_KERNELS * SPAN_CTAS * 16
    load().flint_moe_record_spans(_ptr(buf))


def spans_of(buf) -> dict:
    """{kernel name: (start ns, end ns)} of the kernels that recorded into buf."""
    a = buf.view(torch.int64).cpu().reshape(SPAN_KERNELS, SPAN_CTAS, 2)
    res = {}
    for i, name in enumerate(SPAN_NAMES):
        st, en = a[i, :, 0], a[i, :, 1]
        used = st != 0
        if bool(used.any()):
            start = int((~st[used]).min())
            res[name] = (start, int(en[used].max()))
    return res


def flint_moe_status(workspace, stream=None) -> int:
    """Synchronise `stream` and return (and clear) the workspace status word."""
    return int(load().flint_moe_status(_ptr(workspace), _stream(stream)))


def flint_moe_debug_fault(site: int) -> None:
    """Failure-path test hook (see include/flint_moe.h): leave one device
    signal out so that a bounded wait gives up; FLINT_FAULT_NONE turns it off."""
    rc = load().flint_moe_debug_fault(int(site))
    if rc != FLINT_OK:
        raise FlintMoEError(rc, "flint_moe_debug_fault")


# ---------------------------------------------------------------- helpers
def alloc_workspace(M: int, H: int, E: int, top_k: int, I: int, SI: int,
                    device="cuda") -> torch.Tensor:
    """A zero-filled workspace (do this once, outside graph capture)."""
    n = flint_moe_workspace_bytes(M, H, E, top_k, I, SI)
    if n == 0:
        code = FLINT_ERR_INVALID_ARG
        if all(v % 64 == 0 for v in (H, I, SI)) and not all(v % 128 == 0 for v in (H, I, SI)):
            code = FLINT_ERR_UNSUPPORTED
        raise FlintMoEError(code, "alloc_workspace")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def forward_add_norm_layer(attn_out, residual, ln_weight, eps: float, layer, top_k: int, workspace=None,
                           out=None, residual_out=None, xn_out=None, ids_out=None, tw_out=None,
                           stream=None):
    """flint_moe_forward_add_norm on a synth.MoELayer-like object; returns
    (out, residual_out)."""
    M, H = attn_out.shape
    if workspace is None:
        workspace = alloc_workspace(M, H, layer.E, top_k, layer.I, layer.SI, attn_out.device)
    if out is None:
        out = torch.empty_like(attn_out)
    if residual_out is None:
        residual_out = torch.empty_like(residual)
    flint_moe_forward_add_norm(attn_out, residual, ln_weight, eps, layer.router_w, layer.w13,
                               layer.w13_sf, layer.w13_gs, layer.w2, layer.w2_sf, layer.w2_gs,
                               layer.shared_gu if layer.SI else None,
                               layer.shared_down if layer.SI else None, top_k, out, residual_out,
                               workspace, xn_out=xn_out, ids_out=ids_out, tw_out=tw_out, I=layer.I,
                               SI=layer.SI, stream=stream)
    return out, residual_out


def forward_layer(x, layer, top_k: int, workspace=None, out=None, ids_out=None, tw_out=None,
                  stream=None):
    """flint_moe_forward on a synth.MoELayer-like object (CUDA tensors)."""
    M, H = x.shape
    if workspace is None:
        workspace = alloc_workspace(M, H, layer.E, top_k, layer.I, layer.SI, x.device)
    if out is None:
        out = torch.empty_like(x)
    flint_moe_forward(x, layer.router_w, layer.w13, layer.w13_sf, layer.w13_gs, layer.w2,
                      layer.w2_sf, layer.w2_gs, layer.shared_gu if layer.SI else None,
                      layer.shared_down if layer.SI else None, top_k, out, workspace,
                      ids_out=ids_out, tw_out=tw_out, stream=stream)
    return out


def flint_qkv_workspace_bytes(M: int, H: int, num_q_heads: int, num_kv_heads: int) -> int:
    """Workspace bytes of flint_qkv_fused (0 for an invalid or unsupported shape)."""
    return int(load().flint_qkv_workspace_bytes(int(M), int(H), int(num_q_heads), int(num_kv_heads)))


def flint_qkv_fused(x, residual, norm_weight, eps: float, weight, weight_scale, global_scale, q_norm_weight,
                    k_norm_weight, qk_eps: float, cos_sin_cache, positions, k_cache, v_cache, slot_mapping,
                    num_q_heads: int, num_kv_heads: int, q_out=None, residual_out=None, workspace=None,
                    stream=None):
    """Fused decode qkv (flint_qkv_fused on the qkv_fused page): input
    (add-)RMSNorm, the qkv GEMV (NVFP4 codes uint8 [N, H/2] with e4m3 scale
    bytes [N, H/16] and a one-element fp32 global scale, or BF16 [N, H]),
    per-head q/k RMSNorm, NeoX RoPE and the paged KV-cache write.  k_cache /
    v_cache: bf16 [blocks, block_size, kv_heads, 128] views (any strides but a
    unit last one).  Returns (q, residual_out or None)."""
    M, H = x.shape
    if q_out is None:
        q_out = torch.empty(M, num_q_heads * 128, dtype=torch.bfloat16, device=x.device)
    if residual is not None and residual_out is None:
        residual_out = torch.empty_like(x)
    if workspace is None:
        workspace = torch.zeros(max(1, flint_qkv_workspace_bytes(M, H, num_q_heads, num_kv_heads)),
                                dtype=torch.uint8, device=x.device)
    assert k_cache.stride() == v_cache.stride() and k_cache.stride(-1) == 1
    blocks, bs = k_cache.shape[0], k_cache.shape[1]
    max_pos = cos_sin_cache.shape[0] if cos_sin_cache is not None else 0
    rc = load().flint_qkv_fused(
        _ptr(x), _ptr(residual), _ptr(norm_weight), float(eps), _ptr(weight), _ptr(weight_scale),
        _ptr(global_scale), _ptr(q_norm_weight), _ptr(k_norm_weight), float(qk_eps), _ptr(cos_sin_cache),
        int(max_pos), _ptr(positions), _ptr(k_cache), _ptr(v_cache), int(k_cache.stride(0)),
        int(k_cache.stride(1)), int(k_cache.stride(2)), int(bs), int(blocks), _ptr(slot_mapping),
        int(slot_mapping.shape[0]) if slot_mapping is not None else 0, M, H, int(num_q_heads),
        int(num_kv_heads), _ptr(q_out), _ptr(residual_out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    if rc != FLINT_OK:
        raise FlintMoEError(rc, "flint_qkv_fused")
    return q_out, residual_out
