"""CPU oracle of the Flint NVFP4 W4A16 routed-expert MoE block.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (the C-ABI library and its Python binding) never
imports it, and this package imports nothing from the product path.

The arithmetic lives in ``flint_oracle.c`` (plain C, one IEEE binary32
operation per C operator, compiled with ``-O2 -ffp-contract=off``).  This file
only compiles it with gcc and marshals numpy / torch CPU arrays through ctypes.
Rules and citations are in the C file's header.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "flint_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libflint_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over tokens).  Returns the .so path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
           "-std=c11", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    """Declare the C signatures on a loaded oracle library."""
    P = ctypes.c_void_p
    i32 = ctypes.c_int
    lib.oracle_e2m1_value.restype = ctypes.c_float
    lib.oracle_e2m1_value.argtypes = [i32]
    lib.oracle_e4m3_value.restype = ctypes.c_float
    lib.oracle_e4m3_value.argtypes = [i32]
    lib.oracle_bf16_round.restype = None
    lib.oracle_bf16_round.argtypes = [P, P, ctypes.c_int64]
    lib.oracle_nvfp4_dequant.restype = None
    lib.oracle_nvfp4_dequant.argtypes = [P, P, ctypes.c_int64, i32, P]
    lib.oracle_route.restype = i32
    lib.oracle_route.argtypes = [P, P, i32, i32, i32, i32, P, P, P]
    lib.oracle_topk.restype = i32
    lib.oracle_topk.argtypes = [P, i32, i32, i32, P, P]
    lib.oracle_forward.restype = i32
    lib.oracle_forward.argtypes = [P] * 10 + [i32] * 6 + [P, i32] + [P] * 8 + [i32]
    lib.oracle_shared_nvfp4.restype = i32
    lib.oracle_shared_nvfp4.argtypes = [P, P, P, ctypes.c_float, P, P, ctypes.c_float, i32, i32, i32, P, P]
    lib.oracle_forward_bf16.restype = i32
    lib.oracle_forward_bf16.argtypes = [P] * 5 + [i32] * 5 + [P] * 5 + [i32]
    lib.oracle_add_rms_norm.restype = i32
    lib.oracle_add_rms_norm.argtypes = [P, P, P, i32, i32, ctypes.c_float, P, P]
    lib.oracle_max_threads.restype = i32
    lib.oracle_max_threads.argtypes = []
    lib.oracle_qkv_fused.restype = i32
    lib.oracle_qkv_fused.argtypes = ([P, P, P, ctypes.c_float, P, P, ctypes.c_float, P, P, P, ctypes.c_float,
                                      P, P, P, i32, i32, i32, i32, i32, i32, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_int64] + [P] * 6)
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def build_variant(source: str, out_path: str) -> str:
    """Test hook: compile another version of the oracle's C source (a
    planted mistake) with the oracle's own flags; returns the .so path."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source)
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
                    "-std=c11", "-o", out_path, src, "-lm"], check=True)
    return out_path


@contextlib.contextmanager
def using_library(path: str):
    """Test hook: route every oracle call to the library at `path` (built by
    build_variant) for the duration of the block."""
    global _lib
    _load()
    with _lock:
        saved, _lib = _lib, _bind(ctypes.CDLL(path))
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def source() -> str:
    """The oracle's C source text (for test variants)."""
    with open(_SRC) as f:
        return f.read()


def _np(t, dtype):
    """torch (CPU) tensor or numpy array -> contiguous numpy array of dtype
    (bit reinterpretation for bf16 / fp8, never a value conversion)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                t = t.view(torch.int16)
            elif t.dtype == torch.float8_e4m3fn:
                t = t.view(torch.uint8)
            t = t.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(t)
    if a.dtype != dtype:
        if a.dtype.itemsize == np.dtype(dtype).itemsize and a.dtype.kind in "iu" and np.dtype(dtype).kind in "iu":
            a = a.view(dtype)
        else:
            a = a.astype(dtype)
    return a


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def e2m1_value(code: int) -> float:
    return float(_load().oracle_e2m1_value(int(code)))


def e4m3_value(byte: int) -> float:
    return float(_load().oracle_e4m3_value(int(byte)))


def bf16_round_bits(x) -> np.ndarray:
    """fp32 array -> uint16 bf16 bit patterns, round to nearest even."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(a.shape, dtype=np.uint16)
    _load().oracle_bf16_round(_ptr(a), _ptr(out), a.size)
    return out


def bf16_bits_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits).astype(np.uint32) << 16
    return b.view(np.float32)


def nvfp4_dequant(codes, sf, K: int) -> np.ndarray:
    """Dequantise packed NVFP4 rows ([rows, K/2] codes, [rows, K/16] scales)."""
    c = _np(codes, np.uint8)
    s = _np(sf, np.uint8)
    rows = c.size // (K // 2)
    out = np.empty((rows, K), dtype=np.float32)
    _load().oracle_nvfp4_dequant(_ptr(c), _ptr(s), rows, K, _ptr(out))
    return out.reshape(tuple(c.shape[:-1]) + (K,))


def route(x, router_w, top_k: int):
    """Returns (logits bf16 bits uint16 [M, E], ids int32 [M, k], tw fp32 [M, k])."""
    xa = _np(x, np.uint16)
    wa = _np(router_w, np.uint16)
    M, H = xa.shape
    E = wa.shape[0]
    logits = np.empty((M, E), dtype=np.uint16)
    ids = np.empty((M, top_k), dtype=np.int32)
    tw = np.empty((M, top_k), dtype=np.float32)
    rc = _load().oracle_route(_ptr(xa), _ptr(wa), M, H, E, top_k, _ptr(logits), _ptr(ids), _ptr(tw))
    if rc != 0:
        raise ValueError("oracle_route: invalid shape")
    return logits, ids, tw


def topk(logit_bits, top_k: int):
    """Top-k on given bf16 logits (uint16 bit patterns [M, E])."""
    lb = _np(logit_bits, np.uint16)
    M, E = lb.shape
    ids = np.empty((M, top_k), dtype=np.int32)
    tw = np.empty((M, top_k), dtype=np.float32)
    if _load().oracle_topk(_ptr(lb), M, E, top_k, _ptr(ids), _ptr(tw)) != 0:
        raise ValueError("oracle_topk: invalid shape")
    return ids, tw


def forward(x, layer, top_k: int, tokens=None, intermediates: bool = False, nthreads: int = 0):
    """The whole block for the selected tokens (all by default).

    ``layer`` is a synth.MoELayer (CPU tensors) or anything with the same
    attributes.  Returns a dict of numpy arrays: out (bf16 bits [n, H]), ids,
    tw and, with ``intermediates``, logits, act, y, sact, ys."""
    xa = _np(x, np.uint16)
    M, H = xa.shape
    E, I, SI = int(layer.E), int(layer.I), int(layer.SI)
    k = int(top_k)
    arrs = [
        xa, _np(layer.router_w, np.uint16), _np(layer.w13, np.uint8), _np(layer.w13_sf, np.uint8),
        _np(layer.w13_gs, np.float32), _np(layer.w2, np.uint8), _np(layer.w2_sf, np.uint8),
        _np(layer.w2_gs, np.float32), _np(layer.shared_gu, np.uint16) if SI else None,
        _np(layer.shared_down, np.uint16) if SI else None,
    ]
    tok = None if tokens is None else np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    n = M if tok is None else tok.size
    res = {"out": np.empty((n, H), np.uint16), "ids": np.empty((n, k), np.int32),
           "tw": np.empty((n, k), np.float32)}
    if intermediates:
        res.update(logits=np.empty((n, E), np.uint16), act=np.empty((n, k, I), np.uint16),
                   y=np.empty((n, k, H), np.uint16), sact=np.empty((n, max(SI, 1)), np.uint16),
                   ys=np.empty((n, H), np.uint16))
    g = res.get
    rc = _load().oracle_forward(
        *[_ptr(a) for a in arrs], M, H, E, k, I, SI, _ptr(tok), n,
        _ptr(res["out"]), _ptr(res["ids"]), _ptr(res["tw"]), _ptr(g("logits")), _ptr(g("act")),
        _ptr(g("y")), _ptr(g("sact")), _ptr(g("ys")), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_forward: invalid shape or token list")
    return res


def shared_nvfp4(x, sgu, sgu_sf, sgu_gs: float, sdn, sdn_sf, sdn_gs: float):
    """NVFP4 shared expert (reading R10): returns (ys bits [M, H], sact bits
    [M, SI])."""
    xa = _np(x, np.uint16)
    M, H = xa.shape
    ga, gfa = _np(sgu, np.uint8), _np(sgu_sf, np.uint8)
    da, dfa = _np(sdn, np.uint8), _np(sdn_sf, np.uint8)
    SI = ga.shape[0] // 2
    assert ga.shape == (2 * SI, H // 2) and gfa.shape == (2 * SI, H // 16)
    assert da.shape == (H, SI // 2) and dfa.shape == (H, SI // 16)
    ys = np.empty((M, H), np.uint16)
    sact = np.empty((M, SI), np.uint16)
    rc = _load().oracle_shared_nvfp4(_ptr(xa), _ptr(ga), _ptr(gfa), float(sgu_gs), _ptr(da), _ptr(dfa),
                                     float(sdn_gs), M, H, SI, _ptr(ys), _ptr(sact))
    if rc != 0:
        raise ValueError("oracle_shared_nvfp4: invalid shape")
    return ys, sact


def forward_bf16(x, router_w, w13, w2, top_k: int, shared_out=None, intermediates: bool = False,
                 nthreads: int = 0):
    """BF16 routed experts (reading R9): w13 bf16 [E, 2I, H], w2 bf16 [E, H, I],
    shared_out bf16 [M, H] or None.  Returns out (bits), ids, tw and, with
    ``intermediates``, act [M, k, I] and y [M, k, H] (bits)."""
    xa, wra = _np(x, np.uint16), _np(router_w, np.uint16)
    w13a, w2a = _np(w13, np.uint16), _np(w2, np.uint16)
    M, H = xa.shape
    E, I2, H2 = w13a.shape
    I = I2 // 2
    assert H2 == H and w2a.shape == (E, H, I)
    sh = None if shared_out is None else _np(shared_out, np.uint16)
    k = int(top_k)
    res = {"out": np.empty((M, H), np.uint16), "ids": np.empty((M, k), np.int32),
           "tw": np.empty((M, k), np.float32)}
    if intermediates:
        res.update(act=np.empty((M, k, I), np.uint16), y=np.empty((M, k, H), np.uint16))
    g = res.get
    rc = _load().oracle_forward_bf16(_ptr(xa), _ptr(wra), _ptr(w13a), _ptr(w2a), _ptr(sh), M, H, E, k, I,
                                     _ptr(res["out"]), _ptr(res["ids"]), _ptr(res["tw"]), _ptr(g("act")),
                                     _ptr(g("y")), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_forward_bf16: invalid shape")
    return res


def add_rms_norm(a, r, w, eps: float):
    """norm.fused_add_rms_norm (reading R8) of bf16 rows a + r with bf16
    weight w [H]: returns (residual' bits, xn bits), both [M, H] uint16."""
    aa, ra, wa = _np(a, np.uint16), _np(r, np.uint16), _np(w, np.uint16)
    M, H = aa.shape
    assert ra.shape == (M, H) and wa.shape == (H,)
    res = np.empty((M, H), np.uint16)
    xn = np.empty((M, H), np.uint16)
    rc = _load().oracle_add_rms_norm(_ptr(aa), _ptr(ra), _ptr(wa), M, H, float(eps), _ptr(res), _ptr(xn))
    if rc != 0:
        raise ValueError("oracle_add_rms_norm: invalid shape")
    return res, xn


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def qkv_fused(x, residual, norm_w, eps: float, weight, weight_scale, global_scale, q_norm_w, k_norm_w,
              qk_eps: float, cos_sin, positions, k_cache, v_cache, slot_mapping, nq: int, nkv: int):
    """Fused decode qkv (reading R11).  weight: NVFP4 codes uint8 [N, H/2]
    (with weight_scale uint8 [N, H/16] and the fp32 global_scale) or BF16
    [N, H] (weight_scale None).  k_cache / v_cache: bf16 [blocks,
    block_size, nkv, 128] arrays, updated in place (numpy) at the mapped
    slots.  Returns (q bits [M, nq*128], residual' bits [M, H] or None,
    xn bits [M, H], qkv bits [M, N])."""
    xa = _np(x, np.uint16)
    M, H = xa.shape
    ra = None if residual is None else _np(residual, np.uint16)
    nwa = _np(norm_w, np.uint16)
    N = (nq + 2 * nkv) * 128
    nvfp4 = weight_scale is not None
    if nvfp4:
        wc, wsf, wb = _np(weight, np.uint8), _np(weight_scale, np.uint8), None
        assert wc.shape == (N, H // 2) and wsf.shape == (N, H // 16)
        gs = float(global_scale)
    else:
        wc, wsf, wb = None, None, _np(weight, np.uint16)
        assert wb.shape == (N, H)
        gs = 1.0
    qa, ka = _np(q_norm_w, np.uint16), _np(k_norm_w, np.uint16)
    cs = None if cos_sin is None else np.ascontiguousarray(np.asarray(cos_sin, np.float32))
    pos = np.ascontiguousarray(np.asarray(positions, np.int64))
    slots = np.ascontiguousarray(np.asarray(slot_mapping, np.int64))
    assert isinstance(k_cache, np.ndarray) and isinstance(v_cache, np.ndarray)
    assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous and v_cache.shape == k_cache.shape
    blocks, bs, kv_heads, D = k_cache.shape
    assert kv_heads == nkv and D == 128
    q = np.empty((M, nq * 128), np.uint16)
    res = np.empty((M, H), np.uint16) if ra is not None else None
    xn = np.empty((M, H), np.uint16)
    qkv = np.empty((M, N), np.uint16)
    rc = _load().oracle_qkv_fused(_ptr(xa), _ptr(ra), _ptr(nwa), float(eps), _ptr(wc), _ptr(wsf), gs, _ptr(wb),
                                  _ptr(qa), _ptr(ka), float(qk_eps), _ptr(cs), _ptr(pos), _ptr(slots),
                                  int(slots.shape[0]), M, H, nq, nkv, bs, bs * kv_heads * D, kv_heads * D, D,
                                  _ptr(k_cache), _ptr(v_cache), _ptr(q), _ptr(res), _ptr(xn), _ptr(qkv))
    if rc != 0:
        raise ValueError("oracle_qkv_fused: invalid arguments")
    return q, res, xn, qkv
