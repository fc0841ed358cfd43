"""Independent float64 re-derivation of the MoE block (a pin for the oracle).

Written separately from oracle/flint_oracle.c and sharing nothing with it:
block scales are decoded by torch's float8_e4m3fn conversion (a library
routine), E2M1 codes through their exact embedding into E4M3 (same sign,
exponent shifted by 6, mantissa bit moved to the top mantissa bit, so that
e4m3(embed(c)) = e2m1(c) * 2^-6 for every code, subnormals included), and
every dot product is accumulated in float64 (numpy) and rounded once.  The
rounding points are the ones the vLLM page "vllm.models.flint.ops.moe" states
in its Numerics paragraph.  Because the sums are far more accurate than fp32,
the result differs from the fp32 oracle only by fp32 accumulation noise, and
routing differs only where a float64 logit sits within that noise of a bf16
rounding boundary (reported as "ambiguous").
"""
from __future__ import annotations

import numpy as np
import torch


def bf16_from_f32(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 values (as float32) via torch's RNE conversion."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def tensor_bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def e4m3_decode(bytes_u8: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bytes_u8, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    c = codes.astype(np.uint8)
    embed = ((c & 8) << 4) | ((c & 7) << 2)
    return e4m3_decode(embed) * 64.0


def dequant(packed: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """[rows, K/2] bytes + [rows, K/16] scales -> float64 [rows, K]."""
    lo = packed & 15
    hi = packed >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(packed.shape[0], -1)
    vals = e2m1_decode(codes)
    scale = np.repeat(e4m3_decode(sf), 16, axis=-1)
    return vals * scale


def order_key(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    return np.where(b >= 0x8000, b ^ 0xFFFF, b | 0x8000)


def forward64(x: torch.Tensor, layer, top_k: int, tokens=None):
    """Block output (bf16 bits) plus routing and the per-token ambiguity flag."""
    xb = tensor_bits(x)
    xf = bf16_bits_to_f64(xb)
    M, H = xf.shape
    wr = bf16_bits_to_f64(tensor_bits(layer.router_w))
    E, I, SI = layer.E, layer.I, layer.SI
    toks = range(M) if tokens is None else [int(t) for t in tokens]
    w13 = layer.w13.numpy()
    w13_sf = layer.w13_sf.numpy()
    w2 = layer.w2.numpy()
    w2_sf = layer.w2_sf.numpy()
    gs13 = layer.w13_gs.numpy().astype(np.float64)
    gs2 = layer.w2_gs.numpy().astype(np.float64)
    if SI:
        sgu = bf16_bits_to_f64(tensor_bits(layer.shared_gu))
        sdn = bf16_bits_to_f64(tensor_bits(layer.shared_down))
    deq13, deq2 = {}, {}
    outs, ids_all, tw_all, amb_all = [], [], [], []
    for t in toks:
        xt = xf[t]
        lg64 = wr @ xt
        lg32 = lg64.astype(np.float32)
        lgb = bf16_from_f32(lg32)
        bits = lgb.view(np.uint32) >> 16
        # ambiguity: the fp64 logit is within fp32 accumulation noise of a
        # bf16 rounding midpoint, so an fp32 sum may round either way
        noise = 4 * H * np.finfo(np.float32).eps * (np.abs(wr) @ np.abs(xt))
        lo = bf16_from_f32((lg64 - noise).astype(np.float32))
        hi = bf16_from_f32((lg64 + noise).astype(np.float32))
        amb_e = lo != hi
        key = order_key(bits)
        order = sorted(range(E), key=lambda e: (-key[e], e))
        sel = order[:top_k]
        # selection can only change if an ambiguous logit is at the k boundary
        amb = bool(amb_e[order[: top_k + 1]].any())
        s = 1.0 / (1.0 + np.exp(-lgb[sel].astype(np.float64)))
        tw = bf16_from_f32((s / (s.sum() + 1e-20)).astype(np.float32)).astype(np.float64)
        R = np.zeros(H)
        for j, e in enumerate(sel):
            if e not in deq13:
                deq13[e] = dequant(w13[e], w13_sf[e])
                deq2[e] = dequant(w2[e], w2_sf[e])
            gu = (deq13[e] @ xt) * gs13[e]
            g = gu[:I].astype(np.float32).astype(np.float64)
            u = gu[I:].astype(np.float32).astype(np.float64)
            act = bf16_from_f32((g / (1.0 + np.exp(-g)) * u).astype(np.float32)).astype(np.float64)
            y = bf16_from_f32(((deq2[e] @ act) * gs2[e]).astype(np.float32)).astype(np.float64)
            R += tw[j] * y
        Rb = bf16_from_f32(R.astype(np.float32)).astype(np.float64)
        if SI:
            gS = bf16_from_f32((sgu[:SI] @ xt).astype(np.float32)).astype(np.float64)
            uS = bf16_from_f32((sgu[SI:] @ xt).astype(np.float32)).astype(np.float64)
            sact = bf16_from_f32((gS / (1.0 + np.exp(-gS)) * uS).astype(np.float32)).astype(np.float64)
            ys = bf16_from_f32((sdn @ sact).astype(np.float32)).astype(np.float64)
        else:
            ys = np.zeros(H)
        out = bf16_from_f32((Rb + ys).astype(np.float32))
        outs.append(out.view(np.uint32) >> 16)
        ids_all.append(sel)
        tw_all.append(tw)
        amb_all.append(amb)
    return {
        "out": np.stack(outs).astype(np.uint16),
        "ids": np.array(ids_all, dtype=np.int32),
        "tw": np.array(tw_all, dtype=np.float32),
        "ambiguous": np.array(amb_all, dtype=bool),
    }
