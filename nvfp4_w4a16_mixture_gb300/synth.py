"""Seeded synthetic inputs for the routed-expert NVFP4 MoE block.

This module is the one piece shared by the CUDA path's tests and benchmark and
by the CPU oracle's tests: it only draws random tensors and encodes expert
weights into the NVFP4 interchange layout (it decodes nothing and computes no
part of the block).  The layout is the ModelOpt one named on the vLLM page
"vllm.models.flint.ops.moe" (FlintMoEWeights.from_modelopt docstring):

* w13  uint8 [E, 2I, H/2]   gate rows [0, I), up rows [I, 2I); two e2m1 codes
                            per byte, even K index in the low nibble
* w13_sf  uint8 [E, 2I, H/16]  e4m3 block scales (float8_e4m3fn bit patterns)
* w13_gs  fp32 [E]           one global scale per expert (gate and up share it;
                            FlintNvfp4Experts._repack rejects unequal ones)
* w2   uint8 [E, H, I/2], w2_sf uint8 [E, H, I/16], w2_gs fp32 [E]

Recipe (the tiny / decode / prefill layer configurations of the MoE block):
x ~ N(0, 1) -> bf16; router W[E, H] ~ N(0, H^-1/2) -> bf16; expert weights
~ N(0, 0.02) fp32, quantised per 16-element K block with
gs = amax / (6 * 448) per expert and tensor, scale = e4m3_rne(blockamax / 6 / gs),
code = e2m1_rne(w / (scale * gs)) saturating at 6; shared-expert weights
~ N(0, 0.02) -> bf16.  Draw order: x, router W, w13 (expert by expert), w2
(expert by expert), shared gate_up, shared down.
"""
from __future__ import annotations

import dataclasses

import torch

E4M3_MAX = 448.0
E2M1_MAX = 6.0


@dataclasses.dataclass
class MoELayer:
    """One MoE layer's weights in the interchange layout (all contiguous)."""

    H: int
    E: int
    I: int
    SI: int
    router_w: torch.Tensor  # bf16 [E, H]
    w13: torch.Tensor  # uint8 [E, 2I, H/2]
    w13_sf: torch.Tensor  # uint8 [E, 2I, H/16]
    w13_gs: torch.Tensor  # fp32 [E]
    w2: torch.Tensor  # uint8 [E, H, I/2]
    w2_sf: torch.Tensor  # uint8 [E, H, I/16]
    w2_gs: torch.Tensor  # fp32 [E]
    shared_gu: torch.Tensor  # bf16 [2SI, H], gate rows then up rows
    shared_down: torch.Tensor  # bf16 [H, SI]

    def to(self, device) -> "MoELayer":
        kw = {f.name: getattr(self, f.name) for f in dataclasses.fields(self)}
        for k, v in kw.items():
            if isinstance(v, torch.Tensor):
                kw[k] = v.to(device).contiguous()
        return MoELayer(**kw)

    def expert_bytes(self) -> int:
        """Bytes of one routed expert's packed weights, scales and scales-2."""
        return (
            self.w13[0].numel() + self.w13_sf[0].numel() + self.w2[0].numel()
            + self.w2_sf[0].numel() + 8
        )


def e2m1_codes(q: torch.Tensor) -> torch.Tensor:
    """Round fp32 values to the nearest E2M1 code, ties to the even code,
    saturating at +-6.  Returns uint8 codes (bit 3 = sign)."""
    a = q.abs()
    # magnitude grid 0, .5, 1, 1.5, 2, 3, 4, 6 (codes 0..7); each comparison
    # crosses one midpoint, strict where the lower code is even.
    mag = (
        (a > 0.25).to(torch.uint8) + (a >= 0.75).to(torch.uint8)
        + (a > 1.25).to(torch.uint8) + (a >= 1.75).to(torch.uint8)
        + (a > 2.5).to(torch.uint8) + (a >= 3.5).to(torch.uint8)
        + (a > 5.0).to(torch.uint8)
    )
    sign = torch.signbit(q).to(torch.uint8) << 3
    return mag | sign


def pack_e2m1(codes: torch.Tensor) -> torch.Tensor:
    """[..., K] codes -> [..., K/2] bytes, even K index in the low nibble."""
    lo = codes[..., 0::2]
    hi = codes[..., 1::2]
    return (lo | (hi << 4)).contiguous()


def quantize_nvfp4(w: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """NVFP4-encode one expert's fp32 matrix [rows, K].

    Returns (packed codes uint8 [rows, K/2], e4m3 scale bytes uint8
    [rows, K/16], global scale fp32 scalar tensor)."""
    rows, K = w.shape
    assert K % 16 == 0
    w = w.float()
    gs = w.abs().amax() / (E2M1_MAX * E4M3_MAX)
    blocks = w.reshape(rows, K // 16, 16)
    bamax = blocks.abs().amax(-1)
    if float(gs) > 0:
        sf_f = (bamax / E2M1_MAX / gs).clamp(max=E4M3_MAX)
    else:
        sf_f = torch.zeros_like(bamax)
    sf8 = sf_f.to(torch.float8_e4m3fn)
    denom = sf8.to(torch.float32) * gs
    safe = torch.where(denom > 0, denom, torch.ones_like(denom))
    q = torch.where(denom[..., None] > 0, blocks / safe[..., None], torch.zeros_like(blocks))
    codes = e2m1_codes(q.reshape(rows, K))
    return pack_e2m1(codes), sf8.view(torch.uint8).contiguous(), gs.reshape(()).float()


def make_layer(H: int, E: int, I: int, SI: int, gen: torch.Generator, device="cpu",
               router_row_scale: torch.Tensor | None = None) -> MoELayer:
    """Router, routed experts and shared expert of one layer, drawn from `gen`
    in the recipe's order (after the caller has drawn x).

    router_row_scale (optional fp32 [E]) multiplies router row e; it is the
    knob of the skewed-routing workload and is 1 for every other one."""
    dev = torch.device(device)
    wr = torch.randn(E, H, generator=gen, device=dev) * (H ** -0.5)
    if router_row_scale is not None:
        wr = wr * router_row_scale.to(dev, torch.float32)[:, None]
    router_w = wr.to(torch.bfloat16).contiguous()
    w13 = torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, device=dev)
    w13_sf = torch.empty(E, 2 * I, H // 16, dtype=torch.uint8, device=dev)
    w13_gs = torch.empty(E, dtype=torch.float32, device=dev)
    for e in range(E):
        we = torch.randn(2 * I, H, generator=gen, device=dev) * 0.02
        w13[e], w13_sf[e], w13_gs[e] = quantize_nvfp4(we)
    w2 = torch.empty(E, H, I // 2, dtype=torch.uint8, device=dev)
    w2_sf = torch.empty(E, H, I // 16, dtype=torch.uint8, device=dev)
    w2_gs = torch.empty(E, dtype=torch.float32, device=dev)
    for e in range(E):
        we = torch.randn(H, I, generator=gen, device=dev) * 0.02
        w2[e], w2_sf[e], w2_gs[e] = quantize_nvfp4(we)
    sgu = (torch.randn(2 * SI, H, generator=gen, device=dev) * 0.02).to(torch.bfloat16)
    sdn = (torch.randn(H, SI, generator=gen, device=dev) * 0.02).to(torch.bfloat16)
    return MoELayer(H, E, I, SI, router_w, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs,
                    sgu.contiguous(), sdn.contiguous())


def make_x(M: int, H: int, gen: torch.Generator, device="cpu") -> torch.Tensor:
    return torch.randn(M, H, generator=gen, device=torch.device(device)).to(torch.bfloat16).contiguous()


def make_problem(M: int, H: int, E: int, k: int, I: int, SI: int, seed: int = 0, device="cpu",
                 router_row_scale: torch.Tensor | None = None):
    """(x, layer) of one configuration, seed `seed`, drawn in recipe order."""
    gen = torch.Generator(device=torch.device(device)).manual_seed(seed)
    x = make_x(M, H, gen, device)
    layer = make_layer(H, E, I, SI, gen, device, router_row_scale)
    return x, layer


# ------------------------------------------------------------ configurations
# name -> (M, H, E, k, I, SI).  The shapes of the MoE block's five workloads:
# a tiny layer, single-token decode, the decode batch sweep, the M=4096
# prefill batch and the skewed-routing M=16384 batch (same layer shapes).
CONFIGS = {
    "tiny": (2, 256, 8, 2, 128, 128),
    "decode1": (1, 2048, 128, 8, 768, 768),
    **{f"decode{m}": (m, 2048, 128, 8, 768, 768) for m in (2, 4, 8, 16, 32, 64)},
    "prefill4096": (4096, 2048, 128, 8, 768, 768),
    "skew16384": (16384, 2048, 128, 8, 768, 768),
}


def zipf_router_scale(E: int, alpha: float = 0.9055, seed: int = 1) -> torch.Tensor:
    """Per-expert router-row multipliers for the skewed-routing workload.

    Expert popularity is skewed by scaling router row e by c_r = r^-alpha,
    where r (1..E) is the rank a fixed random permutation (seed `seed`) gives
    e: a larger row norm gives larger-variance logits and so more top-k wins,
    and the rank-frequency curve falls off as a power law.  With x ~ N(0, 1)
    tokens, H = 2048, E = 128, top_k = 8, alpha = 0.9055 makes the 8 most
    popular experts take 40% of the assignments (bisection on 16384 probe
    tokens; the most popular single expert then takes about 6%, below the
    12.5% a top-8 choice without repeats allows).  tests/test_synth.py checks
    the share on independent probe tokens."""
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(E, generator=g)
    r = torch.arange(1, E + 1, dtype=torch.float64)
    c = torch.empty(E, dtype=torch.float64)
    c[perm] = r ** (-alpha)
    return c.float()


def flops_of(M: int, H: int, E: int, k: int, I: int, SI: int) -> dict:
    """Algorithmic flops of one forward (2 per multiply-add)."""
    routed = 2 * M * k * (2 * I * H + H * I)
    shared = 2 * M * (2 * SI * H + H * SI)
    router = 2 * M * E * H
    return {"routed": routed, "shared": shared, "router": router,
            "total": routed + shared + router}


def weight_bytes(H: int, E: int, I: int, SI: int, unique_experts: int) -> dict:
    """Algorithmic weight bytes one forward must read when `unique_experts`
    distinct experts are routed to."""
    per_expert = 2 * I * H // 2 + 2 * I * H // 16 + H * I // 2 + H * I // 16 + 8
    return {"per_expert": per_expert, "experts": unique_experts * per_expert,
            "router": E * H * 2, "shared": 3 * SI * H * 2,
            "total": unique_experts * per_expert + E * H * 2 + 3 * SI * H * 2}


__all__ = ["MoELayer", "CONFIGS", "make_problem", "make_layer", "make_x", "quantize_nvfp4",
           "e2m1_codes", "pack_e2m1", "zipf_router_scale", "flops_of", "weight_bytes"]
