"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test names what fixes the expected value: a library conversion, a closed
form, brute force, an independent float64 re-derivation, or a special case
that reduces to a library matmul.  Everything runs on the CPU.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from fp64_reference import (bf16_bits_to_f64, dequant, e2m1_decode, forward64, order_key,
                            tensor_bits)
from nvfp4_w4a16_mixture_gb300 import synth
from tolerance import bits_to_f64, check_bf16


# ----------------------------------------------------------------- formats
def test_e4m3_decode_matches_torch():
    """All 256 float8_e4m3fn patterns against torch's conversion (library)."""
    lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    ref = lib.to(torch.float32).numpy()
    got = np.array([oracle.e4m3_value(b) for b in range(256)], dtype=np.float32)
    nan = np.isnan(ref)
    assert nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e2m1_decode_via_e4m3_embedding():
    """E2M1 codes through their exact E4M3 embedding, decoded by torch."""
    ref = e2m1_decode(np.arange(16))
    got = np.array([oracle.e2m1_value(c) for c in range(16)])
    assert np.array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.arange(16) >= 8)


def test_e2m1_closed_form_facts():
    """Format facts: 8 magnitudes, max 6, smallest positive 0.5 (subnormal),
    sign-symmetric."""
    v = np.array([oracle.e2m1_value(c) for c in range(16)])
    assert v.max() == 6.0 and v.min() == -6.0
    assert np.min(v[v > 0]) == 0.5
    assert np.array_equal(v[8:], -v[:8])
    assert len(set(np.abs(v).tolist())) == 8


def test_dequant_products_exact_in_bf16():
    """Brute force over all 16 x 254 finite (code, scale) pairs: the oracle's
    dequantised weight equals the float64 product and survives a bf16
    round trip (the pages: weights dequantised exactly)."""
    codes = np.arange(16, dtype=np.uint8)
    scales = np.array([b for b in range(256) if (b & 0x7F) != 0x7F], dtype=np.uint8)
    # one row per scale, 16 codes packed (even K in the low nibble)
    row_codes = np.tile(codes, (scales.size, 1))
    packed = (row_codes[:, 0::2] | (row_codes[:, 1::2] << 4)).astype(np.uint8)
    sf = scales[:, None].astype(np.uint8)
    got = oracle.nvfp4_dequant(packed, sf, 16)
    ref = np.outer(
        torch.from_numpy(scales).view(torch.float8_e4m3fn).to(torch.float64).numpy(),
        e2m1_decode(codes))
    assert np.array_equal(got.astype(np.float64), ref)
    rt = torch.from_numpy(got).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(rt, got)


def test_bf16_rounding_matches_torch():
    """fp32 -> bf16 RNE against torch's conversion: 2^22 random patterns plus
    every exponent with tie, above-tie, below-tie and saturating mantissas."""
    rng = np.random.default_rng(0)
    rand = rng.integers(0, 2 ** 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    exps = np.arange(256, dtype=np.uint32) << 23
    mants = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0x18000, 0x17FFF, 0x7FFFFF, 0x7F8000,
                      0x7F7FFF, 0x10000], dtype=np.uint32)
    special = (exps[:, None] | mants[None, :]).ravel()
    pats = np.concatenate([rand, special, special | 0x80000000])
    f = pats.view(np.float32)
    got = oracle.bf16_round_bits(f)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.isnan(bits_to_f64(got[nan])).all()


def test_nibble_and_scale_placement():
    """Hand-built row: code c at K index c (c = 0..15) and a different scale
    per 16-block lands at the documented positions (even K = low nibble)."""
    K = 32
    codes = np.array(list(range(16)) + list(range(15, -1, -1)), dtype=np.uint8)
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)[None, :]
    sf = np.array([[0x38, 0x40]], dtype=np.uint8)  # 1.0 and 2.0
    got = oracle.nvfp4_dequant(packed, sf, K)[0]
    e2 = e2m1_decode(np.arange(16))
    assert np.array_equal(got[:16], e2)
    assert np.array_equal(got[16:], 2.0 * e2[::-1])


# --------------------------------------------------------------- quantiser
def test_quantiser_round_trip_and_midpoints():
    """Values on the E2M1 grid (times one power-of-two factor) quantise to
    exactly their own codes with a saturated block scale; E2M1 midpoints round
    to the even code."""
    mid = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, -0.25, -5.0, 0.0, -0.0])
    want = torch.tensor([0, 2, 2, 4, 4, 6, 6, 7, 8, 14, 0, 8], dtype=torch.uint8)
    assert torch.equal(synth.e2m1_codes(mid), want)
    g = torch.Generator().manual_seed(3)
    grid = torch.tensor([0.0, 0.5, 1, 1.5, 2, 3, 4, 6])
    vals = grid[torch.randint(0, 8, (64, 128), generator=g)]
    vals = vals * torch.where(torch.rand(64, 128, generator=g) < 0.5, -1.0, 1.0)
    # make every 16-block's max magnitude 6 so the block scale is exactly 1 * gs
    vals[:, ::16] = 6.0
    w = vals * 0.125
    packed, sf, gs = synth.quantize_nvfp4(w)
    # every block max is the tensor max, so every block scale saturates at 448
    assert (sf == 0x7E).all()
    assert float(gs) == np.float32(0.75) / np.float32(6 * 448)
    deq = oracle.nvfp4_dequant(packed.numpy(), sf.numpy(), 128)
    assert np.array_equal(deq, (vals * 448.0).numpy())


# ---------------------------------------------------------------- routing
def _brute_force_rank(logit_bits: np.ndarray, k: int) -> list[int]:
    """Full stable sort: numeric value descending, +0 above -0, then lower
    expert index (the pages' tie rule), written with float comparisons."""
    vals = bits_to_f64(logit_bits)
    neg_zero = (logit_bits == 0x8000)
    items = list(range(len(vals)))
    items.sort(key=lambda e: (-vals[e], 1 if neg_zero[e] else 0, e))
    return items[:k]


@pytest.mark.parametrize("E,k", [(8, 2), (16, 16), (128, 8), (256, 8), (32, 1)])
def test_topk_matches_brute_force_sort(E, k):
    g = torch.Generator().manual_seed(E * 31 + k)
    M, H = 24, 256
    x = synth.make_x(M, H, g)
    wr = (torch.randn(E, H, generator=g) * H ** -0.5).to(torch.bfloat16)
    if E >= 16:  # duplicated rows -> identical logits -> lower index wins
        wr[E - 1] = wr[3]
        wr[E // 2] = wr[E // 2 + 1]
    logits, ids, tw = oracle.route(x, wr, k)
    for t in range(M):
        assert ids[t].tolist() == _brute_force_rank(logits[t], k)


def test_topk_signed_zero_and_ties_constructed():
    """Constructed logits: ties go to the lower index and +0 ranks above -0
    (stand-alone top-k on given logits)."""
    vals = torch.tensor([0.5, -0.0, 0.0, 0.5, -1.0, 2.0, 0.0, -0.0], dtype=torch.bfloat16)
    bits = vals.view(torch.int16).numpy().view(np.uint16)[None, :]
    ids, _ = oracle.topk(bits, 8)
    assert ids[0].tolist() == [5, 0, 3, 2, 6, 1, 7, 4]
    assert ids[0].tolist() == _brute_force_rank(bits[0], 8)


def test_router_sum_never_yields_negative_zero():
    """The router GEMV sums from +0, and +0 + -0 = +0 in IEEE arithmetic: a
    row of -0 products gives a +0 logit, which then ties by index."""
    H, E = 16, 8
    x = torch.zeros(1, H, dtype=torch.bfloat16)
    x[0, 0] = 1.0
    col = torch.tensor([0.5, -0.0, 0.0, 0.5, -1.0, 2.0, 0.0, -0.0], dtype=torch.bfloat16)
    wr = torch.zeros(E, H, dtype=torch.bfloat16)
    wr[:, 0] = col
    logits, ids, _ = oracle.route(x, wr, E)
    assert logits[0, 1] == 0 and logits[0, 7] == 0
    assert ids[0].tolist() == [5, 0, 3, 1, 2, 6, 7, 4]


def test_routing_weights_renormalise():
    """tw is bf16-valued, positive, sums to 1 within k * 2^-9 (bf16 rounding
    of each weight); top_k = 1 gives exactly 1."""
    M, H, E, k = 64, 512, 64, 8
    g = torch.Generator().manual_seed(5)
    x = synth.make_x(M, H, g)
    wr = (torch.randn(E, H, generator=g) * H ** -0.5).to(torch.bfloat16)
    _, ids, tw = oracle.route(x, wr, k)
    assert np.array_equal(tw.view(np.uint32) & 0xFFFF, np.zeros_like(tw.view(np.uint32)))
    assert (tw > 0).all()
    assert np.abs(tw.astype(np.float64).sum(1) - 1.0).max() <= k * 2.0 ** -9
    _, _, tw1 = oracle.route(x, wr, 1)
    assert (tw1 == 1.0).all()


def test_router_logits_match_float64():
    """Canonical-order fp32 logits agree with the exactly summed float64
    logit rounded to bf16, except within fp32 noise of a rounding midpoint."""
    M, H, E = 32, 2048, 128
    g = torch.Generator().manual_seed(11)
    x = synth.make_x(M, H, g)
    wr = (torch.randn(E, H, generator=g) * H ** -0.5).to(torch.bfloat16)
    logits, _, _ = oracle.route(x, wr, 8)
    xf = bf16_bits_to_f64(tensor_bits(x))
    wf = bf16_bits_to_f64(tensor_bits(wr))
    exact = xf @ wf.T
    got = bits_to_f64(logits)
    lsb = np.exp2(np.floor(np.log2(np.abs(exact))) - 7)
    assert (np.abs(got - exact) <= lsb).all()  # within one bf16 ulp always
    rounded = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert (got == rounded).mean() > 0.999


# ------------------------------------------------------- whole-block pins
@pytest.fixture(scope="module")
def tiny():
    M, H, E, k, I, SI = synth.CONFIGS["tiny"]
    x, layer = synth.make_problem(16, H, E, k, I, SI, seed=0)
    return x, layer, k


def test_oracle_matches_float64_tiny(tiny):
    x, layer, k = tiny
    r = oracle.forward(x, layer, k)
    q = forward64(x, layer, k)
    sel = ~q["ambiguous"]
    assert np.array_equal(r["ids"][sel], q["ids"][sel])
    check_bf16(r["out"], q["out"])


@pytest.mark.slow
def test_oracle_matches_float64_decode_layer():
    M, H, E, k, I, SI = synth.CONFIGS["decode8"]
    x, layer = synth.make_problem(M, H, E, k, I, SI, seed=0)
    r = oracle.forward(x, layer, k)
    q = forward64(x, layer, k)
    sel = ~q["ambiguous"]
    assert np.array_equal(r["ids"][sel], q["ids"][sel])
    check_bf16(r["out"], q["out"])


def test_combine_top1_reduces_to_sum(tiny):
    """top_k = 1: tw = 1 exactly, so out = bf16(y_0 + ys) for every element
    (torch's fp32 add and bf16 rounding on the oracle's own intermediates)."""
    x, layer, _ = tiny
    r = oracle.forward(x, layer, 1, intermediates=True)
    assert (r["tw"] == 1.0).all()
    y0 = torch.from_numpy(bits_to_f64(r["y"][:, 0, :]).astype(np.float32))
    ys = torch.from_numpy(bits_to_f64(r["ys"]).astype(np.float32))
    want = (y0 + ys).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(r["out"], want)


def test_all_experts_equals_dense_mixture(tiny):
    """k = E: the routed block equals the dense renormalised-sigmoid mixture of
    every expert (float64 matmuls on torch-decoded weights), within the rule."""
    x, layer, _ = tiny
    E, H, I = layer.E, layer.H, layer.I
    r = oracle.forward(x, layer, E, intermediates=True)
    xf = bf16_bits_to_f64(tensor_bits(x))
    wr = bf16_bits_to_f64(tensor_bits(layer.router_w))
    lg = torch.from_numpy((xf @ wr.T).astype(np.float32)).to(torch.bfloat16).double().numpy()
    s = 1 / (1 + np.exp(-lg))
    tw = torch.from_numpy((s / s.sum(1, keepdims=True)).astype(np.float32)).to(torch.bfloat16).double().numpy()
    R = np.zeros((x.shape[0], H))
    for e in range(E):
        d13 = dequant(layer.w13[e].numpy(), layer.w13_sf[e].numpy())
        d2 = dequant(layer.w2[e].numpy(), layer.w2_sf[e].numpy())
        gu = (xf @ d13.T) * float(layer.w13_gs[e])
        g, u = gu[:, :I], gu[:, I:]
        act = torch.from_numpy((g / (1 + np.exp(-g)) * u).astype(np.float32)).to(torch.bfloat16).double().numpy()
        y = torch.from_numpy(((act @ d2.T) * float(layer.w2_gs[e])).astype(np.float32)).to(torch.bfloat16).double().numpy()
        R += tw[:, e:e + 1] * y
    Rb = torch.from_numpy(R.astype(np.float32)).to(torch.bfloat16).double().numpy()
    ys = bits_to_f64(r["ys"])
    want = torch.from_numpy((Rb + ys).astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    check_bf16(r["out"], want)


def test_unit_scales_reduce_to_matmul():
    """All block scales 1.0 (e4m3 0x38) and global scales 1: the NVFP4 gate/up
    projection is a plain matmul on the E2M1 grid (torch float64 matmul)."""
    M, H, E, k, I, SI = 4, 256, 4, 2, 64, 64
    x, layer = synth.make_problem(M, H, E, k, I, SI, seed=7)
    layer.w13_sf.fill_(0x38)
    layer.w2_sf.fill_(0x38)
    layer.w13_gs.fill_(1.0)
    layer.w2_gs.fill_(1.0)
    r = oracle.forward(x, layer, k, intermediates=True)
    xf = torch.from_numpy(bf16_bits_to_f64(tensor_bits(x)))
    same = []
    for t in range(M):
        for j in range(k):
            e = int(r["ids"][t, j])
            lo = (layer.w13[e] & 15).long()
            hi = (layer.w13[e] >> 4).long()
            codes = torch.stack([lo, hi], -1).reshape(2 * I, H).numpy()
            w = torch.from_numpy(e2m1_decode(codes))
            gu = torch.matmul(w, xf[t])
            g, u = gu[:I], gu[I:]
            act = (g / (1 + torch.exp(-g)) * u).float().to(torch.bfloat16)
            got = torch.from_numpy(r["act"][t, j].view(np.int16)).view(torch.bfloat16)
            diff = (got.float() - act.float()).abs()
            assert (diff <= act.float().abs() * 2 ** -7 + 1e-30).all()  # <= 1 bf16 ulp
            same.append((got == act).float())
    # act differs only where fp32 rounding of g, u or the sigmoid meets a bf16
    # midpoint
    assert torch.cat(same).mean() > 0.97


def test_token_permutation_and_sampling(tiny):
    """Tokens are independent: permuting rows permutes outputs bitwise, and a
    sampled token list reproduces the matching rows."""
    x, layer, k = tiny
    full = oracle.forward(x, layer, k)
    perm = torch.randperm(x.shape[0], generator=torch.Generator().manual_seed(1))
    pr = oracle.forward(x[perm].contiguous(), layer, k)
    assert np.array_equal(pr["out"], full["out"][perm.numpy()])
    assert np.array_equal(pr["ids"], full["ids"][perm.numpy()])
    sub = [5, 0, 9]
    sr = oracle.forward(x, layer, k, tokens=sub)
    assert np.array_equal(sr["out"], full["out"][sub])


def test_golden_tiny_regression():
    """The stored tiny-layer outputs (written by tests/golden/make_golden.py,
    which calls only the oracle) still reproduce bit for bit."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_seed0.json")
    with open(path) as f:
        gold = json.load(f)
    M, H, E, k, I, SI = gold["shape"]
    x, layer = synth.make_problem(M, H, E, k, I, SI, seed=gold["seed"])
    r = oracle.forward(x, layer, k)
    assert r["ids"].tolist() == gold["ids"]
    assert r["tw"].tolist() == gold["tw"]
    assert r["out"].astype(int).tolist() == gold["out_bf16_bits"]


def test_shared_silu_is_the_division_form():
    """The shared expert's SiLU is v / (1 + exp(-v)), not v * sigmoid(v):
    the two fp32 forms differ in the last bit for some v, and for
    (gS, uS) = (0.78515625, 0.87109375) that bit decides the BF16 rounding of
    silu(gS) * uS.  x is one-hot in column 0 and the shared rows carry gS and
    uS in column 0, so gS and uS are exact; the expected bits come from
    numpy's fp32 arithmetic with exp taken in float64 and rounded once."""
    M, H, E, k, I, SI = 1, 128, 4, 1, 128, 128
    x, layer = synth.make_problem(M, H, E, k, I, SI, seed=3)
    x.zero_()
    x[0, 0] = 1.0
    rng = np.random.default_rng(11)
    g = rng.uniform(-4, 4, SI).astype(np.float32)
    u = rng.uniform(-2, 2, SI).astype(np.float32)
    g[0], u[0] = 0.78515625, 0.87109375      # the forms round apart here
    g[1], u[1] = 0.78515625, 0.0272216796875  # and here
    gb = torch.from_numpy(g).to(torch.bfloat16)
    ub = torch.from_numpy(u).to(torch.bfloat16)
    gu = torch.zeros(2 * SI, H, dtype=torch.bfloat16)
    gu[:SI, 0], gu[SI:, 0] = gb, ub
    layer.shared_gu = gu
    r = oracle.forward(x, layer, k, intermediates=True)
    gv, uv = gb.float().numpy(), ub.float().numpy()
    e = np.exp(-gv.astype(np.float64)).astype(np.float32)
    den = (np.float32(1) + e).astype(np.float32)
    div = (gv / den).astype(np.float32)
    mul = (gv * (np.float32(1) / den).astype(np.float32)).astype(np.float32)

    def bf16_bits(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    want_div = bf16_bits((div * uv).astype(np.float32))
    want_mul = bf16_bits((mul * uv).astype(np.float32))
    assert (want_div[:2] != want_mul[:2]).all()  # the constructed rows separate the forms
    assert np.array_equal(r["sact"][0], want_div)


# ------------------------------------------------------------ add-RMSNorm
def _bf16(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def _norm_inputs(M, H, seed):
    g = torch.Generator().manual_seed(seed)
    a = torch.randn(M, H, generator=g).to(torch.bfloat16)
    r = (torch.randn(M, H, generator=g) * 2).to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
    return a, r, w


def test_add_rms_norm_residual_is_the_bf16_sum():
    """residual' = bf16(a + r) with the sum in fp32: torch's fp32 add and
    bf16 cast (library)."""
    a, r, w = _norm_inputs(7, 384, 1)
    res, _ = oracle.add_rms_norm(a, r, w, 1e-6)
    assert np.array_equal(res, _bf16(a.float() + r.float()))


def test_add_rms_norm_matches_float64():
    """xn against an independent float64 derivation (one rounding, to bf16,
    at the end), within the parity rule."""
    a, r, w = _norm_inputs(16, 2048, 2)
    _, xn = oracle.add_rms_norm(a, r, w, 1e-6)
    s = a.double() + r.double()
    inv = 1.0 / torch.sqrt((s * s).mean(dim=1, keepdim=True) + 1e-6)
    want = _bf16(s * inv * w.double())
    st = check_bf16(xn, want)
    assert st["n_exact"] > 0.95 * st["n"]


def test_add_rms_norm_closed_forms():
    """Constant rows c (r = 0, w = 1, eps = 0) normalise to sign(c) exactly;
    w = 2 doubles every output and scaling a, r by 2 changes nothing (both
    exact in binary floating point)."""
    H = 256
    c = torch.tensor([1.5, -3.0, 0.25, -0.75]).repeat_interleave(H).reshape(4, H)
    a = c.to(torch.bfloat16)
    z = torch.zeros_like(a)
    one = torch.ones(H, dtype=torch.bfloat16)
    _, xn = oracle.add_rms_norm(a, z, one, 0.0)
    assert np.array_equal(bits_to_f64(xn), np.sign(c.numpy()).astype(np.float64))
    a2, r2, w2 = _norm_inputs(5, 512, 3)
    _, x1 = oracle.add_rms_norm(a2, r2, w2, 0.0)
    _, x2 = oracle.add_rms_norm((a2.float() * 2).to(torch.bfloat16), (r2.float() * 2).to(torch.bfloat16), w2, 0.0)
    assert np.array_equal(x1, x2)
    _, x3 = oracle.add_rms_norm(a2, r2, (w2.float() * 2).to(torch.bfloat16), 0.0)
    assert np.array_equal(bits_to_f64(x3), 2 * bits_to_f64(x1))


def test_add_rms_norm_eps_enters_before_the_root():
    """Zero rows: s = 0 everywhere, v = eps, inv = 1 / sqrt(eps) and xn = 0;
    a row of all-equal 2^-10 with eps = 3 * 2^-20 gives v = 2^-18, so
    inv = 2^9 and xn = 2^-1 exactly (eps added after the mean)."""
    H = 128
    z = torch.zeros(1, H, dtype=torch.bfloat16)
    one = torch.ones(H, dtype=torch.bfloat16)
    _, xn = oracle.add_rms_norm(z, z, one, 1e-5)
    assert (bits_to_f64(xn) == 0).all()
    a = torch.full((1, H), 2.0 ** -10).to(torch.bfloat16)
    _, xn = oracle.add_rms_norm(a, z, one, 3 * 2.0 ** -20)
    assert (bits_to_f64(xn) == 0.5).all()


# ------------------------------------------------- BF16 routed experts (R9)
def _bf16_layer_from_nvfp4(layer, gs_log2: int):
    """BF16 expert weights equal to the NVFP4 ones times 2^gs_log2 (exact in
    bf16: an e2m1 x e4m3 product has at most 6 significant bits)."""
    E, I, H = layer.E, layer.I, layer.H
    d13 = oracle.nvfp4_dequant(layer.w13.reshape(E * 2 * I, H // 2), layer.w13_sf.reshape(E * 2 * I, H // 16), H)
    d2 = oracle.nvfp4_dequant(layer.w2.reshape(E * H, I // 2), layer.w2_sf.reshape(E * H, I // 16), I)
    s = 2.0 ** gs_log2
    w13 = torch.from_numpy((d13 * s).astype(np.float32)).reshape(E, 2 * I, H).to(torch.bfloat16)
    w2 = torch.from_numpy((d2 * s).astype(np.float32)).reshape(E, H, I).to(torch.bfloat16)
    assert torch.equal(w13.float(), torch.from_numpy((d13 * s).astype(np.float32)).reshape(E, 2 * I, H))
    return w13, w2


def test_bf16_experts_reduce_to_nvfp4_with_power_of_two_scales():
    """With every global scale 2^-9, the NVFP4 block scales the accumulator
    by an exact power of two, so BF16 experts holding the dequantised weights
    times 2^-9 give the same g, u, act, y and outputs bit for bit (shared
    output = the NVFP4 oracle's ys)."""
    M, H, E, k, I, SI = 6, 256, 8, 3, 128, 128
    x, layer = synth.make_problem(M, H, E, k, I, SI, seed=21)
    layer.w13_gs.fill_(2.0 ** -9)
    layer.w2_gs.fill_(2.0 ** -9)
    r4 = oracle.forward(x, layer, k, intermediates=True)
    w13, w2 = _bf16_layer_from_nvfp4(layer, -9)
    ys = torch.from_numpy(r4["ys"].view(np.int16)).view(torch.bfloat16)
    rb = oracle.forward_bf16(x, layer.router_w, w13, w2, k, shared_out=ys, intermediates=True)
    assert np.array_equal(rb["ids"], r4["ids"]) and np.array_equal(rb["tw"], r4["tw"])
    assert np.array_equal(rb["act"], r4["act"])
    assert np.array_equal(rb["y"], r4["y"])
    assert np.array_equal(rb["out"], r4["out"])


def test_bf16_experts_match_float64():
    """An independent float64 derivation (torch matmuls on the bf16 weights,
    the stated BF16 roundings), within the rule; the shared output enters
    as given."""
    M, H, E, k, I = 5, 256, 8, 2, 128
    g = torch.Generator().manual_seed(4)
    x = torch.randn(M, H, generator=g).to(torch.bfloat16)
    wr = (torch.randn(E, H, generator=g) * H ** -0.5).to(torch.bfloat16)
    w13 = (torch.randn(E, 2 * I, H, generator=g) * 0.05).to(torch.bfloat16)
    w2 = (torch.randn(E, H, I, generator=g) * 0.05).to(torch.bfloat16)
    sh = (torch.randn(M, H, generator=g) * 0.1).to(torch.bfloat16)
    r = oracle.forward_bf16(x, wr, w13, w2, k, shared_out=sh)
    xf = x.double()
    want = np.empty((M, H), np.uint16)
    for t in range(M):
        R = torch.zeros(H, dtype=torch.float64)
        for j in range(k):
            e = int(r["ids"][t, j])
            gu = w13[e].double() @ xf[t]
            gg, uu = gu[:I], gu[I:]
            act = (gg / (1 + torch.exp(-gg)) * uu).float().to(torch.bfloat16).double()
            y = (w2[e].double() @ act).float().to(torch.bfloat16).double()
            R += float(r["tw"][t, j]) * y
        Rb = R.float().to(torch.bfloat16).double()
        want[t] = _bf16((Rb + sh[t].double()).float())
    st = check_bf16(r["out"], want)
    assert st["n_exact"] > 0.95 * st["n"]


# ------------------------------------------------ NVFP4 shared expert (R10)
def test_nvfp4_shared_expert_is_a_routed_expert_of_weight_one():
    """The NVFP4 shared expert follows the routed rule: a layer whose only
    routed expert (E = 1, top_k = 1, so tw = 1 and bf16(R) = y) holds the
    same NVFP4 weights and global scales gives ys = y and sact = act, bit
    for bit."""
    M, H, I = 5, 256, 128
    x, layer = synth.make_problem(M, H, 1, 1, I, 0, seed=8)
    r = oracle.forward(x, layer, 1, intermediates=True)
    assert (r["tw"] == 1.0).all()
    ys, sact = oracle.shared_nvfp4(x, layer.w13[0], layer.w13_sf[0], float(layer.w13_gs[0]),
                                   layer.w2[0], layer.w2_sf[0], float(layer.w2_gs[0]))
    assert np.array_equal(ys, r["y"][:, 0, :])
    assert np.array_equal(sact, r["act"][:, 0, :])
    assert np.array_equal(ys, r["out"])  # bf16(bf16(y) + 0) = y


# ------------------------------------------------- fused decode qkv (R11)
def _qkv_problem(M=3, H=256, nq=2, nkv=1, nvfp4=True, seed=5, residual=True, rope=True):
    g = torch.Generator().manual_seed(seed)
    N = (nq + 2 * nkv) * 128
    x = synth.make_x(M, H, g)
    res = synth.make_x(M, H, g) if residual else None
    nw = (1 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
    w = torch.randn(N, H, generator=g) * 0.05
    if nvfp4:
        codes, sf, gs = synth.quantize_nvfp4(w)
        weight, scale, gsv = codes, sf, float(gs)
    else:
        weight, scale, gsv = w.to(torch.bfloat16), None, None
    qn = (1 + 0.1 * torch.randn(128, generator=g)).to(torch.bfloat16)
    kn = (1 + 0.1 * torch.randn(128, generator=g)).to(torch.bfloat16)
    max_pos = 16
    if rope:
        ang = torch.arange(max_pos, dtype=torch.float64)[:, None] * (10000.0 ** (-torch.arange(64) / 64.0))[None, :]
        cs = torch.cat([torch.cos(ang), torch.sin(ang)], dim=1).float().numpy()
    else:
        cs = None
    pos = np.array([3, 0, 11, 7, 1, 2, 5, 9][:M], np.int64)
    return dict(x=x, residual=res, norm_w=nw, eps=1e-6, weight=weight, weight_scale=scale, global_scale=gsv,
                q_norm_w=qn, k_norm_w=kn, qk_eps=1e-6, cos_sin=cs, positions=pos, nq=nq, nkv=nkv)


def _caches(nkv=1, blocks=4, bs=4):
    k = np.full((blocks, bs, nkv, 128), 0x7FC1, np.uint16)  # NaN marker: untouched
    return k, k.copy()


def _run_qkv(p, slots, blocks=4, bs=4, **over):
    q = dict(p, **over)
    kc, vc = _caches(q["nkv"], blocks, bs)
    assert kc.shape[2] == q["nkv"]
    out = oracle.qkv_fused(q["x"], q["residual"], q["norm_w"], q["eps"], q["weight"], q["weight_scale"],
                           q["global_scale"], q["q_norm_w"], q["k_norm_w"], q["qk_eps"], q["cos_sin"],
                           q["positions"], kc, vc, np.asarray(slots, np.int64), q["nq"], q["nkv"])
    return out, kc, vc


def test_qkv_input_norm_is_the_add_rms_norm():
    """xn and residual' equal the add-RMSNorm oracle's (itself pinned); with
    no residual xn is the RMSNorm of x, i.e. add_rms_norm(x, 0)."""
    p = _qkv_problem()
    (q, res, xn, qkv), _, _ = _run_qkv(p, [0, 1, 2])
    r_ref, xn_ref = oracle.add_rms_norm(p["x"], p["residual"], p["norm_w"], p["eps"])
    assert np.array_equal(res, r_ref) and np.array_equal(xn, xn_ref)
    p0 = _qkv_problem(residual=False)
    (q0, res0, xn0, _), _, _ = _run_qkv(p0, [0, 1, 2])
    assert res0 is None
    _, xn0_ref = oracle.add_rms_norm(p0["x"], torch.zeros_like(p0["x"]), p0["norm_w"], p0["eps"])
    assert np.array_equal(xn0, xn0_ref)


@pytest.mark.parametrize("nvfp4", [True, False])
def test_qkv_gemv_is_the_exact_dot(nvfp4):
    """qkv = bf16(fp32(exact dot) * gs): with the weights decoded by torch
    (float8 scales, the e2m1 embedding) and a float64 matmul, whose sums of
    these few-bit products are exact, the values agree bit for bit."""
    p = _qkv_problem(nvfp4=nvfp4)
    (q, res, xn, qkv), _, _ = _run_qkv(p, [0, 1, 2])
    xn64 = bf16_bits_to_f64(xn)
    if nvfp4:
        N, H = p["weight"].shape[0], p["x"].shape[1]
        w64 = dequant(p["weight"].numpy(), p["weight_scale"].numpy())
        acc = (xn64 @ w64.T).astype(np.float32) * np.float32(p["global_scale"])
    else:
        w64 = bf16_bits_to_f64(tensor_bits(p["weight"]))
        acc = (xn64 @ w64.T).astype(np.float32)
    assert np.array_equal(qkv, tensor_bits(torch.from_numpy(acc).to(torch.bfloat16)))


def test_qkv_rope_identity_and_quarter_turn():
    """NeoX RoPE on closed forms: a table with cos = 1, sin = 0 gives the
    output without RoPE; cos = 0, sin = 1 (a quarter turn) gives
    o[d] = -n[d + 64], o[d + 64] = n[d] exactly (pairs d, d + 64, signs)."""
    p = _qkv_problem(rope=False)
    (q_plain, _, _, _), k_plain, _ = _run_qkv(p, [0, 1, 2])
    ident = np.concatenate([np.ones((16, 64)), np.zeros((16, 64))], axis=1).astype(np.float32)
    (q_id, _, _, _), k_id, _ = _run_qkv(p, [0, 1, 2], cos_sin=ident)
    assert np.array_equal(q_id, q_plain) and np.array_equal(k_id, k_plain)
    quarter = np.concatenate([np.zeros((16, 64)), np.ones((16, 64))], axis=1).astype(np.float32)
    (q_qt, _, _, _), k_qt, _ = _run_qkv(p, [0, 1, 2], cos_sin=quarter)
    M, nq = q_plain.shape[0], p["nq"]
    a = q_plain.reshape(M, nq, 128)
    b = q_qt.reshape(M, nq, 128)
    assert np.array_equal(b[..., 64:], a[..., :64])
    assert np.array_equal(b[..., :64], a[..., 64:] ^ np.uint16(0x8000))  # -n: the sign bit


def test_qkv_head_norm_closed_forms():
    """A head whose 128 values are equal normalises to sign * w exactly (eps
    0); doubling the q rows of the weight changes no q output (the norm is
    scale-free in binary floating point)."""
    p = _qkv_problem(nvfp4=False, rope=False, M=2)
    w = p["weight"].clone()
    w[:128] = w[0]  # q head 0: every row alike, so every value alike
    (q, _, _, qkv), _, _ = _run_qkv(p, [0, 1], weight=w, qk_eps=0.0)
    qn = bf16_bits_to_f64(tensor_bits(p["q_norm_w"]))
    for t in range(2):
        c = bf16_bits_to_f64(qkv[t, 0])
        assert np.all(bf16_bits_to_f64(qkv[t, :128]) == c) and c != 0
        assert np.array_equal(bf16_bits_to_f64(q[t, :128]), np.sign(c) * qn)
    w2 = p["weight"].clone()
    w2[:256] = (w2[:256].float() * 2).to(torch.bfloat16)  # both q heads, exactly doubled
    (q2, _, _, _), _, _ = _run_qkv(p, [0, 1], weight=w2, qk_eps=0.0)
    (q1, _, _, _), _, _ = _run_qkv(p, [0, 1], qk_eps=0.0)
    assert np.array_equal(q2, q1)


def test_qkv_cache_slots():
    """Brute force over the paged layout: token t's k and v land at block
    slot // block_size, offset slot % block_size; a negative slot and the
    tokens past the mapping's length write nothing; v is the qkv values."""
    p = _qkv_problem(M=3, nkv=2, rope=False)
    (q, _, _, qkv), kc, vc = _run_qkv(p, [6, -1], blocks=4, bs=4)
    (q_all, _, _, _), kc_all, _ = _run_qkv(p, [6, 1, 13], blocks=4, bs=4)
    written = ~np.all(kc == 0x7FC1, axis=-1)
    # slot 6 -> block 1, offset 2, both kv heads
    assert written.sum() == 2 and written[1, 2, 0] and written[1, 2, 1]
    assert np.array_equal(vc[1, 2, 0], qkv[0, 512:640]) and np.array_equal(vc[1, 2, 1], qkv[0, 640:768])
    assert not np.array_equal(kc[1, 2, 0], kc[1, 2, 1])
    assert np.array_equal(kc_all[1, 2], kc[1, 2])
    assert np.all(kc_all[0, 1] != 0x7FC1) and np.all(kc_all[3, 1] != 0x7FC1)
    # without RoPE the cached k is the normalised k head, as q is for q heads
    assert np.array_equal(q, q_all)


def test_qkv_matches_float64():
    """An independent float64 derivation of the whole chain (torch decode of
    the weights, float64 sums and sqrt, the stated roundings), within the
    rule; q and the cached k and v."""
    p = _qkv_problem(M=3, nq=2, nkv=1)
    (q, res, xn, qkv), kc, vc = _run_qkv(p, [2, 5, 9], blocks=4, bs=4)
    x = bf16_bits_to_f64(tensor_bits(p["x"]))
    r = bf16_bits_to_f64(tensor_bits(p["residual"]))
    s = (x + r).astype(np.float32).astype(np.float64)
    nw = bf16_bits_to_f64(tensor_bits(p["norm_w"]))
    inv = 1.0 / np.sqrt((s * s).sum(1, keepdims=True) / s.shape[1] + p["eps"])
    xn64 = bf16_bits_to_f64(tensor_bits(torch.from_numpy(s * inv * nw).to(torch.bfloat16)))
    H = s.shape[1]
    w64 = dequant(p["weight"].numpy(), p["weight_scale"].numpy()) * p["global_scale"]
    qkv64 = bf16_bits_to_f64(tensor_bits(torch.from_numpy(xn64 @ w64.T).to(torch.bfloat16)))
    cs = p["cos_sin"].astype(np.float64)
    want_q = np.empty_like(q)
    want_k = []
    for t in range(3):
        c, sn = cs[p["positions"][t], :64], cs[p["positions"][t], 64:]
        for hh in range(3):
            v = qkv64[t, hh * 128:(hh + 1) * 128]
            wv = bf16_bits_to_f64(tensor_bits(p["q_norm_w"] if hh < 2 else p["k_norm_w"]))
            n = v / np.sqrt((v * v).mean() + p["qk_eps"]) * wv
            o = np.concatenate([n[:64] * c - n[64:] * sn, n[64:] * c + n[:64] * sn])
            ob = tensor_bits(torch.from_numpy(o).to(torch.bfloat16))
            if hh < 2:
                want_q[t, hh * 128:(hh + 1) * 128] = ob
            else:
                want_k.append(ob)
    st = check_bf16(q, want_q)
    assert st["n_exact"] > 0.9 * st["n"]
    got_k = np.stack([kc[0, 2, 0], kc[1, 1, 0], kc[2, 1, 0]])
    check_bf16(got_k, np.stack(want_k))
    got_v = np.stack([vc[0, 2, 0], vc[1, 1, 0], vc[2, 1, 0]])
    check_bf16(got_v, tensor_bits(torch.from_numpy(qkv64[:, 384:512]).to(torch.bfloat16)))


# ------------------------------------------------------- exact sums (R7)
def test_expert_sums_are_exact_not_sequential():
    """Reading R7 on a constructed row: x = (2^24, 1, -2^24, 0, ...) against
    unit weights.  The exact sum is 1; an fp32 loop in index order would
    lose the 1 (2^24 + 1 rounds to 2^24) and give 0.  So g = u = 1 and act =
    bf16(silu(1) * 1), with silu(1) from float64."""
    M, H, E, k, I, SI = 1, 256, 1, 1, 64, 0
    x, layer = synth.make_problem(M, H, E, k, I, SI, seed=3)
    xv = torch.zeros(M, H)
    xv[0, 0], xv[0, 1], xv[0, 2] = 2.0 ** 24, 1.0, -(2.0 ** 24)
    x = xv.to(torch.bfloat16)
    layer.w13.fill_(0x22)  # two e2m1 codes 2 = 1.0 per byte
    layer.w13_sf.fill_(0x38)  # e4m3 1.0
    layer.w13_gs.fill_(1.0)
    r = oracle.forward(x, layer, k, intermediates=True)
    want = torch.tensor(1.0 / (1.0 + np.exp(-1.0)), dtype=torch.float64).float().to(torch.bfloat16)
    assert np.array_equal(r["act"][0, 0], np.full(I, tensor_bits(want), np.uint16))


def test_router_order_is_the_lane_butterfly():
    """Reading R1 on a constructed row (H = 256: lane l holds the products of
    elements 8 l .. 8 l + 7): lane 0's partial is 2^24, lane 1's 1, lane
    16's -2^24.  The butterfly (offsets 16, 8, 4, 2, 1 as seen from lane 0)
    cancels 2^24 first and keeps the 1: the logit is 1.  A loop in index
    order, or the butterfly run from offset 1 up, loses the 1 and gives 0."""
    H = 256
    x = torch.zeros(1, H)
    w = torch.zeros(1, H)
    x[0, 0], w[0, 0] = 2.0 ** 12, 2.0 ** 12    # lane 0
    x[0, 8], w[0, 8] = 1.0, 1.0                # lane 1
    x[0, 128], w[0, 128] = 2.0 ** 12, -(2.0 ** 12)  # lane 16
    logits, _, _ = oracle.route(x.to(torch.bfloat16), w.to(torch.bfloat16), 1)
    assert bf16_bits_to_f64(logits[0, 0]) == 1.0
