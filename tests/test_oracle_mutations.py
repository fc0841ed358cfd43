"""Planted mistakes: each case edits one expression of a copy of the oracle's
C source (a plausible slip: a swapped operand, a wrong constant, a dropped
term), builds the copy and checks that the pin guarding that step fails on
it.  The product path is not involved; everything runs on the CPU."""
from __future__ import annotations

import os

import pytest

import oracle
import test_oracle_pins as pins
from nvfp4_w4a16_mixture_gb300 import synth


def _tiny():
    M, H, E, k, I, SI = synth.CONFIGS["tiny"]
    x, layer = synth.make_problem(16, H, E, k, I, SI, seed=0)
    return x, layer, k


CASES = [
    ("e2m1 nibble order swapped (reading R3)",
     "unsigned code = (k & 1) ? (byte >> 4) : (byte & 15u);",
     "unsigned code = (k & 1) ? (byte & 15u) : (byte >> 4);",
     pins.test_unit_scales_reduce_to_matmul),
    ("router butterfly run from offset 1 up (reading R1)",
     "for (int o = 16; o >= 1; o >>= 1) {",
     "for (int o = 1; o <= 16; o <<= 1) {",
     pins.test_router_order_is_the_lane_butterfly),
    ("e4m3 exponent bias 8 instead of 7",
     "mag = ldexpf(1.0f + (float)m / 8.0f, (int)e - 7);",
     "mag = ldexpf(1.0f + (float)m / 8.0f, (int)e - 8);",
     pins.test_e4m3_decode_matches_torch),
    ("top-k ties to the higher expert index",
     "bf16_order(logit_bits[e]) > bf16_order(logit_bits[best])",
     "bf16_order(logit_bits[e]) >= bf16_order(logit_bits[best])",
     pins.test_topk_signed_zero_and_ties_constructed),
    ("routing weights not renormalised",
     "tw[j] = round_bf16(s[j] / denom);",
     "tw[j] = round_bf16(s[j]);",
     pins.test_routing_weights_renormalise),
    ("expert gate/up summed in an fp32 loop (reading R7)",
     "double sg = 0.0, su = 0.0; /* reading R7 */\n      for (int h = 0; h < H; ++h) {\n"
     "        sg += (double)(nvfp4_deq(c13, s13, r, H, h) * xf[h]);",
     "float sg = 0.0f, su = 0.0f; /* reading R7 */\n      for (int h = 0; h < H; ++h) {\n"
     "        sg += (double)(nvfp4_deq(c13, s13, r, H, h) * xf[h]);",
     pins.test_expert_sums_are_exact_not_sequential),
    ("expert output without its global scale",
     "float y = round_bf16(acc * gs2);",
     "float y = round_bf16(acc);",
     lambda: pins.test_oracle_matches_float64_tiny(_tiny())),
    ("shared SiLU in the product form (reading R5)",
     "sact[r] = round_bf16(silu_div(gS) * uS);",
     "sact[r] = round_bf16(silu_exact(gS) * uS);",
     pins.test_shared_silu_is_the_division_form),
    ("add-RMSNorm eps after the root (reading R8)",
     "    const float v = (float)sq / (float)H + eps;\n    const float inv = (float)(1.0 / sqrt((double)v));\n"
     "    for (int h = 0; h < H; ++h) {\n      const float p = s[h] * inv;",
     "    const float v = (float)sq / (float)H;\n    const float inv = (float)(1.0 / (sqrt((double)v) + eps));\n"
     "    for (int h = 0; h < H; ++h) {\n      const float p = s[h] * inv;",
     pins.test_add_rms_norm_eps_enters_before_the_root),
    ("NVFP4 shared gate/up without its global scale (reading R10)",
     "const float g = (float)sg * sgu_gs, u = (float)su * sgu_gs;",
     "const float g = (float)sg, u = (float)su;",
     pins.test_nvfp4_shared_expert_is_a_routed_expert_of_weight_one),
    ("BF16 expert output not rounded before the combine (reading R9)",
     "const float y = round_bf16((float)sum); /* y_e = bf16(acc) */",
     "const float y = (float)sum;",
     pins.test_bf16_experts_reduce_to_nvfp4_with_power_of_two_scales),
    ("RoPE with the wrong sign (reading R11)",
     "o[d] = nrm[d] * c - nrm[d + D / 2] * sn;",
     "o[d] = nrm[d] * c + nrm[d + D / 2] * sn;",
     pins.test_qkv_rope_identity_and_quarter_turn),
    ("cache offset with the head stride (reading R11)",
     "(slot % block_size) * s1",
     "(slot % block_size) * s2",
     pins.test_qkv_cache_slots),
    ("head norm over 127 values (reading R11)",
     "const float hvar = (float)hs / (float)D + qk_eps;",
     "const float hvar = (float)hs / (float)(D - 1) + qk_eps;",
     pins.test_qkv_head_norm_closed_forms),
]


@pytest.mark.parametrize("name,old,new,pin", CASES, ids=[c[0] for c in CASES])
def test_pin_fails_on_planted_mistake(name, old, new, pin, tmp_path):
    src = oracle.source()
    assert src.count(old) == 1, f"{name}: the edited expression must occur once"
    lib = oracle.build_variant(src.replace(old, new), os.path.join(str(tmp_path), "libvariant.so"))
    pin()  # the pin passes on the oracle itself
    with oracle.using_library(lib):
        with pytest.raises(AssertionError):
            pin()
