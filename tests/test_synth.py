"""The synthetic workloads have the shapes and statistics the configurations
ask for."""
from __future__ import annotations

import torch

from nvfp4_w4a16_mixture_gb300 import synth


def test_skew_share():
    """Skewed routing: the 8 most popular experts take about 40% of the
    top-8 assignments (the configuration's target), measured on probe tokens
    independent of the calibration's."""
    E, H, k = 128, 2048, 8
    c = synth.zipf_router_scale(E)
    g = torch.Generator().manual_seed(12345)
    W = (torch.randn(E, H, generator=g) * H ** -0.5 * c[:, None]).to(torch.bfloat16).float()
    x = torch.randn(8192, H, generator=g).to(torch.bfloat16).float()
    ids = (x @ W.T).topk(k, dim=1).indices
    cnt = torch.bincount(ids.flatten(), minlength=E).double()
    top = cnt.sort(descending=True).values
    share8 = float(top[:8].sum() / cnt.sum())
    assert 0.39 <= share8 <= 0.41, share8
    assert float(top[0] / cnt.sum()) <= 0.125  # an expert is chosen at most once per token


def test_config_shapes():
    assert synth.CONFIGS["decode1"] == (1, 2048, 128, 8, 768, 768)
    assert synth.CONFIGS["prefill4096"][0] == 4096
    assert synth.CONFIGS["skew16384"][0] == 16384
    assert synth.CONFIGS["tiny"] == (2, 256, 8, 2, 128, 128)


def test_quantiser_scales_within_e4m3_range():
    gen = torch.Generator().manual_seed(0)
    w = torch.randn(64, 256, generator=gen) * 0.02
    codes, sf, gs = synth.quantize_nvfp4(w)
    f = sf.view(torch.float8_e4m3fn).float()
    assert torch.isfinite(f).all() and float(f.max()) <= 448.0
    assert codes.dtype == torch.uint8 and codes.shape == (64, 128) and sf.shape == (64, 16)
