"""Pins of the seeded input generator and of the algorithmic byte / flop counts."""
import numpy as np
import torch

from moe_layer_bit_gb300 import workloads as wk

_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _deq(c, s, gs):
    lo = (c & 0xF).astype(np.int64)
    hi = (c >> 4).astype(np.int64)
    nib = np.stack([lo, hi], -1).reshape(c.shape[0], -1)
    mag = _GRID[nib & 7] * np.where(nib & 8, -1.0, 1.0)
    sc = torch.from_numpy(s.copy()).view(torch.float8_e4m3fn).double().numpy()
    return mag * np.repeat(sc, 16, axis=1) * gs


def test_quantizer_round_trips_representable_values():
    rng = np.random.default_rng(5)
    N, K = 8, 64
    gs = 0.01
    sc_codes = rng.integers(0x30, 0x70, size=(N, K // 16)).astype(np.uint8)
    sc_codes[0, 0] = 0x7E                               # 448: amax / (6*448) == gs exactly
    sc = torch.from_numpy(sc_codes).view(torch.float8_e4m3fn).double().numpy()
    mags = rng.integers(0, 8, size=(N, K))
    mags[:, ::16] = 7                                   # each block reaches 6 * scale
    sign = rng.integers(0, 2, size=(N, K))
    W = _GRID[mags] * np.where(sign, -1.0, 1.0) * np.repeat(sc, 16, axis=1) * gs
    c, s, g = wk.quantize_nvfp4(torch.from_numpy(W.astype(np.float32)))
    back = _deq(c.numpy(), s.numpy(), g)
    assert np.allclose(back, W.astype(np.float32), rtol=1e-6, atol=0)


def test_quantizer_error_within_half_grid_step():
    g = torch.Generator().manual_seed(9)
    W = torch.randn(32, 256, generator=g) / 16
    c, s, gs = wk.quantize_nvfp4(W)
    back = _deq(c.numpy(), s.numpy(), gs)
    sc = torch.from_numpy(s.numpy().copy()).view(torch.float8_e4m3fn).double().numpy()
    unit = np.repeat(sc, 16, axis=1) * gs                # value of code 1.0 in each block
    a = np.abs(W.numpy()) / unit
    step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    err = np.abs(back - W.numpy()) / unit
    assert np.all(err <= step / 2 + 1e-6)
    # the largest element of the matrix maps to code 6 with the largest scale
    assert float(gs) == float(np.float32(W.abs().max() / (6 * 448)))


def test_zero_matrix_quantises_to_zero_codes():
    c, s, gs = wk.quantize_nvfp4(torch.zeros(4, 32))
    assert gs == 1.0 and c.sum() == 0 and s.sum() == 0


def test_zipf_bias_closed_form_values():
    # 3 ln p_r = -3.6 ln r - 3 ln S with S = sum_{r<=128} r^-1.2 ~= zeta(1.2) - 128^-0.2 / 0.2 ~= 3.698
    b = wk.zipf_bias(128)
    assert abs(b[0] - (-3.9237)) < 1e-3
    assert abs(b[7] - (b[0] - 3.6 * np.log(8))) < 1e-12
    assert abs(b[127] - (b[0] - 3.6 * np.log(128))) < 1e-12
    assert abs(b[127] - (-21.391)) < 1e-3


def test_tiny_workload_shapes_and_determinism():
    wl = wk.by_name("tiny")
    a = wk.generate(wl)
    b = wk.generate(wl)
    assert a["x"].shape == (16, 256) and a["x"].dtype == torch.bfloat16
    assert a["logits"].shape == (16, 8) and a["logits"].dtype == torch.float32
    assert a["gu"][0].shape == (8, 256, 128) and a["gu"][1].shape == (8, 256, 16)
    assert a["dn"][0].shape == (8, 256, 64) and a["dn"][1].shape == (8, 256, 8)
    for k in ("x", "logits"):
        assert torch.equal(a[k], b[k])
    for i in range(3):
        assert torch.equal(a["gu"][i], b["gu"][i]) and torch.equal(a["dn"][i], b["dn"][i])


def test_weight_bytes_match_atlas_article(golden):
    g = dict(golden("atlas_weight_bytes.txt"))
    H, I, E = 2048, 512, 256
    bf16_both = E * 3 * H * I * 2
    nvfp4_gu = E * 2 * I * H * 9 // 16
    nvfp4_both = E * 3 * H * I * 9 // 16
    assert bf16_both == int(g["bf16_both_projections"])
    assert nvfp4_gu == int(g["nvfp4_gate_up_only"])
    assert nvfp4_both == int(g["nvfp4_both_projections"])
    assert round(bf16_both / 1e6) == int(g["article_mb_bf16"])
    assert round(nvfp4_gu / 1e6) == int(g["article_mb_nvfp4"])
    assert round(bf16_both / nvfp4_both, 1) == float(g["article_ratio"])
    counts = np.ones(E)
    assert wk.algorithmic_bytes(800, H, I, E, 8, counts) == nvfp4_both + E * 8 + 800 * H * 4 + 800 * E * 4


def test_flops():
    assert wk.algorithmic_flops(800, 2048, 512, 8) == 40_265_318_400
