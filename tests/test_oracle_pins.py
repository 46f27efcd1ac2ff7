"""Pins of the fp64 oracle against things other than itself.

Every check here compares the oracle with a value the format specification
prints (tests/golden), a library routine (torch float8 / bfloat16 conversion,
numpy stable sort, scipy softmax, torch fp64 matmul), a closed form, or brute
force on tiny inputs.  None of them retypes the oracle's own formula.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

from oracle import oracle as orc
from moe_layer_bit_gb300 import workloads as wk


# ------------------------------------------------------------------ decoders
def test_e2m1_all_codes_match_spec_table(golden):
    rows = golden("e2m1_values.txt")
    assert len(rows) == 16
    for code, val in rows:
        c = int(code, 16)
        got = orc.dec_e2m1(c)
        exp = float(val)
        assert got == exp and math.copysign(1.0, got) == math.copysign(1.0, exp), (c, got, exp)


def test_e4m3_all_256_codes_match_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = orc.dec_e4m3(c)
        if np.isnan(lib[c]):
            assert np.isnan(got), c
        else:
            assert got == lib[c] and math.copysign(1, got) == math.copysign(1, lib[c]), (c, got, lib[c])


def test_e4m3_anchor_codes(golden):
    for code, val in golden("e4m3_anchors.txt"):
        got = orc.dec_e4m3(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), code


def test_e4m3_monotone_and_max():
    vals = [orc.dec_e4m3(c) for c in range(0x7F)]
    assert all(b > a for a, b in zip(vals, vals[1:]))
    assert max(vals) == 448.0 and vals[1] == 2.0 ** -9


def test_bf16_rne_matches_torch_on_fp32_values():
    # fp32-representable inputs: torch's float32 -> bfloat16 conversion is a single RNE rounding.
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),      # bf16 subnormal range
        (rng.uniform(-3.39e38, 3.39e38, 2000)).astype(np.float32),    # near overflow
        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 1.0078125, 3.3895314e38, 3.4e38], np.float32),
    ])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([orc.bf16_rne(float(a)) for a in v], np.uint16)
    mism = np.nonzero(got != ref)[0]
    assert mism.size == 0, [(float(v[i]), hex(got[i]), hex(ref[i])) for i in mism[:5]]


def test_bf16_rne_ties_to_even():
    # 1 + 2^-8 lies exactly between 1 and 1 + 2^-7 -> even (1.0); 1 + 3*2^-8 -> 1 + 2^-6.
    assert orc.bf16_rne(1.0 + 2.0 ** -8) == 0x3F80
    assert orc.bf16_rne(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert orc.bf16_rne(-(1.0 + 2.0 ** -8 + 2.0 ** -30)) == 0xBF81


def test_weight_element_and_row_agree_with_torch_dequant():
    g = torch.Generator().manual_seed(3)
    W = torch.randn(6, 64, generator=g)
    c, s, gs = wk.quantize_nvfp4(W)
    codes = c.numpy()[None]
    scales = s.numpy()[None]
    gsa = np.array([gs], np.float32)
    ref = _torch_dequant(c, s, gs)
    for n in range(6):
        row = orc.decode_row(codes, scales, gsa, 6, 64, 0, n)
        assert np.array_equal(row, ref[n])
        for kk in (0, 1, 15, 16, 63):
            assert orc.weight(codes, scales, gsa, 6, 64, 0, n, kk) == ref[n, kk]


# ----------------------------------------------- independent torch dequant
_E2M1 = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                      -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0], dtype=torch.float64)


def _torch_dequant(codes, scales, gs):
    """codes u8 [N,K/2], scales u8 [N,K/16] -> float64 [N,K] (library decode of E4M3,
    table decode of E2M1, low nibble = even element)."""
    codes = torch.as_tensor(codes)
    scales = torch.as_tensor(scales)
    lo = (codes & 0xF).long()
    hi = (codes >> 4).long()
    nib = torch.stack([lo, hi], dim=-1).reshape(codes.shape[0], -1)
    v = _E2M1[nib]
    sc = scales.contiguous().view(torch.float8_e4m3fn).to(torch.float64)
    return (v * sc.repeat_interleave(16, dim=1) * float(gs)).numpy()


def _dense_ffn(x_bf16, gu, dn, e, I):
    """Dense SwiGLU FFN of expert e in torch fp64, h rounded to bf16 (via an fp32
    value, exact for the products checked below only up to rare double-rounding)."""
    x = x_bf16.to(torch.float64)
    Wgu = torch.from_numpy(_torch_dequant(gu[0][e], gu[1][e], float(gu[2][e])))
    Wd = torch.from_numpy(_torch_dequant(dn[0][e], dn[1][e], float(dn[2][e])))
    g = x @ Wgu[:I].T
    u = x @ Wgu[I:].T
    h = torch.nn.functional.silu(g) * u
    h = h.to(torch.bfloat16).to(torch.float64)
    return h @ Wd.T


def _bits(x_bf16):
    return x_bf16.contiguous().view(torch.int16).numpy().astype(np.uint16)


# ------------------------------------------------------------------- routing
def _brute_route(logits, k):
    ids = np.empty((logits.shape[0], k), np.int64)
    for t in range(logits.shape[0]):
        key = np.where(np.isnan(logits[t]), -np.inf, logits[t]).astype(np.float64)
        order = np.argsort(-key, kind="stable")     # stable: equal keys keep ascending index
        ids[t] = order[:k]
    return ids


def test_route_brute_force_T16_E8():
    rng = np.random.default_rng(11)
    logits = rng.standard_normal((16, 8)).astype(np.float32)
    for k in (1, 2, 3, 8):
        ids, w = orc.route(logits, k)
        ref = _brute_route(logits, k)
        assert np.array_equal(ids, ref)
        sel = np.take_along_axis(logits.astype(np.float64), ref, axis=1)
        assert np.allclose(w, scipy.special.softmax(sel, axis=1), rtol=1e-14, atol=0)
        assert np.allclose(w.sum(1), 1.0, rtol=0, atol=1e-14)
        for t in range(16):
            assert len(set(ids[t])) == k


def test_route_k_equals_E_is_full_softmax():
    rng = np.random.default_rng(12)
    logits = rng.standard_normal((5, 8)).astype(np.float32)
    ids, w = orc.route(logits, 8)
    full = scipy.special.softmax(logits.astype(np.float64), axis=1)
    assert np.allclose(np.take_along_axis(full, ids, axis=1), w, rtol=1e-14, atol=0)


def test_route_ties_go_to_lower_index():
    logits = np.zeros((3, 8), np.float32)
    logits[1, [2, 5, 6]] = 1.0
    logits[2, :] = [0.5, 1.0, 1.0, 0.25, 1.0, 0.0, 0.0, 0.0]
    ids, w = orc.route(logits, 3)
    assert ids[0].tolist() == [0, 1, 2]
    assert ids[1].tolist() == [2, 5, 6]
    assert ids[2].tolist() == [1, 2, 4]
    assert np.allclose(w[0], 1 / 3) and np.allclose(w[2], 1 / 3)


def test_route_nan_is_minus_infinity():
    logits = np.array([[np.nan, 0.5, -1.0, 2.0]], np.float32)
    ids, w = orc.route(logits, 3)
    assert ids[0].tolist() == [3, 1, 2]
    all_nan = np.full((1, 4), np.nan, np.float32)
    ids, w = orc.route(all_nan, 2)
    assert ids[0].tolist() == [0, 1] and np.allclose(w, 0.5)


# --------------------------------------------------------------- permutation
@pytest.mark.parametrize("T,E,k,seed", [(16, 8, 2, 1), (37, 5, 3, 2), (64, 128, 8, 3), (1, 4, 4, 4)])
def test_permute_equals_stable_sort(T, E, k, seed):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, sorted_token, inv_perm = orc.permute(ids, E)
    flat = ids.reshape(-1)
    order = np.argsort(flat, kind="stable")
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and offsets[-1] == T * k
    assert np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(sorted_token, order // k)
    assert np.array_equal(inv_perm[order], np.arange(T * k))
    # every token appears exactly k times
    assert np.array_equal(np.bincount(sorted_token, minlength=T), np.full(T, k))


def test_permute_skewed_routing_has_empty_experts():
    wl = wk.by_name("skewed")
    d = wk.generate(wk.Workload("s", 512, 64, 64, wl.E, wl.k, "zipf", wl.seed), with_weights=False)
    ids, _ = orc.route(d["logits"].numpy(), wl.k)
    counts, offsets, _, _ = orc.permute(ids, wl.E)
    assert (counts == 0).sum() > 10 and counts.sum() == 512 * wl.k


# --------------------------------------------------------------------- layer
def _small_layer(T, H, I, E, k, seed):
    d = wk.generate_dims(T, H, I, E, k, seed)
    gu = tuple(a.numpy() for a in d["gu"])
    dn = tuple(a.numpy() for a in d["dn"])
    return d, gu, dn


def test_single_expert_equals_dense_ffn():
    d, gu, dn = _small_layer(T=8, H=64, I=32, E=1, k=1, seed=21)
    out, ids, w = orc.layer(_bits(d["x"]), d["logits"].numpy(), gu, dn, 1)
    assert np.all(ids == 0) and np.all(w == 1.0)
    ref = _dense_ffn(d["x"], gu, dn, 0, 32).numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_identical_experts_equal_dense_ffn_for_any_routing():
    d, gu, dn = _small_layer(T=12, H=64, I=32, E=4, k=3, seed=22)
    gu = tuple(np.broadcast_to(a[:1], a.shape).copy() for a in gu)
    dn = tuple(np.broadcast_to(a[:1], a.shape).copy() for a in dn)
    out, ids, w = orc.layer(_bits(d["x"]), d["logits"].numpy(), gu, dn, 3)
    ref = _dense_ffn(d["x"], gu, dn, 0, 32).numpy()      # weights sum to 1
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_layer_is_weighted_sum_of_dense_experts():
    d, gu, dn = _small_layer(T=6, H=32, I=16, E=5, k=2, seed=23)
    out, ids, w = orc.layer(_bits(d["x"]), d["logits"].numpy(), gu, dn, 2)
    dense = [_dense_ffn(d["x"], gu, dn, e, 16).numpy() for e in range(5)]
    ref = np.zeros_like(out)
    for t in range(6):
        for j in range(2):
            ref[t] += w[t, j] * dense[ids[t, j]][t]
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_unrouted_experts_contribute_nothing():
    d, gu, dn = _small_layer(T=4, H=32, I=16, E=6, k=2, seed=24)
    logits = d["logits"].numpy().copy()
    logits[:, 3:] -= 100.0                     # experts 3..5 never selected
    out, ids, _ = orc.layer(_bits(d["x"]), logits, gu, dn, 2)
    assert ids.max() < 3
    gu2 = (gu[0].copy(), gu[1].copy(), gu[2].copy())
    dn2 = (dn[0].copy(), dn[1].copy(), dn[2].copy())
    gu2[1][3:] = 0x7F                          # NaN block scales
    dn2[1][3:] = 0x7F
    gu2[2][3:] = np.nan
    out2, _, _ = orc.layer(_bits(d["x"]), logits, gu2, dn2, 2)
    assert np.all(np.isfinite(out2)) and np.array_equal(out, out2)


def test_layer_rows_matches_full_layer():
    d, gu, dn = _small_layer(T=9, H=32, I=16, E=4, k=2, seed=25)
    out, ids, w = orc.layer(_bits(d["x"]), d["logits"].numpy(), gu, dn, 2)
    rows = np.array([8, 0, 4], np.int32)
    sub = orc.layer_rows(_bits(d["x"]), ids, w, gu, dn, rows)
    assert np.array_equal(sub, out[rows])


def test_stage_functions_compose_to_layer():
    d, gu, dn = _small_layer(T=5, H=32, I=16, E=3, k=2, seed=26)
    x = _bits(d["x"])
    out, ids, w = orc.layer(x, d["logits"].numpy(), gu, dn, 2)
    counts, offsets, sorted_token, inv_perm = orc.permute(ids, 3)
    experts = np.repeat(np.arange(3), counts)
    _, h = orc.gate_up_swiglu_rows(x[sorted_token], experts, gu, 16)
    y = orc.down_rows(h, experts, dn, 32)
    ref = np.zeros_like(out)
    for t in range(5):
        for j in range(2):
            ref[t] += w[t, j] * y[inv_perm[t * 2 + j]]
    assert np.array_equal(ref, out)
    assert np.array_equal(orc.combine(y, inv_perm, w), out)


# ------------------------------------------------------------ router logits
def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_router_logits_exact_matches_fp64_matmul():
    g = torch.Generator().manual_seed(11)
    x = torch.randn(7, 384, generator=g).to(torch.bfloat16)
    w = torch.randn(9, 384, generator=g).to(torch.bfloat16)
    b = torch.randn(9, generator=g)
    got = orc.router_logits_exact(_bf16_bits(x), _bf16_bits(w), b.numpy())
    ref = (x.double() @ w.double().T + b.double()[None, :]).numpy()
    assert np.allclose(got, ref, rtol=0, atol=1e-12 * np.abs(ref).max())


def test_router_logits_ordered_within_fp32_bound():
    # each part sums at most 8*ceil(H/256) products with fma (one rounding
    # each), then five pairwise rounds and the bias: first-order bound
    # (n_fma + 6) * 2^-24 * sum |x w| + |bias| 2^-24
    g = torch.Generator().manual_seed(12)
    for H in (128, 256, 2048, 4096):
        x = torch.randn(5, H, generator=g).to(torch.bfloat16)
        w = (torch.randn(6, H, generator=g) / math.sqrt(H)).to(torch.bfloat16)
        b = torch.randn(6, generator=g)
        got = orc.router_logits(_bf16_bits(x), _bf16_bits(w), b.numpy()).astype(np.float64)
        ref = orc.router_logits_exact(_bf16_bits(x), _bf16_bits(w), b.numpy())
        absprod = (x.double().abs() @ w.double().abs().T).numpy()
        n_fma = 8 * ((H + 255) // 256)
        bound = (n_fma + 6) * 2.0 ** -24 * absprod + 2.0 ** -24 * np.abs(b.numpy())[None, :] + 1e-30
        assert np.all(np.abs(got - ref) <= bound), f"H={H}"


def test_router_logits_integer_inputs_are_exact():
    # small integers: every product and partial sum is an exact fp32 integer,
    # so any summation order gives the exact value (a dropped or doubled term
    # would not)
    g = torch.Generator().manual_seed(13)
    x = torch.randint(-8, 9, (4, 512), generator=g).float()
    w = torch.randint(-8, 9, (6, 512), generator=g).float()
    b = torch.randint(-100, 101, (6,), generator=g).float()
    got = orc.router_logits(_bf16_bits(x), _bf16_bits(w), b.numpy())
    assert np.array_equal(got.astype(np.float64), (x.double() @ w.double().T + b.double()).numpy())


def test_router_logits_order_fixture():
    # H = 16: part 0 takes h = 0..7, part 1 takes h = 8..15, the others are 0.
    # x = 1 everywhere; w[0] = 2^24, w[1..15] = 1.
    # part 0: fma gives 2^24, then adding 1 seven times stays at 2^24 (2^24+1
    #         is a tie that rounds to the even 2^24);
    # part 1: 8;  pairwise rounds: part 0 = 2^24 + 8 = 16777224 (exact).
    # (The exact sum 16777231 would round to 16777232; a sequential sum over
    # h stays at 16777216.)  With bias -2^24 the result is exactly 8.
    x = torch.ones(1, 16)
    w = torch.ones(1, 16)
    w[0, 0] = 2.0 ** 24
    got = orc.router_logits(_bf16_bits(x), _bf16_bits(w))
    assert got[0, 0] == np.float32(16777224.0)
    got_b = orc.router_logits(_bf16_bits(x), _bf16_bits(w), np.array([-(2.0 ** 24)], np.float32))
    assert got_b[0, 0] == np.float32(8.0)


# ------------------------------------------------- W4A4 activation quantizer
def _e4m3_values():
    """Values of the non-negative finite E4M3 codes 0x00..0x7E by torch's float8 decode."""
    c = torch.arange(0, 0x7F, dtype=torch.uint8)
    return c.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_rne_matches_torch_float8_conversion():
    # torch's fp32 -> float8_e4m3fn conversion (a library routine, round to
    # nearest even) on random values, exact codes and every midpoint (ties)
    vals = _e4m3_values()
    rng = np.random.default_rng(3)
    xs = list(rng.uniform(0, 448, 3000)) + list(rng.uniform(0, 2 ** -5, 1000)) + list(vals)
    xs += list((vals[1:] + vals[:-1]) / 2)             # ties between neighbours
    xs = np.array(xs, np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_rne(v) for v in xs], np.uint8)
    assert np.array_equal(got, ref)


def test_e2m1_rne_nearest_with_ties_to_even(golden):
    # brute force over the typed OCP E2M1 table: the nearest magnitude, ties to
    # the code with the even mantissa bit, saturating at 6, sign applied
    table = {int(c, 16) if c.startswith("0x") else int(c): float(v) for c, v in golden("e2m1_values.txt")}
    mags = sorted((v, c) for c, v in table.items() if c < 8)
    grid = np.concatenate([np.linspace(-7, 7, 2801), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -5.0, -0.25]])
    for v in grid.astype(np.float32):
        a = min(abs(float(v)), 6.0)
        best = min(mags, key=lambda mc: (abs(mc[0] - a), mc[1] & 1))
        want = best[1] | (8 if (v < 0 and best[1] != 0) else 0)
        assert orc.e2m1_rne(v) == want, (v, orc.e2m1_rne(v), want)


def test_quant_nvfp4_round_trips_representable_blocks():
    # a block whose largest code is 6 and whose scale is an E4M3 value comes
    # back unchanged: amax / 6 is that scale exactly, every element on the grid
    rng = np.random.default_rng(5)
    vals = _e4m3_values()
    e2m1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for _ in range(200):
        s = int(rng.integers(0x08, 0x7E))
        mags = rng.choice(e2m1, 16)
        mags[rng.integers(16)] = 6.0
        sign = rng.choice([-1.0, 1.0], 16)
        v = (sign * mags * vals[s]).astype(np.float32)
        codes, scales = orc.quant_nvfp4(v)
        assert scales[0] == s
        back = _torch_dequant(codes[None], scales[None], 1.0)[0]
        assert np.array_equal(back, v.astype(np.float64))


def test_quant_nvfp4_error_within_half_a_grid_step():
    rng = np.random.default_rng(6)
    v = (rng.standard_normal((64, 256)) * np.exp(rng.uniform(-6, 6, (64, 1)))).astype(np.float32)
    codes, scales = orc.quant_nvfp4(v)
    back = _torch_dequant(codes, scales, 1.0)
    sc = torch.from_numpy(scales).view(torch.float8_e4m3fn).to(torch.float64).numpy().repeat(16, axis=1)
    # the scale is the E4M3 value nearest amax/6; relative to it the grid step
    # is at most 2 (between 4 and 6), and elements beyond 6 * scale saturate
    amax = np.abs(v.reshape(64, 16, 16)).max(axis=2).repeat(16, axis=1)
    assert np.all(np.abs(sc - amax / 6) <= (amax / 6) * 2 ** -4 + 2 ** -10)
    err = np.abs(back - v)
    assert np.all(err <= sc * 1.0 + np.maximum(np.abs(v) - 6 * sc, 0) + 1e-30)


def test_w4a4_single_expert_equals_dense_ffn_on_quantized_activations():
    # E = 1, k = 1: the W4A4 layer equals a torch fp64 SwiGLU FFN on the
    # quantized x, with h rounded to fp32 and quantized by the (pinned)
    # quantizer above
    d, gu, dn = _small_layer(T=6, H=128, I=64, E=1, k=1, seed=23)
    xb = _bits(d["x"])
    ids = np.zeros((6, 1), np.int32)
    w = np.ones((6, 1))
    got = orc.w4a4_layer_rows(xb, ids, w, gu, dn, np.arange(6, dtype=np.int32))
    xc, xs = orc.quant_nvfp4(d["x"].to(torch.float32).numpy())
    xq = torch.from_numpy(_torch_dequant(xc, xs, 1.0))
    Wgu = torch.from_numpy(_torch_dequant(gu[0][0], gu[1][0], float(gu[2][0])))
    Wd = torch.from_numpy(_torch_dequant(dn[0][0], dn[1][0], float(dn[2][0])))
    g, u = xq @ Wgu[:64].T, xq @ Wgu[64:].T
    h = (torch.nn.functional.silu(g) * u).to(torch.float32).numpy()
    hc, hs = orc.quant_nvfp4(h)
    ref = torch.from_numpy(_torch_dequant(hc, hs, 1.0)) @ Wd.T
    assert np.allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_quant_nvfp4_codes_round_the_exact_quotient():
    # brute force in fp64 (exact here): each code is the grid value whose
    # product with the block scale is nearest to the element, ties to the
    # even mantissa; elements on, and one fp32 ulp either side of, the grid
    # midpoints times the scale are included
    vals = _e4m3_values()
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    rng = np.random.default_rng(8)
    for _ in range(100):
        s = int(rng.integers(0x10, 0x70))
        d = vals[s]
        mids = np.array([.25, .75, 1.25, 1.75, 2.5, 3.5, 5.0]) * d
        pick = rng.choice(mids, 15)
        v = np.concatenate([[6 * d], pick * (1 + rng.choice([-1, 0, 1], 15) * 2.0 ** -23)]).astype(np.float32)
        v *= rng.choice([-1, 1], 16).astype(np.float32)
        codes, scales = orc.quant_nvfp4(v)
        assert scales[0] == s
        got = np.stack([codes & 15, codes >> 4], -1).reshape(-1)
        for i, x in enumerate(v.astype(np.float64)):
            dist = np.abs(grid * d - abs(x))
            best = min(range(8), key=lambda c: (dist[c], c & 1))
            want = best | (8 if (x < 0 and best) else 0)
            assert got[i] == want, (s, x, got[i], want)


def test_quant_nvfp4_exact_quotient_equals_fp32_division():
    # the block scale has at most 4 significant bits and every E2M1 midpoint
    # at most 3, so an fp32 quotient never rounds onto a midpoint that the
    # exact quotient misses: both readings give the same codes
    rng = np.random.default_rng(21)
    v = (rng.standard_normal((400, 64)) * np.exp(rng.standard_normal((400, 1)) * 4)).astype(np.float32)
    codes, scales = orc.quant_nvfp4(v)
    got = np.stack([codes & 15, codes >> 4], -1).reshape(400, 64)
    for r in range(0, 400, 7):
        for b in range(4):
            d = np.float32(orc.dec_e4m3(int(scales[r, b])))
            for i in range(16):
                x = v[r, 16 * b + i]
                want = orc.e2m1_rne(float(np.float32(x / d))) if d != 0 else 0
                assert got[r, 16 * b + i] == want
