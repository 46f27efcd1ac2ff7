"""Parity of the block-scaled FP4 layer (W4A4: NVFP4 weights and NVFP4
activations on tcgen05 kind::mxf4nvf4), called through the C ABI, with the
fp64 W4A4 oracle (the activation quantizer of oracle.c, the products in
fp64)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from moe_layer_bit_gb300 import workloads as wk
from tests.gpu_helpers import bf16_to_f64, bits, check_layer, numpy_weights, sample_tokens

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from moe_layer_bit_gb300 import _lib, build
    from moe_layer_bit_gb300.layer import W4A4Layer

    build.build()
    _lib.load()

DEV = "cuda"
# the tiny workload's I = 128 is below the W4A4 stage of 256 K elements: its
# W4A4 case keeps T, H, E, k and takes I = 256
TINY = wk.Workload("tiny_w4a4_T16_H256_I256_E8_k2", 16, 256, 256, 8, 2, "weight", 1000)
CASES = {"tiny": (TINY, None), "decode": (wk.by_name("decode"), None), "grouped": (wk.by_name("grouped"), 96),
         "skewed": (wk.by_name("skewed"), 128), "prefill": (wk.by_name("prefill"), 48)}


def _quant_gpu(x: torch.Tensor, rows=None):
    n, K = (len(rows) if rows is not None else x.shape[0]), x.shape[1]
    codes = torch.empty(n, K // 2, dtype=torch.uint8, device=DEV)
    scales = torch.empty(n, K // 16, dtype=torch.uint8, device=DEV)
    src = None if rows is None else torch.as_tensor(rows, dtype=torch.int32, device=DEV)
    _lib.moe_quantize_nvfp4(x.to(DEV), src, n, K, codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


def test_quantizer_bit_exact_with_edge_blocks():
    # random magnitudes over many binades, an all-zero block, blocks below the
    # smallest E4M3 scale, a block saturating the scale, ties of the E2M1 grid
    g = torch.Generator().manual_seed(11)
    x = (torch.randn(96, 512, generator=g) * torch.exp(torch.randn(96, 1, generator=g) * 3)).to(torch.bfloat16)
    x[1, :16] = 0
    x[2, 16:32] = 1e-30
    x[3, 32:48] = 3.0e4
    x[4, :16] = torch.tensor([6, 5, 3.5, 2.5, 1.75, 1.25, .75, .25, -6, -5, -3.5, -2.5, -1.75, -1.25, -.75, -.25])
    codes, scales = _quant_gpu(x)
    rc, rs = orc.quant_nvfp4(x.to(torch.float32).numpy())
    assert np.array_equal(scales, rs)
    assert np.array_equal(codes, rc)
    # the gathered form: row r is row rows[r] of x
    rows = np.array([5, 5, 0, 95, 17], np.int32)
    gc, gs = _quant_gpu(x, rows)
    assert np.array_equal(gc, rc[rows]) and np.array_equal(gs, rs[rows])


def _ulps(x, k):
    # the fp32 value k ulps above (k > 0) or below (k < 0) x > 0
    x = np.float32(x)
    for _ in range(abs(int(k))):
        x = np.nextafter(x, np.float32(np.inf) if k > 0 else np.float32(0), dtype=np.float32)
    return np.float32(x)


def test_fp32_quantizer_bit_exact_around_every_midpoint():
    # fp32 blocks (the precision of h), one block per row: for every E4M3
    # scale s, blocks whose amax 6 e4m3(s) makes s their scale and whose other
    # elements sit on, or 1..3 ulps either side of, an E2M1 midpoint times
    # e4m3(s); then blocks whose amax is 6 x an E4M3 midpoint, or 1..2 ulps
    # either side of it
    e4 = np.array([orc.dec_e4m3(c) for c in range(127)])
    mids = np.array([.25, .75, 1.25, 1.75, 2.5, 3.5, 5.0])
    rng = np.random.default_rng(5)
    rows = []
    for s in range(1, 127):
        d = e4[s]
        for _ in range(4):
            v = np.empty(16, np.float32)
            v[0] = np.float32(6 * d)
            for j in range(1, 16):
                v[j] = _ulps(rng.choice(mids) * d, rng.integers(-3, 4))
            rows.append(v * rng.choice([-1, 1], 16).astype(np.float32))
    for s in range(126):
        for k in (-2, -1, 0, 1, 2):
            a = _ulps(3 * (e4[s] + e4[s + 1]), k)  # 6 x the midpoint, exact in fp32
            v = np.clip(rng.standard_normal(16).astype(np.float32) * np.float32(a / 4), -a, a)
            v[int(rng.integers(16))] = -a if k % 2 else a
            rows.append(v)
    X = torch.from_numpy(np.stack(rows).astype(np.float32))
    n, K = X.shape
    codes = torch.empty(n, K // 2, dtype=torch.uint8, device=DEV)
    scales = torch.empty(n, K // 16, dtype=torch.uint8, device=DEV)
    _lib.moe_quantize_nvfp4_f32(X.to(DEV), None, n, K, codes, scales)
    torch.cuda.synchronize()
    rc, rs = orc.quant_nvfp4(X.numpy())
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def _deq(codes, scales):
    e2m1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])
    v = e2m1[np.stack([codes & 15, codes >> 4], -1).reshape(codes.shape[0], -1)]
    sc = np.array([orc.dec_e4m3(s) for s in range(256)])[scales]
    return v * np.repeat(sc, 16, axis=1)


@pytest.mark.parametrize("T,H,I,E", [(40, 256, 512, 3), (200, 512, 256, 5)])
def test_down_projection_matches_fp64_products(T, H, I, E):
    # the down GEMM alone on random NVFP4 activations and weights: every
    # product is exact, so y differs from the fp64 sum only by fp32 accumulation
    rng = np.random.default_rng(T + E)
    ac = rng.integers(0, 256, (T, I // 2), dtype=np.uint8)
    asc = rng.integers(0x28, 0x40, (T, I // 16), dtype=np.uint8)
    wc = rng.integers(0, 256, (E, H, I // 2), dtype=np.uint8)
    wsc = rng.integers(0x28, 0x40, (E, H, I // 16), dtype=np.uint8)
    gs = rng.uniform(0.5, 2, E).astype(np.float32)
    counts = np.bincount(rng.integers(0, E, T), minlength=E)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    d = _lib.dims(T, H, I, E, 1)
    y = torch.empty(T, H, dtype=torch.float32, device=DEV)
    st = torch.zeros(64, dtype=torch.int32, device=DEV)
    w = [torch.from_numpy(a).to(DEV) for a in (wc, wsc, gs)]
    _lib.moe_debug_w4a4_gemm(1, torch.from_numpy(ac).to(DEV), torch.from_numpy(asc).to(DEV),
                             torch.from_numpy(offs).to(DEV), _lib.w4n(*w), d, y, None, st)
    assert _lib.moe_get_device_status(st) == _lib.MOE_OK
    A = _deq(ac, asc)
    ref = np.empty((T, H))
    for e in range(E):
        W = _deq(wc[e], wsc[e]) * float(gs[e])
        ref[offs[e]:offs[e + 1]] = A[offs[e]:offs[e + 1]] @ W.T
    got = y.cpu().numpy().astype(np.float64)
    # fp32 accumulation of I exact products: relative error ~ sqrt(I) * 2^-24
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 4 * np.sqrt(I) * 2.0 ** -24


@pytest.mark.parametrize("T,H,I,E", [(40, 256, 256, 3), (300, 512, 512, 5)])
def test_gate_up_projection_h_codes(T, H, I, E):
    # the gate_up GEMM alone (ragged expert groups, several token and feature
    # tiles): h = SwiGLU of exact-product sums, quantized.  The kernel's h is
    # fp32 (fp32 accumulation, fast exp): its NVFP4 form may differ from the
    # fp64 one only where h lies within a few ulps of a rounding boundary
    rng = np.random.default_rng(T + I)
    ac = rng.integers(0, 256, (T, H // 2), dtype=np.uint8)
    asc = rng.integers(0x18, 0x28, (T, H // 16), dtype=np.uint8)
    wc = rng.integers(0, 256, (E, 2 * I, H // 2), dtype=np.uint8)
    wsc = rng.integers(0x18, 0x28, (E, 2 * I, H // 16), dtype=np.uint8)
    gs = rng.uniform(0.5, 2, E).astype(np.float32)
    counts = np.bincount(rng.integers(0, E, T), minlength=E)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    hc = torch.empty(T, I // 2, dtype=torch.uint8, device=DEV)
    hs = torch.empty(T, I // 16, dtype=torch.uint8, device=DEV)
    st = torch.zeros(64, dtype=torch.int32, device=DEV)
    w = [torch.from_numpy(a).to(DEV) for a in (wc, wsc, gs)]
    _lib.moe_debug_w4a4_gemm(0, torch.from_numpy(ac).to(DEV), torch.from_numpy(asc).to(DEV),
                             torch.from_numpy(offs).to(DEV), _lib.w4n(*w), _lib.dims(T, H, I, E, 1), hc, hs, st)
    assert _lib.moe_get_device_status(st) == _lib.MOE_OK
    A = _deq(ac, asc)
    h = np.empty((T, I))
    for e in range(E):
        W = _deq(wc[e], wsc[e]) * float(gs[e])
        g = A[offs[e]:offs[e + 1]] @ W[:I].T
        u = A[offs[e]:offs[e + 1]] @ W[I:].T
        h[offs[e]:offs[e + 1]] = g / (1 + np.exp(-g)) * u
    rc, rs = orc.quant_nvfp4(h.astype(np.float32))
    gc, gsc = hc.cpu().numpy(), hs.cpu().numpy()
    assert (gsc != rs).mean() < 2e-3
    nib = lambda c: np.stack([c & 15, c >> 4], -1)
    assert (nib(gc) != nib(rc)).mean() < 2e-3
    # every element of a block below the scale's saturation (amax <= 6 x 448)
    # within one grid step (2 x its scale) of the fp64 h
    got = _deq(gc, gsc)
    step = np.repeat(np.array([orc.dec_e4m3(int(c)) for c in range(256)])[gsc], 16, axis=1) * 2
    inside = np.repeat(np.abs(h).reshape(T, -1, 16).max(-1) <= 6 * 448, 16, axis=1)
    assert inside.mean() > 0.9
    assert np.all((np.abs(got - h) <= step + 1e-6 * np.abs(h))[inside])


@pytest.mark.parametrize("name", list(CASES))
def test_w4a4_layer_parity(name):
    wl, nsample = CASES[name]
    d = wk.generate(wl)
    gu, dn = numpy_weights(d)
    layer = W4A4Layer(d["gu"], d["dn"], wl.H, wl.I, wl.E, wl.k, wl.T, DEV)
    ids = torch.empty(wl.T, wl.k, dtype=torch.int32, device=DEV)
    w = torch.empty(wl.T, wl.k, dtype=torch.float32, device=DEV)
    out = layer.forward(d["x"].to(DEV), d["logits"].to(DEV), topk_ids=ids, topk_w=w)
    out2 = layer.forward(d["x"].to(DEV), d["logits"].to(DEV))
    assert layer.device_status() == _lib.MOE_OK
    assert np.array_equal(bits(out), bits(out2)), "W4A4 layer output not deterministic"
    rids, rw = orc.route(d["logits"].numpy(), wl.k)
    assert np.array_equal(ids.cpu().numpy(), rids)
    assert np.abs(w.cpu().numpy() - rw).max() <= 2e-6
    if nsample is None:
        rows = np.arange(wl.T, dtype=np.int32)
    else:
        rows = sample_tokens(rids, wl.E, nsample, seed=13, tile=128, seams=nsample // 2)
    ref = orc.w4a4_layer_rows(bits(d["x"]), rids, rw, gu, dn, rows)
    check_layer(bits(out)[rows], ref, f"W4A4 {name}")


@pytest.mark.parametrize("T,H,I,E,k", [
    (1, 256, 256, 4, 2),        # one token: 32-row token tiles with one valid row; one K stage per tile
    (37, 512, 512, 5, 5),       # k = E, ragged T: every expert holds all 37 tokens (128-row tiles)
    (64, 256, 768, 1, 1),       # one dense expert; down K = 768 (three stages)
    (300, 1024, 256, 64, 4),    # 64-row tiles, ragged groups, experts without tokens
    (40, 256, 256, 1024, 32),   # 1024 experts, k = 32: 1-3 rows per expert, a large tile table
])
def test_w4a4_layer_edge_shapes(T, H, I, E, k):
    d = wk.generate_dims(T, H, I, E, k, seed=T + E)
    gu, dn = numpy_weights(d)
    layer = W4A4Layer(d["gu"], d["dn"], H, I, E, k, T, DEV)
    ids = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, dtype=torch.float32, device=DEV)
    out = layer.forward(d["x"].to(DEV), d["logits"].to(DEV), topk_ids=ids, topk_w=w)
    assert layer.device_status() == _lib.MOE_OK
    rids, rw = orc.route(d["logits"].numpy(), k)
    assert np.array_equal(ids.cpu().numpy(), rids)
    ref = orc.w4a4_layer_rows(bits(d["x"]), rids, rw, gu, dn, np.arange(T, dtype=np.int32))
    check_layer(bits(out), ref, f"W4A4 T={T} H={H} I={I} E={E} k={k}")


def test_w4a4_zero_tokens():
    wl = TINY
    d = wk.generate(wl)
    layer = W4A4Layer(d["gu"], d["dn"], wl.H, wl.I, wl.E, wl.k, wl.T, DEV)
    out = layer.forward(d["x"][:0].to(DEV), d["logits"][:0].to(DEV))
    torch.cuda.synchronize()
    assert out.shape == (0, wl.H) and layer.device_status() == _lib.MOE_OK
    assert _lib.moe_w4a4_kernel_launches(_lib.dims(0, wl.H, wl.I, wl.E, wl.k)) == 0


def test_w4a4_rejects_shapes_below_its_stage():
    # I = 128 is below the 256-element K stage: refused before any launch
    d = _lib.dims(16, 256, 128, 8, 2)
    assert _lib.moe_w4a4_workspace_bytes(d) == 0
    z = torch.zeros(16, dtype=torch.uint8, device=DEV)
    wn = _lib.w4n(z, z, z.view(torch.float32))
    with pytest.raises(_lib.MoeError) as exc:
        _lib.moe_layer_forward_w4a4(z, z, wn, wn, d, z, None, None, z, 16)
    assert exc.value.status == _lib.MOE_ERR_UNSUPPORTED_SHAPE


def test_w4a4_profiled_entry_equals_plain_entry():
    wl = TINY
    d = wk.generate(wl)
    layer = W4A4Layer(d["gu"], d["dn"], wl.H, wl.I, wl.E, wl.k, wl.T, DEV)
    x, lg = d["x"].to(DEV), d["logits"].to(DEV)
    ref = layer.forward(x, lg)
    out = torch.empty_like(ref)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in evs:
        e.record()  # torch creates its events lazily; the library records them again
    _lib.moe_layer_forward_w4a4_profiled(x, lg, layer._abi[0], layer._abi[1], _lib.dims(wl.T, wl.H, wl.I, wl.E, wl.k),
                                         out, None, None, layer.ws, layer.ws_bytes, evs)
    torch.cuda.synchronize()
    assert layer.device_status() == _lib.MOE_OK
    assert np.array_equal(bits(out), bits(ref))
    assert evs[0].elapsed_time(evs[5]) > 0
