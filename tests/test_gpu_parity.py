"""Parity of the CUDA path (called through the C ABI) with the fp64 oracle."""
from __future__ import annotations

import functools
import math
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from moe_layer_bit_gb300 import workloads as wk
from tests.gpu_helpers import (bf16_to_f64, bits, check_layer, numpy_weights, sample_tokens, workload_inputs)

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from moe_layer_bit_gb300 import _lib, build
    from moe_layer_bit_gb300.layer import MoELayer, pack_projection

    build.build()
    _lib.load()

DEV = "cuda"
ALL = [w.name.split("_")[0] for w in wk.WORKLOADS]
# the layer at full size is checked on all tokens where the oracle is quick,
# on a stratified token sample otherwise: every expert that has tokens, the
# first and last token of (up to SEAMS of) the experts' 128-row token tiles,
# then random tokens up to the count
LAYER_SAMPLE = {"tiny": None, "decode": None, "grouped": 96, "prefill": 128, "skewed": 256}
SEAMS = {"grouped": 64, "prefill": 128, "skewed": 128}


def _layer_rows(name, rids, E, seed):
    if LAYER_SAMPLE[name] is None:
        return np.arange(rids.shape[0], dtype=np.int32)
    return sample_tokens(rids, E, LAYER_SAMPLE[name], seed=seed, tile=128, seams=SEAMS[name])


def _route_gpu(logits: torch.Tensor, k: int):
    T, E = logits.shape
    d = _lib.dims(T, 128, 64, E, k)
    ids = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, dtype=torch.float32, device=DEV)
    _lib.moe_route_topk(logits.to(DEV), d, ids, w)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


def _permute_gpu(ids: np.ndarray, x: torch.Tensor, E: int, I: int = 64):
    T, k = ids.shape
    H = x.shape[1]
    d = _lib.dims(T, H, I, E, k)
    n = T * k
    ws_bytes = _lib.moe_stage_workspace_bytes(d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    st = torch.empty(max(n, 1), dtype=torch.int32, device=DEV)
    inv = torch.empty(max(n, 1), dtype=torch.int32, device=DEV)
    xp = torch.empty(max(n, 1), H, dtype=torch.bfloat16, device=DEV)
    _lib.moe_permute(torch.from_numpy(ids).to(DEV), x.to(DEV), d, counts, offsets, st, inv, xp, ws, ws_bytes)
    torch.cuda.synchronize()
    return (counts.cpu().numpy(), offsets.cpu().numpy(), st.cpu().numpy()[:n], inv.cpu().numpy()[:n],
            xp[:n])


# ------------------------------------------------------------ dequantiser
def test_dequant_table_bit_exact():
    out = torch.empty(2 * 256 * 16, dtype=torch.int16, device=DEV)
    _lib.moe_debug_dequant_table(out)
    got = bits(out).reshape(2, 256, 16)
    for s in range(256):
        sv = orc.dec_e4m3(s)
        for c in range(16):
            ref = orc.dec_e2m1(c) * sv
            for half in range(2):
                g = bf16_to_f64(got[half, s, c:c + 1])[0]
                if np.isnan(ref):
                    assert np.isnan(g), (half, s, c)
                else:
                    assert g == ref, (half, hex(s), c, g, ref)


# ---------------------------------------------------------------- routing
@pytest.mark.parametrize("name", ALL)
def test_route_parity(name):
    wl = wk.by_name(name)
    d = wk.generate(wl, with_weights=False)
    ids, w = _route_gpu(d["logits"], wl.k)
    rids, rw = orc.route(d["logits"].numpy(), wl.k)
    assert np.array_equal(ids, rids)
    assert np.abs(w - rw).max() <= 2e-6


def test_route_edge_cases():
    logits = torch.zeros(6, 8)
    logits[1, [2, 5, 6]] = 1.0
    logits[2, 0] = float("nan")
    logits[3, :] = float("nan")
    logits[4, [0, 3, 4]] = -0.0            # -0 and +0 tie: the lower index goes first
    logits[5, :] = -float("inf")           # one finite logit among -inf
    logits[5, 6] = 1.0
    for k in (1, 3, 8):
        ids, w = _route_gpu(logits, k)
        rids, rw = orc.route(logits.numpy(), k)
        assert np.array_equal(ids, rids)
        assert np.abs(w - rw).max() <= 2e-6
    # max experts and top-k
    g = torch.Generator().manual_seed(4)
    logits = torch.randn(37, 1024, generator=g)
    ids, w = _route_gpu(logits, 32)
    rids, rw = orc.route(logits.numpy(), 32)
    assert np.array_equal(ids, rids) and np.abs(w - rw).max() <= 2e-6


# ------------------------------------------------------------ router logits
@pytest.mark.parametrize("name", ALL)
def test_router_logits_bit_exact(name):
    wl = wk.by_name(name)
    d = wk.generate(wl, with_weights=False)
    Wr, b = wk.router_weights(wl)
    x = d["x"]
    logits = torch.empty(wl.T, wl.E, dtype=torch.float32, device=DEV)
    _lib.moe_router_logits(x.to(DEV), Wr.to(DEV), b.to(DEV), _lib.dims(wl.T, wl.H, wl.I, wl.E, wl.k), logits)
    got = logits.cpu().numpy()
    rows = np.arange(wl.T) if wl.T <= 1024 else np.random.default_rng(5).choice(wl.T, 512, replace=False)
    ref = orc.router_logits(bits(x)[rows], bits(Wr), b.numpy())
    assert np.array_equal(got[rows].view(np.uint32), ref.view(np.uint32))


def test_router_logits_without_bias_and_ragged_h():
    g = torch.Generator().manual_seed(21)
    for T, H, E in [(3, 128, 5), (17, 384, 70), (1, 65536, 2)]:
        x = torch.randn(T, H, generator=g).to(torch.bfloat16)
        Wr = (torch.randn(E, H, generator=g) / math.sqrt(H)).to(torch.bfloat16)
        logits = torch.empty(T, E, dtype=torch.float32, device=DEV)
        _lib.moe_router_logits(x.to(DEV), Wr.to(DEV), None, _lib.dims(T, H, 64, E, 1), logits)
        ref = orc.router_logits(bits(x), bits(Wr))
        assert np.array_equal(logits.cpu().numpy().view(np.uint32), ref.view(np.uint32)), (T, H, E)


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_layer_with_router_logits(name):
    # the layer computing its own gate logits: logits bit-exact, routing
    # exact, the output identical to the layer fed the same logits, and within
    # tolerance of the oracle layer
    wl, d = workload_inputs(name)
    Wr, b = wk.router_weights(wl)
    layer = _layer(wl, d)
    x = d["x"].to(DEV)
    logits = torch.empty(wl.T, wl.E, dtype=torch.float32, device=DEV)
    ids = torch.empty(wl.T, wl.k, dtype=torch.int32, device=DEV)
    w = torch.empty(wl.T, wl.k, dtype=torch.float32, device=DEV)
    out = layer.forward_router(x, Wr.to(DEV), b.to(DEV), logits_out=logits, topk_ids=ids, topk_w=w)
    assert layer.device_status() == _lib.MOE_OK
    ref_logits = orc.router_logits(bits(d["x"]), bits(Wr), b.numpy())
    assert np.array_equal(logits.cpu().numpy().view(np.uint32), ref_logits.view(np.uint32))
    rids, rw = orc.route(ref_logits, wl.k)
    assert np.array_equal(ids.cpu().numpy(), rids)
    assert np.abs(w.cpu().numpy() - rw).max() <= 2e-6
    out2 = layer.forward(x, torch.from_numpy(ref_logits).to(DEV))
    assert np.array_equal(bits(out), bits(out2))
    gu, dn = numpy_weights(d)
    ref = orc.layer_rows(bits(d["x"]), rids, rw, gu, dn, np.arange(wl.T, dtype=np.int32))
    check_layer(bits(out), ref, f"{name} with router")


# ------------------------------------------------------------ shared expert
@pytest.mark.parametrize("name", ["tiny", "decode", "grouped", "skewed"])
def test_layer_with_shared_expert(name):
    # routed output plus a shared expert every token uses (weight 1), in the
    # same grouped launches; gate logits given
    wl, d = workload_inputs(name)
    sgu, sdn = wk.shared_expert(wl)
    gu, dn = numpy_weights(d)
    layer = MoELayer(d["gu"], d["dn"], wl.H, wl.I, wl.E, wl.k, wl.T, DEV, shared=(sgu, sdn))
    ids = torch.empty(wl.T, wl.k, dtype=torch.int32, device=DEV)
    w = torch.empty(wl.T, wl.k, dtype=torch.float32, device=DEV)
    out = layer.forward_shared(d["x"].to(DEV), logits=d["logits"].to(DEV), topk_ids=ids, topk_w=w)
    out2 = layer.forward_shared(d["x"].to(DEV), logits=d["logits"].to(DEV))
    assert layer.device_status() == _lib.MOE_OK
    assert np.array_equal(bits(out), bits(out2)), "not deterministic"
    rids, rw = orc.route(d["logits"].numpy(), wl.k)
    assert np.array_equal(ids.cpu().numpy(), rids)
    rows = _layer_rows(name, rids, wl.E, seed=9)
    sgu_np = tuple(a.numpy() for a in sgu)
    sdn_np = tuple(a.numpy() for a in sdn)
    ref = orc.layer_rows(bits(d["x"]), rids, rw, gu, dn, rows) + orc.shared_rows(bits(d["x"]), sgu_np, sdn_np, rows)
    check_layer(bits(out)[rows], ref, f"{name} + shared expert")


def test_layer_with_shared_expert_and_router():
    # logits from router weights and a shared expert, in one call
    wl, d = workload_inputs("decode")
    sgu, sdn = wk.shared_expert(wl)
    Wr, b = wk.router_weights(wl)
    gu, dn = numpy_weights(d)
    layer = MoELayer(d["gu"], d["dn"], wl.H, wl.I, wl.E, wl.k, wl.T, DEV, shared=(sgu, sdn))
    logits = torch.empty(wl.T, wl.E, dtype=torch.float32, device=DEV)
    out = layer.forward_shared(d["x"].to(DEV), router_weight=Wr.to(DEV), router_bias=b.to(DEV), logits_out=logits)
    assert layer.device_status() == _lib.MOE_OK
    ref_logits = orc.router_logits(bits(d["x"]), bits(Wr), b.numpy())
    assert np.array_equal(logits.cpu().numpy().view(np.uint32), ref_logits.view(np.uint32))
    rids, rw = orc.route(ref_logits, wl.k)
    rows = np.arange(wl.T, dtype=np.int32)
    ref = orc.layer_rows(bits(d["x"]), rids, rw, gu, dn, rows) + orc.shared_rows(
        bits(d["x"]), tuple(a.numpy() for a in sgu), tuple(a.numpy() for a in sdn), rows)
    check_layer(bits(out), ref, "decode + router + shared expert")


# ------------------------------------------------------------ permutation
@pytest.mark.parametrize("name", ALL)
def test_permute_parity_and_determinism(name):
    wl = wk.by_name(name)
    d = wk.generate(wl, with_weights=False)
    rids, _ = orc.route(d["logits"].numpy(), wl.k)
    x = d["x"]
    ref = orc.permute(rids, wl.E)
    a = _permute_gpu(rids, x, wl.E)
    b = _permute_gpu(rids, x, wl.E)
    for i, nm in enumerate(["counts", "offsets", "sorted_token", "inv_perm"]):
        assert np.array_equal(a[i], ref[i]), nm
        assert np.array_equal(a[i], b[i]), nm
    xp = bits(a[4])
    assert np.array_equal(xp, bits(x)[ref[2]])
    assert np.array_equal(xp, bits(b[4]))


@pytest.mark.parametrize("T,E,k", [(1, 4, 1), (3, 8, 8), (37, 5, 3), (1100, 16, 4), (2049, 1024, 32)])
def test_permute_ragged_shapes(T, E, k):
    rng = np.random.default_rng(T)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    x = torch.randn(T, 128).to(torch.bfloat16)
    got = _permute_gpu(ids, x, E)
    ref = orc.permute(ids, E)
    for i in range(4):
        assert np.array_equal(got[i], ref[i])
    assert np.array_equal(bits(got[4]), bits(x)[ref[2]])


# ------------------------------------------------------- GEMM stages
def _stage_setup(name):
    wl, d = workload_inputs(name)
    gu, dn = numpy_weights(d)
    rids, rw = orc.route(d["logits"].numpy(), wl.k)
    counts, offsets, st, inv = orc.permute(rids, wl.E)
    x_perm = d["x"][torch.from_numpy(st.astype(np.int64))].contiguous()
    experts = np.repeat(np.arange(wl.E), counts)
    return wl, d, gu, dn, rids, rw, counts, offsets, st, inv, x_perm, experts


def _rows_for(name, n_rows, counts, offsets, seed=0):
    if LAYER_SAMPLE[name] is None:
        return np.arange(n_rows)
    rng = np.random.default_rng(seed)
    rows = set()
    for e in np.nonzero(counts)[0]:          # first and last row of every non-empty expert
        rows.add(int(offsets[e]))
        rows.add(int(offsets[e + 1] - 1))
    rows.update(int(r) for r in rng.choice(n_rows, size=min(n_rows, 64), replace=False))
    if len(rows) > 400:
        rows = set(sorted(rows)[:: max(1, len(rows) // 400)])
    return np.array(sorted(rows))


@pytest.mark.parametrize("name", ALL)
def test_gate_up_down_stages(name):
    wl, d, gu, dn, rids, rw, counts, offsets, st, inv, x_perm, experts = _stage_setup(name)
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    dims = _lib.dims(T, H, I, E, k)
    wgu = pack_projection(*d["gu"], _lib.MOE_PROJ_GATE_UP, DEV)
    wdn = pack_projection(*d["dn"], _lib.MOE_PROJ_DOWN, DEV)
    ws_bytes = _lib.moe_stage_workspace_bytes(dims)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=DEV)
    offs = torch.from_numpy(offsets).to(DEV)
    h = torch.empty(T * k, I, dtype=torch.bfloat16, device=DEV)
    y = torch.empty(T * k, H, dtype=torch.float32, device=DEV)
    _lib.moe_w4a16_gate_up_swiglu(x_perm.to(DEV), offs, wgu.abi, dims, h, ws, ws_bytes)
    _lib.moe_w4a16_down(h, offs, wdn.abi, dims, y, ws, ws_bytes)
    assert _lib.moe_get_device_status(ws) == _lib.MOE_OK
    rows = _rows_for(name, T * k, counts, offsets)
    xb = bits(x_perm)[rows]
    h_exact, h_ref = orc.gate_up_swiglu_rows(xb, experts[rows], gu, I)
    h_gpu = bits(h)[rows]
    # h: the GPU rounds fp32 silu(g)*u to bf16, the oracle rounds the fp64 value;
    # they may differ by one bf16 ulp where the value sits on a rounding edge.
    hg = bf16_to_f64(h_gpu)
    scale = np.sqrt(np.mean(h_exact ** 2))
    err = np.abs(hg - h_exact)
    assert np.all(err <= 2 ** -8 * np.abs(h_exact) + 1e-4 * scale), float((err / (np.abs(h_exact) + scale)).max())
    mism = np.mean(h_gpu != h_ref)
    assert mism < 2e-3, mism
    # down: the oracle takes the GPU's h rows as input, so y isolates the down GEMM
    y_ref = orc.down_rows(h_gpu, experts[rows], dn, H)
    y_gpu = y.cpu().numpy()[rows].astype(np.float64)
    # fp32 accumulation over K = I products: relative error ~ sqrt(I) * 2^-24
    bound = 4.0 * np.sqrt(I) * 2.0 ** -24
    yerr = np.linalg.norm(y_gpu - y_ref) / np.linalg.norm(y_ref)
    assert yerr < bound, (yerr, bound)
    assert np.abs(y_gpu - y_ref).max() <= 10 * bound * np.sqrt(np.mean(y_ref ** 2))


def test_combine_parity():
    g = torch.Generator().manual_seed(31)
    T, H, k, E = 37, 256, 3, 6
    logits = torch.randn(T, E, generator=g)
    rids, rw = orc.route(logits.numpy(), k)
    _, _, _, inv = orc.permute(rids, E)
    y = torch.randn(T * k, H, generator=g)
    d = _lib.dims(T, H, 64, E, k)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    w32 = torch.from_numpy(rw.astype(np.float32)).to(DEV)
    _lib.moe_unpermute_combine(y.to(DEV), torch.from_numpy(inv).to(DEV), w32, d, out)
    ref = orc.combine(y.numpy().astype(np.float64), inv, rw.astype(np.float32).astype(np.float64))
    got = bf16_to_f64(bits(out))
    # one bf16 rounding of an fp32 sum of k terms
    assert np.all(np.abs(got - ref) <= 2 ** -8 * np.abs(ref) + 1e-6)


# ------------------------------------------------------------------ layer
def _layer(wl, d, T_max=None):
    return MoELayer(d["gu"], d["dn"], wl.H, wl.I, wl.E, wl.k, T_max or wl.T, DEV)


@pytest.mark.parametrize("name", ALL)
def test_layer_parity(name):
    wl, d = workload_inputs(name)
    gu, dn = numpy_weights(d)
    layer = _layer(wl, d)
    x = d["x"].to(DEV)
    logits = d["logits"].to(DEV)
    ids = torch.empty(wl.T, wl.k, dtype=torch.int32, device=DEV)
    w = torch.empty(wl.T, wl.k, dtype=torch.float32, device=DEV)
    out = layer.forward(x, logits, topk_ids=ids, topk_w=w)
    out2 = layer.forward(x, logits)
    assert layer.device_status() == _lib.MOE_OK
    got = bits(out)
    assert np.array_equal(got, bits(out2)), "layer output not deterministic"
    rids, rw = orc.route(d["logits"].numpy(), wl.k)
    assert np.array_equal(ids.cpu().numpy(), rids)
    assert np.abs(w.cpu().numpy() - rw).max() <= 2e-6
    rows = _layer_rows(name, rids, wl.E, seed=7)
    ref = orc.layer_rows(bits(d["x"]), rids, rw, gu, dn, rows)
    check_layer(got[rows], ref, name)


def test_layer_host_entry_matches_device_entry():
    wl, d = workload_inputs("tiny")
    layer = _layer(wl, d)
    out = layer.forward(d["x"].to(DEV), d["logits"].to(DEV))
    xh = d["x"].pin_memory()
    lh = d["logits"].pin_memory()
    oh = torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory()
    layer.forward_host(xh, lh, oh)
    assert np.array_equal(bits(out), bits(oh))


@pytest.mark.parametrize("pinned", [False, True])
def test_layer_host_entry_pageable_and_pinned(pinned):
    # pageable host buffers take the copy path through the workspace; pinned
    # ones let the kernels read the logits and write the output in place
    wl, d = workload_inputs("decode")
    layer = _layer(wl, d)
    ref = layer.forward(d["x"].to(DEV), d["logits"].to(DEV))
    torch.cuda.synchronize()
    xh, lh = d["x"].clone(), d["logits"].clone()
    oh = torch.full((wl.T, wl.H), float("nan"), dtype=torch.bfloat16)
    if pinned:
        xh, lh, oh = xh.pin_memory(), lh.pin_memory(), oh.pin_memory()
    layer.forward_host(xh, lh, oh)
    assert np.array_equal(bits(oh), bits(ref))
    assert layer.device_status() == _lib.MOE_OK


@pytest.mark.parametrize("T,H,I,E,k", [
    (128, 4096, 256, 32, 8),  # routing in one launch: x (1 MiB) copied by 16 extra blocks of it; 64-row tiles
    (200, 256, 128, 16, 8),   # routing, then histogram / scan / scatter: x copied before the routing
])
def test_host_entry_x_copy_paths(T, H, I, E, k):
    # page-locked buffers: x reaches the workspace through the routing launch
    # or through a copy of its own; either way the host entry and a host plan
    # equal the device entry bit for bit
    d = wk.generate_dims(T, H, I, E, k, seed=T + H)
    layer = MoELayer(d["gu"], d["dn"], H, I, E, k, T, DEV)
    ref = layer.forward(d["x"].to(DEV), d["logits"].to(DEV))
    torch.cuda.synchronize()
    xh, lh = d["x"].clone().pin_memory(), d["logits"].clone().pin_memory()
    oh = torch.full((T, H), float("nan"), dtype=torch.bfloat16).pin_memory()
    layer.forward_host(xh, lh, oh)
    assert np.array_equal(bits(oh), bits(ref))
    oh.fill_(float("nan"))
    s = torch.cuda.Stream()
    with layer.host_plan(xh, lh, oh, s) as plan:
        plan.run()
        plan.run()
    assert np.array_equal(bits(oh), bits(ref))
    assert layer.device_status() == _lib.MOE_OK


def test_host_plan_replays_with_new_host_contents():
    # a caller-owned plan (recorded graph) on page-locked buffers and a created
    # stream: every run must read the host inputs' current contents
    wl, d = workload_inputs("decode")
    layer = _layer(wl, d)
    s = torch.cuda.Stream()
    xh = d["x"].pin_memory()
    lh = d["logits"].pin_memory()
    oh = torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory()
    with layer.host_plan(xh, lh, oh, s) as plan:
        for rnd in range(3):
            x = torch.roll(d["x"], shifts=rnd, dims=0)
            lg = torch.roll(d["logits"], shifts=2 * rnd, dims=1)
            xh.copy_(x)
            lh.copy_(lg)
            ref = layer.forward(x.to(DEV), lg.to(DEV))
            # both calls use the layer's one workspace: the device call must end
            # before the plan runs on its own stream
            torch.cuda.synchronize()
            plan.run()
            assert np.array_equal(bits(oh), bits(ref)), f"round {rnd}"
    assert layer.device_status() == _lib.MOE_OK


def test_host_entries_with_freed_and_recreated_buffers():
    # page-locked buffers freed and allocated again (often at the same
    # address) between calls: the stateless host entry and a plan created on
    # the new buffers both equal the device entry bit for bit
    wl, d = workload_inputs("decode")
    layer = _layer(wl, d)
    s = torch.cuda.Stream()
    for rnd in range(3):
        x = torch.roll(d["x"], shifts=3 * rnd, dims=0)
        lg = torch.roll(d["logits"], shifts=rnd, dims=1)
        ref = layer.forward(x.to(DEV), lg.to(DEV))
        torch.cuda.synchronize()
        xh, lh = x.clone().pin_memory(), lg.clone().pin_memory()
        oh = torch.full((wl.T, wl.H), float("nan"), dtype=torch.bfloat16).pin_memory()
        layer.forward_host(xh, lh, oh, s)
        assert np.array_equal(bits(oh), bits(ref)), f"host entry, round {rnd}"
        oh.fill_(float("nan"))
        with layer.host_plan(xh, lh, oh, s) as plan:
            plan.run()
        assert np.array_equal(bits(oh), bits(ref)), f"host plan, round {rnd}"
        del xh, lh, oh
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        # torch keeps freed page-locked blocks for reuse, so the next round's
        # buffers usually come back at the same host addresses
    assert layer.device_status() == _lib.MOE_OK


def test_host_plan_rejects_pageable_buffers_and_default_stream():
    wl, d = workload_inputs("tiny")
    layer = _layer(wl, d)
    xh, lh = d["x"].clone(), d["logits"].clone()
    oh = torch.empty(wl.T, wl.H, dtype=torch.bfloat16)
    with pytest.raises(_lib.MoeError) as exc:
        layer.host_plan(xh, lh, oh, torch.cuda.Stream())
    assert exc.value.status == _lib.MOE_ERR_INVALID_ARG
    with pytest.raises(_lib.MoeError) as exc:
        layer.host_plan(xh.pin_memory(), lh.pin_memory(), oh.pin_memory(), 0)
    assert exc.value.status == _lib.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("T,H,I,E,k", [
    (1, 128, 64, 4, 1),      # single token
    (37, 256, 128, 8, 8),    # k = E, ragged T
    (24, 128, 64, 1, 1),     # one expert: dense FFN
    (300, 256, 192, 16, 2),  # several token tiles for hot experts, I not a multiple of 128
    (5, 128, 64, 1024, 32),  # maximum E and k
    (40, 256, 256, 64, 4),   # 16-row tiles in both projections, rows gathered by the GEMM
    (96, 512, 256, 64, 8),   # 32-row tiles
])
def test_layer_edge_shapes(T, H, I, E, k):
    d = wk.generate_dims(T, H, I, E, k, seed=T * 7 + E)
    gu, dn = numpy_weights(d)
    layer = MoELayer(d["gu"], d["dn"], H, I, E, k, T, DEV)
    out = layer.forward(d["x"].to(DEV), d["logits"].to(DEV))
    assert layer.device_status() == _lib.MOE_OK
    ref, _, _ = orc.layer(bits(d["x"]), d["logits"].numpy(), gu, dn, k)
    check_layer(bits(out), ref, f"T{T} H{H} I{I} E{E} k{k}")


@pytest.mark.parametrize("T,E,k", [
    (1, 4, 1), (33, 1024, 31), (128, 8, 8),   # one fused routing + grouping block (T*k <= 1024)
    (64, 1024, 4),                            # T*E too large to route inside the grouping block
    (129, 8, 8), (300, 96, 5),                # routing, then histogram / scan / scatter
])
def test_layer_routing_and_grouping_outputs(T, E, k):
    # the layer's own top-k ids and weights, NaN and tied logits included
    H, I = 128, 64
    d = wk.generate_dims(T, H, I, E, k, seed=T + 31 * E)
    logits = d["logits"].clone()
    logits[0, : min(E, 3)] = float("nan")
    if T > 2:
        logits[1, :] = float("nan")
        logits[2, :] = 0.5
    layer = MoELayer(d["gu"], d["dn"], H, I, E, k, T, DEV)
    ids = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, dtype=torch.float32, device=DEV)
    out = layer.forward(d["x"].to(DEV), logits.to(DEV), topk_ids=ids, topk_w=w)
    assert layer.device_status() == _lib.MOE_OK
    rids, rw = orc.route(logits.numpy(), k)
    assert np.array_equal(ids.cpu().numpy(), rids)
    assert np.abs(w.cpu().numpy() - rw).max() <= 2e-6
    gu, dn = numpy_weights(d)
    rows = np.arange(min(T, 16), dtype=np.int32)
    ref = orc.layer_rows(bits(d["x"]), rids, rw, gu, dn, rows)
    check_layer(bits(out)[rows], ref, f"T{T} E{E} k{k}")


@pytest.mark.parametrize("T,H,I,E,k", [(64, 256, 256, 32, 4), (48, 512, 512, 32, 8)])
def test_layer_skewed_narrow_tiles(T, H, I, E, k):
    # zipf-biased routing: hot experts span several narrow token tiles, cold ones none
    d = wk.generate_dims(T, H, I, E, k, seed=5 * T + E, router="zipf")
    gu, dn = numpy_weights(d)
    layer = MoELayer(d["gu"], d["dn"], H, I, E, k, T, DEV)
    out = layer.forward(d["x"].to(DEV), d["logits"].to(DEV))
    assert layer.device_status() == _lib.MOE_OK
    ref, _, _ = orc.layer(bits(d["x"]), d["logits"].numpy(), gu, dn, k)
    check_layer(bits(out), ref, f"zipf T{T} H{H} I{I} E{E} k{k}")


def test_layer_zero_tokens():
    d = wk.generate_dims(4, 128, 64, 4, 2, seed=3)
    layer = MoELayer(d["gu"], d["dn"], 128, 64, 4, 2, 4, DEV)
    out = torch.empty(0, 128, dtype=torch.bfloat16, device=DEV)
    layer.forward(torch.empty(0, 128, dtype=torch.bfloat16, device=DEV),
                  torch.empty(0, 4, dtype=torch.float32, device=DEV), out=out)
    assert layer.device_status() == _lib.MOE_OK


def test_unrouted_experts_are_never_read():
    # experts that receive no token get NaN scales; the output must be finite and unchanged
    T, H, I, E, k = 40, 256, 128, 12, 2
    d = wk.generate_dims(T, H, I, E, k, seed=77)
    d["logits"][:, 6:] -= 100.0
    base = MoELayer(d["gu"], d["dn"], H, I, E, k, T, DEV).forward(d["x"].to(DEV), d["logits"].to(DEV))
    gu = [a.clone() for a in d["gu"]]
    dn = [a.clone() for a in d["dn"]]
    gu[1][6:] = 0x7F
    dn[1][6:] = 0x7F
    gu[2][6:] = float("nan")
    dn[2][6:] = float("nan")
    out = MoELayer(gu, dn, H, I, E, k, T, DEV).forward(d["x"].to(DEV), d["logits"].to(DEV))
    assert torch.isfinite(out.float()).all()
    assert np.array_equal(bits(out), bits(base))


def test_output_guard_bands_untouched():
    wl, d = workload_inputs("tiny")
    layer = _layer(wl, d)
    guard = 4096
    buf = torch.full((guard + wl.T * wl.H + guard,), 0x5A5A, dtype=torch.int16, device=DEV)
    out = buf[guard:guard + wl.T * wl.H].view(torch.bfloat16).view(wl.T, wl.H)
    layer.forward(d["x"].to(DEV), d["logits"].to(DEV), out=out)
    torch.cuda.synchronize()
    b = buf.cpu()
    assert bool((b[:guard] == 0x5A5A).all()) and bool((b[guard + wl.T * wl.H:] == 0x5A5A).all())


def test_cross_cta_counter_wait_reports_timeout_and_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    _lib.moe_debug_counter_timeout_probe(ws, 20_000_000)    # 20 ms limit
    assert _lib.moe_get_device_status(ws) == _lib.MOE_ERR_DEVICE_TIMEOUT
    assert _lib.moe_get_device_status(ws) == _lib.MOE_OK
    wl, d = workload_inputs("decode")
    layer = _layer(wl, d)
    out = layer.forward(d["x"].to(DEV), d["logits"].to(DEV))
    assert layer.device_status() == _lib.MOE_OK
    assert torch.isfinite(out.float()).all()


def test_bounded_wait_reports_timeout_and_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    _lib.moe_debug_timeout_probe(ws, 20_000_000)            # 20 ms limit
    assert _lib.moe_get_device_status(ws) == _lib.MOE_ERR_DEVICE_TIMEOUT
    assert _lib.moe_get_device_status(ws) == _lib.MOE_OK     # the read clears it
    wl, d = workload_inputs("tiny")
    out = _layer(wl, d).forward(d["x"].to(DEV), d["logits"].to(DEV))
    assert torch.isfinite(out.float()).all()


# ------------------------------------------- token-tile width x tile schedule
@functools.lru_cache(maxsize=4)
def _oracle_ref(name):
    wl, d = workload_inputs(name)
    gu, dn = numpy_weights(d)
    rids, rw = orc.route(d["logits"].numpy(), wl.k)
    rows = _layer_rows(name, rids, wl.E, seed=11)
    return rows, orc.layer_rows(bits(d["x"]), rids, rw, gu, dn, rows)


@pytest.mark.parametrize("name", ["tiny", "decode", "grouped"])
def test_layer_every_tile_width_and_schedule(name):
    # every token-tile width (16/32 gather rows in the GEMM and run both
    # projections in one launch unless grid3d; 64/128 read a permuted copy)
    # and every schedule (static, claim, the 3-D grid): within tolerance of
    # the oracle and bit-identical to the library's default choice
    wl, d = workload_inputs(name)
    layer = _layer(wl, d)
    x, logits = d["x"].to(DEV), d["logits"].to(DEV)
    dims = layer.dims(wl.T)
    rows, ref = _oracle_ref(name)
    default = bits(layer.forward(x, logits))
    for bn in (16, 32, 64, 128):
        outs = []
        for sched in (0, 1, 2):
            out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=DEV)
            _lib.moe_debug_layer_forward_config(x, logits, layer.w_gate_up.abi, layer.w_down.abi, dims, out, None,
                                                None, layer.ws, layer.ws_bytes, bn, sched)
            assert layer.device_status() == _lib.MOE_OK, (bn, sched)
            check_layer(bits(out)[rows], ref, f"{name} bn={bn} sched={sched}")
            outs.append(bits(out))
        # every MMA runs the same K order for a given output element, whatever
        # the token-tile width or schedule: the results are the same bits
        for o in outs:
            assert np.array_equal(o, default), f"{name} bn={bn}: differs from the default choice"


def test_forced_config_rejects_bad_choices():
    wl, d = workload_inputs("tiny")
    layer = _layer(wl, d)
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=DEV)
    for bn, sched in [(48, 0), (16, 3), (16, -2)]:
        with pytest.raises(_lib.MoeError) as exc:
            _lib.moe_debug_layer_forward_config(d["x"].to(DEV), d["logits"].to(DEV), layer.w_gate_up.abi,
                                                layer.w_down.abi, layer.dims(wl.T), out, None, None, layer.ws,
                                                layer.ws_bytes, bn, sched)
        assert exc.value.status == _lib.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["decode", "grouped"])
def test_concurrent_layer_calls_on_two_streams(name):
    # Two layer calls on two streams, each with its own workspace, launched
    # back to back so that their GEMMs compete for the SMs: both finish with
    # MOE_OK and equal the same calls run one after the other, bit for bit.
    wl, d = workload_inputs(name)
    a = _layer(wl, d)
    b = _layer(wl, d)
    xa, la = d["x"].to(DEV), d["logits"].to(DEV)
    xb, lb = torch.roll(xa, 1, 0).contiguous(), torch.roll(la, 3, 1).contiguous()
    ref_a = a.forward(xa, la)
    ref_b = b.forward(xb, lb)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    for rnd in range(5):
        oa = torch.empty_like(ref_a)
        ob = torch.empty_like(ref_b)
        torch.cuda.synchronize()
        a.forward(xa, la, out=oa, stream=sa)
        b.forward(xb, lb, out=ob, stream=sb)
        torch.cuda.synchronize()
        assert a.device_status(sa) == _lib.MOE_OK and b.device_status(sb) == _lib.MOE_OK, rnd
        assert np.array_equal(bits(oa), bits(ref_a)) and np.array_equal(bits(ob), bits(ref_b)), rnd


def test_layer_while_another_stream_holds_sms():
    # A long GEMM of another library on a second stream keeps SMs busy while
    # the one-launch layer starts: the layer must still end with MOE_OK and
    # the same output.
    wl, d = workload_inputs("decode")
    layer = _layer(wl, d)
    x, logits = d["x"].to(DEV), d["logits"].to(DEV)
    ref = layer.forward(x, logits)
    torch.cuda.synchronize()
    m = torch.randn(8192, 8192, device=DEV, dtype=torch.bfloat16)
    other = torch.cuda.Stream()
    for rnd in range(3):
        with torch.cuda.stream(other):
            busy = m @ m
        out = layer.forward(x, logits)
        torch.cuda.synchronize()
        assert layer.device_status() == _lib.MOE_OK, rnd
        assert np.array_equal(bits(out), bits(ref)), rnd
    del busy
