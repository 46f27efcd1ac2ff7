"""Shared helpers of the GPU parity tests: cached seeded inputs, device upload,
the layer tolerance, and sampling of tokens for the large workloads."""
from __future__ import annotations

import functools

import numpy as np
import torch

from moe_layer_bit_gb300 import workloads as wk

# Layer-output tolerance of the bf16 result against the fp64 oracle:
# relative Frobenius error <= 5e-3 and, per element,
# |err| <= 2e-2 * |ref| + 2e-3 * rms(ref).
REL_FRO = 5e-3
ELEM_REL = 2e-2
ELEM_RMS = 2e-3


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 numpy bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@functools.lru_cache(maxsize=5)
def workload_inputs(name: str):
    wl = wk.by_name(name)
    d = wk.generate(wl)
    return wl, d


def numpy_weights(d):
    gu = tuple(a.numpy() for a in d["gu"])
    dn = tuple(a.numpy() for a in d["dn"])
    return gu, dn


def check_layer(out_gpu_bf16: np.ndarray, ref: np.ndarray, what: str = ""):
    """Apply the layer tolerance; returns (rel_fro, worst element ratio)."""
    got = bf16_to_f64(out_gpu_bf16)
    err = got - ref
    rel_fro = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300)
    rms = np.sqrt(np.mean(ref ** 2))
    bound = ELEM_REL * np.abs(ref) + ELEM_RMS * rms
    ratio = np.abs(err) / bound
    worst = float(ratio.max()) if ratio.size else 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert rel_fro <= REL_FRO, f"{what}: relative Frobenius error {rel_fro:.3e} > {REL_FRO}"
    assert worst <= 1.0, (f"{what}: {int((ratio > 1).sum())} elements over the per-element bound, "
                          f"worst ratio {worst:.3f}")
    return rel_fro, worst


def seam_tokens(ids: np.ndarray, E: int, tile: int) -> np.ndarray:
    """Tokens at the seams of the GEMMs' token tiles: for every expert and every
    `tile`-row tile of its rows (rows grouped by expert, then token), the tokens
    of the tile's first and last row."""
    flat = ids.reshape(-1)
    order = np.argsort(flat, kind="stable")          # rows sorted by (expert, token)
    tok = order // ids.shape[1]
    counts = np.bincount(flat, minlength=E)
    off = np.concatenate([[0], np.cumsum(counts)])
    out = set()
    for e in np.nonzero(counts)[0]:
        for r0 in range(int(off[e]), int(off[e + 1]), tile):
            out.add(int(tok[r0]))
            out.add(int(tok[min(r0 + tile, int(off[e + 1])) - 1]))
    return np.array(sorted(out), np.int32)


def sample_tokens(ids: np.ndarray, E: int, n: int, seed: int, tile: int = 0, seams: int = 0) -> np.ndarray:
    """Seeded token sample covering every expert that has tokens (stratified: for
    each expert not yet covered, one of its tokens), plus up to `seams` tokens
    at the seams of `tile`-row token tiles, topped up to n tokens."""
    rng = np.random.default_rng(seed)
    T = ids.shape[0]
    chosen, covered = set(), set()
    if tile > 0 and seams > 0:
        st = seam_tokens(ids, E, tile)
        if st.size > seams:
            st = rng.choice(st, size=seams, replace=False)
        chosen.update(int(t) for t in st)
    for e in rng.permutation(E):
        if e in covered:
            continue
        rows = np.nonzero((ids == e).any(axis=1))[0]
        if rows.size == 0:
            continue
        t = int(rng.choice(rows))
        chosen.add(t)
        covered.update(int(v) for v in ids[t])
    for t in rng.permutation(T):
        if len(chosen) >= n:
            break
        chosen.add(int(t))
    return np.array(sorted(chosen), np.int32)
