"""Seeded synthetic workloads for the W4A16 NVFP4 MoE layer.

This module only draws inputs.  It holds none of the layer's arithmetic: no
decoding, no routing, no GEMM.  Both the CUDA path and the fp64 oracle consume
what it returns; neither is imported here.

Shapes follow the pages' workloads:
  * the grouped-GEMM shape of the Atlas article (f.mffb.com.cn/a/497905.html,
    section "编译时内核选择和W4A16 Grouped GEMM"): 800 tokens, 256 experts,
    gate_up and down projections;
  * the MoE families in the ATOM article's model table
    (itsolotime.com/archives/33112): 128 experts top-8 (Qwen3-MoE class) and
    8 experts top-2 (Mixtral class).
The pages' measurements use trained checkpoints, which are not available; the
seeded draws below stand in for them with the same shapes.

Weights are drawn in fp32 and quantised here to NVFP4: E2M1 codes packed two
per byte (element 2i in the low nibble), one E4M3 block scale per 16 elements
along K, one fp32 global scale per expert matrix.  The quantiser choices
(global scale = amax / (6 * 448), block scale = RNE_e4m3(amax16 / 6 / gs),
code = RNE_e2m1(w / (scale * gs)) saturating at +-6) define the inputs only;
both sides read the same bytes.
"""
from __future__ import annotations

import dataclasses
import math
import re

import numpy as np
import torch

__all__ = ["Workload", "WORKLOADS", "by_name", "generate", "quantize_nvfp4", "algorithmic_bytes",
           "algorithmic_flops", "touched_experts"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    router: str          # "weight": logits = x @ Wr^T, Wr ~ N(0, 1/H); "normal": N(0,1); "zipf": N(0,1) + bias
    seed: int
    note: str = ""

    @property
    def dims(self):
        return dict(T=self.T, H=self.H, I=self.I, E=self.E, k=self.k)


WORKLOADS = [
    Workload("tiny_T16_H256_I128_E8_k2", 16, 256, 128, 8, 2, "weight", 1000,
             "correctness gate; the oracle finishes in well under a second"),
    Workload("decode_T32_H2048_I768_E128_k8", 32, 2048, 768, 128, 8, "weight", 1001,
             "decode-shaped, weight-bandwidth bound (128 experts, top-8)"),
    Workload("grouped_T800_H2048_I512_E256_k8", 800, 2048, 512, 256, 8, "normal", 1002,
             "the Atlas article's grouped-GEMM shape: 800 tokens x 256 experts"),
    Workload("prefill_T4096_H4096_I14336_E8_k2", 4096, 4096, 14336, 8, 2, "normal", 1003,
             "prefill-shaped, compute bound (8 experts, top-2)"),
    Workload("skewed_T8192_H2048_I768_E128_k8", 8192, 2048, 768, 128, 8, "zipf", 1004,
             "skewed routing: Zipf(1.2) expert bias, several experts receive no tokens"),
]


def by_name(name: str) -> Workload:
    """A workload of WORKLOADS by its name or its first word, or an arbitrary
    shape named custom_T<T>_H<H>_I<I>_E<E>_k<k> (normal router, seed 2000)."""
    for w in WORKLOADS:
        if w.name == name or w.name.split("_")[0] == name:
            return w
    m = re.fullmatch(r"custom_T(\d+)_H(\d+)_I(\d+)_E(\d+)_k(\d+)", name)
    if m:
        T, H, I, E, k = (int(g) for g in m.groups())
        return Workload(name, T, H, I, E, k, "normal", 2000)
    raise KeyError(name)


# ---------------------------------------------------------------- quantiser
_E4M3_MAX = 448.0
_E2M1_MAX = 6.0


def quantize_nvfp4(W: torch.Tensor):
    """fp32 [N, K] -> (codes uint8 [N, K/2], scales uint8 [N, K/16], gs float).

    gs = amax / (6 * 448) (1.0 if the matrix is all zero); per block of 16:
    s = RNE_e4m3(min(amax16 / 6 / gs, 448)); code = RNE_e2m1(w / (dec(s) * gs)),
    ties to the even mantissa, saturating at +-6, all zero if dec(s) == 0.
    """
    assert W.dtype == torch.float32 and W.dim() == 2 and W.shape[1] % 16 == 0
    N, K = W.shape
    amax = float(W.abs().max()) if W.numel() else 0.0
    gs = np.float32(amax / (6.0 * _E4M3_MAX)) if amax > 0 else np.float32(1.0)
    Wb = W.view(N, K // 16, 16)
    bmax = Wb.abs().amax(dim=-1)
    s8 = (bmax / 6.0 / float(gs)).clamp(max=_E4M3_MAX).to(torch.float8_e4m3fn)
    sv = s8.to(torch.float32)
    denom = (sv * float(gs)).unsqueeze(-1)
    q = torch.where(denom > 0, Wb / torch.where(denom > 0, denom, torch.ones_like(denom)), torch.zeros_like(Wb))
    a = q.abs()
    # E2M1 magnitude grid {0, .5, 1, 1.5, 2, 3, 4, 6}; midpoints resolved to the
    # even mantissa: .25->0, .75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4.
    idx = ((a > 0.25).to(torch.uint8) + (a >= 0.75).to(torch.uint8) + (a > 1.25).to(torch.uint8)
           + (a >= 1.75).to(torch.uint8) + (a > 2.5).to(torch.uint8) + (a >= 3.5).to(torch.uint8)
           + (a > 5.0).to(torch.uint8))
    sign = ((q < 0) & (idx > 0)).to(torch.uint8)
    code = (idx | (sign << 3)).view(N, K)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).contiguous()
    return packed, s8.view(torch.uint8).contiguous(), float(gs)


def _draw_matrix(gen: torch.Generator, N: int, K: int) -> torch.Tensor:
    # "N(0, 1/sqrt(K))" read as standard deviation 1/sqrt(K).
    return torch.randn(N, K, generator=gen, dtype=torch.float32) * (1.0 / math.sqrt(K))


def _quantize_experts(gen, E, N, K):
    codes = torch.empty(E, N, K // 2, dtype=torch.uint8)
    scales = torch.empty(E, N, K // 16, dtype=torch.uint8)
    gs = torch.empty(E, dtype=torch.float32)
    for e in range(E):
        c, s, g = quantize_nvfp4(_draw_matrix(gen, N, K))
        codes[e], scales[e], gs[e] = c, s, g
    return codes, scales, gs


def zipf_bias(E: int, s: float = 1.2) -> np.ndarray:
    """bias_e = 3 * ln p_rank(e), p_r = r^-s / sum_r r^-s, rank(e) = e + 1 (expert 0 hottest)."""
    r = np.arange(1, E + 1, dtype=np.float64)
    p = r ** (-s)
    p /= p.sum()
    return 3.0 * np.log(p)


def generate(wl: Workload, seed: int | None = None, with_weights: bool = True):
    """Return a dict of CPU tensors:
    x bf16 [T,H]; logits f32 [T,E]; gu = (codes u8 [E,2I,H/2], scales u8 [E,2I,H/16], gs f32 [E]);
    dn = (codes u8 [E,H,I/2], scales u8 [E,H,I/16], gs f32 [E])."""
    seed = wl.seed if seed is None else seed
    gen = torch.Generator().manual_seed(seed)
    T, H, I, E = wl.T, wl.H, wl.I, wl.E
    x = torch.randn(T, H, generator=gen, dtype=torch.float32).to(torch.bfloat16)
    if wl.router == "weight":
        # router weight Wr ~ N(0, 1/H) (variance 1/H); logits computed in fp64
        # from the bf16 activations and rounded once to fp32, so that routing
        # is a fixed input rather than a reduction order.
        Wr = torch.randn(E, H, generator=gen, dtype=torch.float32) * (1.0 / math.sqrt(H))
        logits = (x.double() @ Wr.double().T).float()
    elif wl.router == "normal":
        logits = torch.randn(T, E, generator=gen, dtype=torch.float32)
    elif wl.router == "zipf":
        logits = (torch.randn(T, E, generator=gen, dtype=torch.float64)
                  + torch.from_numpy(zipf_bias(E))[None, :]).float()
    else:
        raise ValueError(wl.router)
    out = dict(x=x.contiguous(), logits=logits.contiguous())
    if with_weights:
        out["gu"] = _quantize_experts(gen, E, 2 * I, H)
        out["dn"] = _quantize_experts(gen, E, H, I)
    return out


def router_weights(wl: Workload, seed: int | None = None, bias: bool = True):
    """bf16 router weights Wr [E,H] ~ N(0, 1/H) (variance 1/H) and an fp32 bias
    [E] ~ N(0, 0.1^2) (or None), from a generator of their own (seed + 7777),
    for the layer that computes its own gate logits."""
    seed = (wl.seed if seed is None else seed) + 7777
    gen = torch.Generator().manual_seed(seed)
    Wr = (torch.randn(wl.E, wl.H, generator=gen, dtype=torch.float32) * (1.0 / math.sqrt(wl.H))).to(torch.bfloat16)
    b = (torch.randn(wl.E, generator=gen, dtype=torch.float32) * 0.1) if bias else None
    return Wr.contiguous(), b


def shared_expert(wl: Workload, seed: int | None = None):
    """NVFP4 weights of one shared expert with the routed experts' H and I, from a
    generator of their own (seed + 4242): (gu, dn) in the layout of generate()'s,
    with E = 1."""
    seed = (wl.seed if seed is None else seed) + 4242
    gen = torch.Generator().manual_seed(seed)
    return _quantize_experts(gen, 1, 2 * wl.I, wl.H), _quantize_experts(gen, 1, wl.H, wl.I)


def generate_dims(T, H, I, E, k, seed, router="normal"):
    """Same recipe for an arbitrary shape (used by edge-case tests)."""
    return generate(Workload(f"custom_T{T}_H{H}_I{I}_E{E}_k{k}", T, H, I, E, k, router, seed))


# ------------------------------------------------------- algorithmic volume
def touched_experts(counts) -> int:
    return int(np.count_nonzero(np.asarray(counts)))


def algorithmic_bytes(T, H, I, E, k, counts) -> int:
    """Bytes the layer must move at minimum: NVFP4 weights (codes + E4M3 scales,
    0.5625 B per element, plus the fp32 global scales of both projections) of the
    experts that receive tokens, x (bf16), out (bf16) and the fp32 logits."""
    n = touched_experts(counts)
    w = n * (3 * H * I * 9 // 16 + 8)
    return w + T * H * 2 + T * H * 2 + T * E * 4


def algorithmic_flops(T, H, I, k) -> int:
    """2 * (T*k) * (2I*H + H*I): gate_up and down over the routed rows only."""
    return 6 * T * k * H * I
