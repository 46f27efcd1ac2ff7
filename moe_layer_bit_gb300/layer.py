"""Python-side convenience around the C ABI: device weights, workspace, forward.

Marshalling only -- allocation of device buffers with torch and calls into
libmoe_w4a16.so.  The layer is the W4A16 NVFP4 MoE FFN of the Atlas article
(f.mffb.com.cn/a/497905.html, section "编译时内核选择和W4A16 Grouped GEMM").
"""
from __future__ import annotations

import dataclasses

import torch

from . import _lib


@dataclasses.dataclass
class PackedProjection:
    packed: torch.Tensor        # uint8, moe_packed_w4_bytes(E, N, K)
    global_scale: torch.Tensor  # float32 [E]
    E: int
    N: int
    K: int

    @property
    def abi(self) -> _lib.W4:
        # built once per pair of device buffers (rebuilt if a field is replaced)
        key = (self.packed.data_ptr(), self.global_scale.data_ptr())
        cached = self.__dict__.get("_abi")
        if cached is None or cached[0] != key:
            cached = self.__dict__["_abi"] = (key, _lib.w4(self.packed, self.global_scale))
        return cached[1]


def pack_projection(codes: torch.Tensor, scales: torch.Tensor, global_scale: torch.Tensor, proj: int,
                    device="cuda", stream=None) -> PackedProjection:
    """Upload natural-layout NVFP4 weights (codes [E,N,K/2], scales [E,N,K/16], gs [E]) and
    re-lay them out once with moe_prepack_w4."""
    E, N, K2 = codes.shape
    K = 2 * K2
    c = codes.to(device, non_blocking=False).contiguous()
    s = scales.to(device).contiguous()
    out = torch.empty(_lib.moe_packed_w4_bytes(E, N, K), dtype=torch.uint8, device=device)
    _lib.moe_prepack_w4(c, s, E, N, K, proj, out, stream)
    gs = global_scale.to(device=device, dtype=torch.float32).contiguous()
    torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
    del c, s
    return PackedProjection(out, gs, E, N, K)


class MoELayer:
    """W4A16 NVFP4 MoE FFN layer for up to T_max tokens per call."""

    def __init__(self, gu, dn, H: int, I: int, E: int, k: int, T_max: int, device="cuda", shared=None):
        """shared: optional (gate_up, down) natural-layout weights of a shared expert
        (one expert, the routed experts' H and I), used by forward_shared."""
        self.H, self.I, self.E, self.k, self.T_max = H, I, E, k, T_max
        self.device = torch.device(device)
        self.w_gate_up = pack_projection(*gu, _lib.MOE_PROJ_GATE_UP, device)
        self.w_down = pack_projection(*dn, _lib.MOE_PROJ_DOWN, device)
        self.shared = None
        if shared is not None:
            self.shared = (pack_projection(*shared[0], _lib.MOE_PROJ_GATE_UP, device),
                           pack_projection(*shared[1], _lib.MOE_PROJ_DOWN, device))
        self._dims = {}
        d = _lib.dims(T_max, H, I, E, k)
        self.ws_bytes = _lib.moe_workspace_bytes(d)
        if self.ws_bytes == 0:
            raise _lib.MoeError(_lib.MOE_ERR_UNSUPPORTED_SHAPE, "MoELayer")
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=self.device)  # status word starts at 0

    def dims(self, T: int) -> _lib.Dims:
        if T > self.T_max:
            raise ValueError(f"T={T} > T_max={self.T_max}")
        d = self._dims.get(T)
        if d is None:
            d = self._dims[T] = _lib.dims(T, self.H, self.I, self.E, self.k)
        return d

    def forward(self, x: torch.Tensor, logits: torch.Tensor, out: torch.Tensor | None = None,
                topk_ids: torch.Tensor | None = None, topk_w: torch.Tensor | None = None, stream=None):
        T = x.shape[0]
        if out is None:
            out = torch.empty(T, self.H, dtype=torch.bfloat16, device=self.device)
        _lib.moe_layer_forward(x, logits, self.w_gate_up.abi, self.w_down.abi, self.dims(T), out, topk_ids, topk_w,
                               self.ws, self.ws_bytes, stream)
        return out

    def forward_router(self, x: torch.Tensor, router_weight: torch.Tensor, router_bias: torch.Tensor | None = None,
                       out: torch.Tensor | None = None, logits_out: torch.Tensor | None = None,
                       topk_ids: torch.Tensor | None = None, topk_w: torch.Tensor | None = None, stream=None):
        """The layer with its gate logits computed from bf16 router weights [E][H] (+ fp32 bias [E])."""
        T = x.shape[0]
        if out is None:
            out = torch.empty(T, self.H, dtype=torch.bfloat16, device=self.device)
        _lib.moe_layer_forward_router(x, router_weight, router_bias, self.w_gate_up.abi, self.w_down.abi, self.dims(T),
                                      out, logits_out, topk_ids, topk_w, self.ws, self.ws_bytes, stream)
        return out

    def forward_shared(self, x: torch.Tensor, logits: torch.Tensor | None = None,
                       router_weight: torch.Tensor | None = None, router_bias: torch.Tensor | None = None,
                       out: torch.Tensor | None = None, logits_out: torch.Tensor | None = None,
                       topk_ids: torch.Tensor | None = None, topk_w: torch.Tensor | None = None, stream=None):
        """The layer plus the shared expert; gate logits given, or computed from router weights."""
        if self.shared is None:
            raise ValueError("MoELayer was built without shared expert weights")
        T = x.shape[0]
        if out is None:
            out = torch.empty(T, self.H, dtype=torch.bfloat16, device=self.device)
        _lib.moe_layer_forward_shared(x, logits, router_weight, router_bias, self.w_gate_up.abi, self.w_down.abi,
                                      self.shared[0].abi, self.shared[1].abi, self.dims(T), out, logits_out,
                                      topk_ids, topk_w, self.ws, self.ws_bytes, stream)
        return out

    def forward_host(self, x_host: torch.Tensor, logits_host: torch.Tensor, out_host: torch.Tensor, stream=None):
        """Host buffers in, host buffer out (copies inside the call; synchronises)."""
        T = x_host.shape[0]
        _lib.moe_layer_forward_host(x_host, logits_host, self.w_gate_up.abi, self.w_down.abi, self.dims(T), out_host,
                                    self.ws, self.ws_bytes, stream)
        return out_host

    def host_plan(self, x_host: torch.Tensor, logits_host: torch.Tensor, out_host: torch.Tensor, stream):
        """A recorded host-buffer call on these page-locked buffers and this stream (HostPlan.run() per
        call; close() or the context manager frees it)."""
        return HostPlan(self, x_host, logits_host, out_host, stream)

    def device_status(self, stream=None) -> int:
        return _lib.moe_get_device_status(self.ws, stream)


class HostPlan:
    """Caller-owned moe_host_plan: the layer on fixed page-locked host buffers, replayed as one graph."""

    def __init__(self, layer: MoELayer, x_host, logits_host, out_host, stream):
        self.handle = None
        self._keep = (x_host, logits_host, out_host, stream, layer)
        self.handle = _lib.moe_host_plan_create(x_host, logits_host, layer.w_gate_up.abi, layer.w_down.abi,
                                                layer.dims(x_host.shape[0]), out_host, layer.ws, layer.ws_bytes,
                                                stream)

    def run(self):
        _lib.moe_host_plan_run(self.handle)

    def close(self):
        if self.handle is not None:
            _lib.moe_host_plan_destroy(self.handle)
            self.handle = None
            self._keep = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class W4A4Layer:
    """The block-scaled FP4 layer (NVFP4 weights and NVFP4 activations) for up to T_max tokens:
    weights stay in their natural NVFP4 layout on the device."""

    def __init__(self, gu, dn, H: int, I: int, E: int, k: int, T_max: int, device="cuda"):
        self.H, self.I, self.E, self.k, self.T_max = H, I, E, k, T_max
        self.device = torch.device(device)
        self.gu = tuple(t.to(self.device).contiguous() for t in gu[:2]) + (gu[2].to(self.device, torch.float32),)
        self.dn = tuple(t.to(self.device).contiguous() for t in dn[:2]) + (dn[2].to(self.device, torch.float32),)
        self.ws_bytes = _lib.moe_w4a4_workspace_bytes(_lib.dims(T_max, H, I, E, k))
        if self.ws_bytes == 0:
            raise _lib.MoeError(_lib.MOE_ERR_UNSUPPORTED_SHAPE, "W4A4Layer")
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=self.device)
        self._abi = (_lib.w4n(*self.gu), _lib.w4n(*self.dn))

    def forward(self, x: torch.Tensor, logits: torch.Tensor, out: torch.Tensor | None = None,
                topk_ids: torch.Tensor | None = None, topk_w: torch.Tensor | None = None, stream=None):
        T = x.shape[0]
        if T > self.T_max:
            raise ValueError(f"T={T} > T_max={self.T_max}")
        if out is None:
            out = torch.empty(T, self.H, dtype=torch.bfloat16, device=self.device)
        _lib.moe_layer_forward_w4a4(x, logits, self._abi[0], self._abi[1], _lib.dims(T, self.H, self.I, self.E, self.k),
                                    out, topk_ids, topk_w, self.ws, self.ws_bytes, stream)
        return out

    def device_status(self, stream=None) -> int:
        return _lib.moe_get_device_status(self.ws, stream)
