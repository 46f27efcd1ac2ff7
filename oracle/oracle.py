"""ctypes wrapper around oracle.c -- the fp64 CPU oracle of the W4A16 NVFP4 MoE layer.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline leg; never by the library.  It shares no code with the
CUDA path.  Every function here is argument marshalling around the C code; the
arithmetic, and the citations of what it follows, are in oracle.c.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# -std=c11 keeps fp contraction off (also given explicitly) so x86 and Arm
# hosts produce the same bits; no -ffast-math, no OpenMP, no BLAS.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, single-threaded code)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i = ctypes.c_int
            lib.oracle_dec_e2m1.restype = ctypes.c_double
            lib.oracle_dec_e2m1.argtypes = [ctypes.c_uint]
            lib.oracle_dec_e4m3.restype = ctypes.c_double
            lib.oracle_dec_e4m3.argtypes = [ctypes.c_uint]
            lib.oracle_bf16_rne.restype = ctypes.c_uint16
            lib.oracle_bf16_rne.argtypes = [ctypes.c_double]
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_weight.restype = ctypes.c_double
            lib.oracle_weight.argtypes = [P, P, P, i, i, i, i, i]
            lib.oracle_decode_row.restype = None
            lib.oracle_decode_row.argtypes = [P, P, P, i, i, i, i, P]
            lib.oracle_router_logits.restype = None
            lib.oracle_router_logits.argtypes = [P, P, P, i, i, i, P]
            lib.oracle_router_logits_exact.restype = None
            lib.oracle_router_logits_exact.argtypes = [P, P, P, i, i, i, P]
            lib.oracle_route.restype = None
            lib.oracle_route.argtypes = [P, i, i, i, P, P]
            lib.oracle_permute.restype = None
            lib.oracle_permute.argtypes = [P, i, i, i, P, P, P, P]
            lib.oracle_gate_up_swiglu_row.restype = None
            lib.oracle_gate_up_swiglu_row.argtypes = [P, i, i, P, P, P, i, P, P]
            lib.oracle_down_row.restype = None
            lib.oracle_down_row.argtypes = [P, i, i, P, P, P, i, P]
            lib.oracle_combine.restype = None
            lib.oracle_combine.argtypes = [P, P, P, i, i, i, P]
            lib.oracle_layer_rows.restype = None
            lib.oracle_layer_rows.argtypes = [P, P, P, P, P, P, P, P, P, i, i, i, P, i, P]
            lib.oracle_e4m3_rne.restype = ctypes.c_uint
            lib.oracle_e4m3_rne.argtypes = [ctypes.c_float]
            lib.oracle_e2m1_rne.restype = ctypes.c_uint
            lib.oracle_e2m1_rne.argtypes = [ctypes.c_float]
            lib.oracle_quant_nvfp4.restype = None
            lib.oracle_quant_nvfp4.argtypes = [P, i, P, P]
            lib.oracle_w4a4_layer_rows.restype = None
            lib.oracle_w4a4_layer_rows.argtypes = [P, P, P, P, P, P, P, P, P, i, i, i, P, i, P]
            lib.oracle_layer.restype = None
            lib.oracle_layer.argtypes = [P, P, P, P, P, P, P, P, i, i, i, i, i, P, P, P]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


# ------------------------------------------------------------------ decoders
def dec_e2m1(code: int) -> float:
    return _load().oracle_dec_e2m1(int(code))


def dec_e4m3(code: int) -> float:
    return _load().oracle_dec_e4m3(int(code))


def bf16_rne(v: float) -> int:
    return int(_load().oracle_bf16_rne(float(v)))


def bf16_to_float(bits: int) -> float:
    return _load().oracle_bf16_to_double(int(bits))


def weight(codes, scales, gs, N, K, e, n, kk) -> float:
    codes, scales, gs = _c(codes, np.uint8), _c(scales, np.uint8), _c(gs, np.float32)
    return _load().oracle_weight(_ptr(codes), _ptr(scales), _ptr(gs), N, K, e, n, kk)


def decode_row(codes, scales, gs, N, K, e, n) -> np.ndarray:
    codes, scales, gs = _c(codes, np.uint8), _c(scales, np.uint8), _c(gs, np.float32)
    out = np.empty(K, np.float64)
    _load().oracle_decode_row(_ptr(codes), _ptr(scales), _ptr(gs), N, K, e, n, _ptr(out))
    return out


# ------------------------------------------------------------- router logits
def router_logits(x_bf16, wr_bf16, bias=None) -> np.ndarray:
    """fp32 [T,E] gate logits in the library's fixed reduction order (bit-exact target)."""
    x, wr = _c(x_bf16, np.uint16), _c(wr_bf16, np.uint16)
    T, H = x.shape
    E = wr.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((T, E), np.float32)
    _load().oracle_router_logits(_ptr(x), _ptr(wr), None if b is None else _ptr(b), T, H, E, _ptr(out))
    return out


def router_logits_exact(x_bf16, wr_bf16, bias=None) -> np.ndarray:
    """fp64 [T,E] gate logits, the exact sum (the definition)."""
    x, wr = _c(x_bf16, np.uint16), _c(wr_bf16, np.uint16)
    T, H = x.shape
    E = wr.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((T, E), np.float64)
    _load().oracle_router_logits_exact(_ptr(x), _ptr(wr), None if b is None else _ptr(b), T, H, E, _ptr(out))
    return out


# ------------------------------------------------------------------- routing
def route(logits, k: int):
    """-> (ids int32 [T,k], w float64 [T,k])."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    _load().oracle_route(_ptr(logits), T, E, k, _ptr(ids), _ptr(w))
    return ids, w


def permute(ids, E: int):
    """-> (counts [E], offsets [E+1], sorted_token [T*k], inv_perm [T*k]) all int32."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    sorted_token = np.empty(T * k, np.int32)
    inv_perm = np.empty(T * k, np.int32)
    _load().oracle_permute(_ptr(ids), T, E, k, _ptr(counts), _ptr(offsets), _ptr(sorted_token), _ptr(inv_perm))
    return counts, offsets, sorted_token, inv_perm


# ------------------------------------------------------------- expert stages
def gate_up_swiglu_rows(x_rows_bf16, experts, gu, I: int):
    """x_rows_bf16: uint16 [P,H] (bf16 bits); experts: [P] expert per row;
    gu = (codes [E,2I,H/2], scales [E,2I,H/16], gs [E]).
    -> (h_exact float64 [P,I], h_bf16 uint16 [P,I])."""
    x = _c(x_rows_bf16, np.uint16)
    P_, H = x.shape
    codes, scales, gs = _c(gu[0], np.uint8), _c(gu[1], np.uint8), _c(gu[2], np.float32)
    h_exact = np.empty((P_, I), np.float64)
    h_bf16 = np.empty((P_, I), np.uint16)
    lib = _load()
    for p in range(P_):
        lib.oracle_gate_up_swiglu_row(_ptr(x[p]), H, I, _ptr(codes), _ptr(scales), _ptr(gs), int(experts[p]),
                                      _ptr(h_exact[p]), _ptr(h_bf16[p]))
    return h_exact, h_bf16


def down_rows(h_rows_bf16, experts, dn, H: int):
    """h_rows_bf16: uint16 [P,I]; dn = (codes [E,H,I/2], scales [E,H,I/16], gs [E]). -> y float64 [P,H]."""
    h = _c(h_rows_bf16, np.uint16)
    P_, I = h.shape
    codes, scales, gs = _c(dn[0], np.uint8), _c(dn[1], np.uint8), _c(dn[2], np.float32)
    y = np.empty((P_, H), np.float64)
    lib = _load()
    for p in range(P_):
        lib.oracle_down_row(_ptr(h[p]), H, I, _ptr(codes), _ptr(scales), _ptr(gs), int(experts[p]), _ptr(y[p]))
    return y


def combine(y, inv_perm, w):
    """y f64 [T*k,H] (sorted rows), inv_perm [T*k], w [T,k] -> out f64 [T,H]."""
    y = _c(y, np.float64)
    inv_perm = _c(inv_perm, np.int32)
    w = _c(w, np.float64)
    T, k = w.shape
    H = y.shape[1]
    out = np.empty((T, H), np.float64)
    _load().oracle_combine(_ptr(y), _ptr(inv_perm), _ptr(w), T, H, k, _ptr(out))
    return out


# --------------------------------------------------------------------- layer
def layer(x_bf16, logits, gu, dn, k: int):
    """Whole layer. x_bf16 uint16 [T,H]; logits f32 [T,E]. -> (out f64 [T,H], ids, w)."""
    x = _c(x_bf16, np.uint16)
    logits = _c(logits, np.float32)
    T, H = x.shape
    E = logits.shape[1]
    I = gu[0].shape[1] // 2
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    out = np.empty((T, H), np.float64)
    a = [_c(gu[0], np.uint8), _c(gu[1], np.uint8), _c(gu[2], np.float32),
         _c(dn[0], np.uint8), _c(dn[1], np.uint8), _c(dn[2], np.float32)]
    _load().oracle_layer(_ptr(x), _ptr(logits), *[_ptr(v) for v in a], T, H, I, E, k,
                         _ptr(ids), _ptr(w), _ptr(out))
    return out, ids, w


def layer_rows(x_bf16, ids, w, gu, dn, rows):
    """Layer output for a subset of tokens, given the routing. -> out f64 [len(rows), H]."""
    x = _c(x_bf16, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float64)
    rows = _c(rows, np.int32)
    T, H = x.shape
    k = ids.shape[1]
    I = gu[0].shape[1] // 2
    out = np.empty((len(rows), H), np.float64)
    a = [_c(gu[0], np.uint8), _c(gu[1], np.uint8), _c(gu[2], np.float32),
         _c(dn[0], np.uint8), _c(dn[1], np.uint8), _c(dn[2], np.float32)]
    _load().oracle_layer_rows(_ptr(x), _ptr(ids), _ptr(w), *[_ptr(v) for v in a], H, I, k,
                              _ptr(rows), len(rows), _ptr(out))
    return out


def shared_rows(x_bf16, sgu, sdn, rows):
    """Shared-expert output y_shared for a subset of tokens (f64 [len(rows), H]):
    the same SwiGLU FFN as a routed expert's (h rounded to bf16), on a one-expert
    matrix, with weight 1 -- i.e. layer_rows with every token routed to expert 0."""
    x = _c(x_bf16, np.uint16)
    T = x.shape[0]
    return layer_rows(x, np.zeros((T, 1), np.int32), np.ones((T, 1), np.float64), sgu, sdn, rows)


# ------------------------------------------------- W4A4 (NVFP4 activations)
def e4m3_rne(v: float) -> int:
    """fp32 value in [0, 448] -> nearest E4M3 code, ties to the even mantissa."""
    return int(_load().oracle_e4m3_rne(float(v)))


def e2m1_rne(v: float) -> int:
    """fp32 value -> nearest E2M1 code (sign bit 3), ties to even, saturating at +-6."""
    return int(_load().oracle_e2m1_rne(float(v)))


def quant_nvfp4(v) -> tuple:
    """fp32 rows [..., n] (n % 16 == 0) -> (codes uint8 [..., n/2], E4M3 scales uint8 [..., n/16]):
    per 16 elements s = RNE_e4m3(min(amax/6, 448)) (amax/6 in fp32), codes RNE_e2m1 of the exact
    quotient v / e4m3(s)."""
    a = _c(v, np.float32)
    shp = a.shape
    n = shp[-1]
    flat = a.reshape(-1, n)
    codes = np.empty((flat.shape[0], n // 2), np.uint8)
    scales = np.empty((flat.shape[0], n // 16), np.uint8)
    lib = _load()
    for r in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[r])
        c = np.empty(n // 2, np.uint8)
        sc = np.empty(n // 16, np.uint8)
        lib.oracle_quant_nvfp4(_ptr(row), n, _ptr(c), _ptr(sc))
        codes[r], scales[r] = c, sc
    return codes.reshape(shp[:-1] + (n // 2,)), scales.reshape(shp[:-1] + (n // 16,))


def w4a4_layer_rows(x_bf16, ids, w, gu, dn, rows):
    """The W4A4 layer (x and h quantized to NVFP4, fp64 products) for a subset of tokens,
    given the routing. -> out f64 [len(rows), H]."""
    x = _c(x_bf16, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float64)
    rows = _c(rows, np.int32)
    T, H = x.shape
    k = ids.shape[1]
    I = gu[0].shape[1] // 2
    out = np.empty((len(rows), H), np.float64)
    a = [_c(gu[0], np.uint8), _c(gu[1], np.uint8), _c(gu[2], np.float32),
         _c(dn[0], np.uint8), _c(dn[1], np.uint8), _c(dn[2], np.float32)]
    _load().oracle_w4a4_layer_rows(_ptr(x), _ptr(ids), _ptr(w), *[_ptr(v) for v in a], H, I, k,
                                   _ptr(rows), len(rows), _ptr(out))
    return out
