"""CPU oracle of the MXFP4 routed-expert MoE layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and this package never
imports the product path.  The two share only the seeded input generators.

The arithmetic lives in ``moe_oracle.c`` (plain C, float32-exact decode, double
arithmetic); this module only builds that file with gcc and marshals numpy
arrays into it with ctypes.  Each function cites the passage it follows:

* MXFP4 decode and size -- "DeepSeek-V4-Flash on a four-GPU Ampere
  workstation", section "MXFP4 is not NVFP4, and the difference matters on
  Ampere".
* SwiGLU experts, weighted reduction, shared experts, routing as IDs + weights,
  and the sigmoid + bias routing variant -- "Cascadia: Resident 975B MoE
  Inference on Eleven AI PCs" §3.1 and Eq. (1) of §3.3.
* Dense FFN as all-active slices -- same paper, §3.4, Eq. (2).
* Group-32 INT4 weights with FP16 group scales and zero points -- same paper,
  §3.1 (the exporter's packed nibbles and FP16 group scales) and §3.5 (scale
  and zero-point overhead in the expert bytes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off keeps every double operation a separately rounded IEEE
# operation on both x86-64 and aarch64 (gcc would otherwise fuse a*b+c).
GCC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off"]


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into libmoe_oracle.so next to it (gcc)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *GCC_FLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Layer(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int), ("inter", ctypes.c_int), ("n_experts", ctypes.c_int),
        ("n_shared", ctypes.c_int), ("weight_format", ctypes.c_int),
        ("gu_codes", ctypes.POINTER(ctypes.c_void_p)), ("gu_scales", ctypes.POINTER(ctypes.c_void_p)),
        ("d_codes", ctypes.POINTER(ctypes.c_void_p)), ("d_scales", ctypes.POINTER(ctypes.c_void_p)),
        ("gu_zeros", ctypes.POINTER(ctypes.c_void_p)), ("d_zeros", ctypes.POINTER(ctypes.c_void_p)),
    ]

_FORMATS = {"mxfp4": 0, "bf16": 1, "int4g32": 2}


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            L.oracle_e2m1_value.argtypes = [ci]
            L.oracle_e2m1_value.restype = ctypes.c_double
            L.oracle_mx_value.argtypes = [ci, ci]
            L.oracle_mx_value.restype = ctypes.c_float
            L.oracle_mx_bytes.argtypes = [i64, i64]
            L.oracle_mx_bytes.restype = i64
            L.oracle_mx_decode.argtypes = [vp, vp, i64, i64, vp]
            L.oracle_mx_decode.restype = ci
            L.oracle_bf16_decode.argtypes = [vp, i64, vp]
            L.oracle_bf16_decode.restype = None
            L.oracle_fp16_value.argtypes = [ci]
            L.oracle_fp16_value.restype = ctypes.c_double
            L.oracle_i4_value.argtypes = [ci, ci, ci]
            L.oracle_i4_value.restype = ctypes.c_float
            L.oracle_i4_bytes.argtypes = [i64, i64, ci]
            L.oracle_i4_bytes.restype = i64
            L.oracle_i4_decode.argtypes = [vp, vp, vp, i64, i64, vp]
            L.oracle_i4_decode.restype = ci
            L.oracle_route.argtypes = [vp, i64, ci, ci, vp, vp]
            L.oracle_route.restype = None
            L.oracle_route_sigmoid.argtypes = [vp, vp, i64, ci, ci, ctypes.c_double, vp, vp]
            L.oracle_route_sigmoid.restype = None
            L.oracle_permute.argtypes = [vp, i64, ci, ci, vp, vp, vp]
            L.oracle_permute.restype = None
            L.oracle_swiglu_ffn.argtypes = [vp, vp, i64, vp, i64, ci, ci, vp, vp]
            L.oracle_swiglu_ffn.restype = None
            L.oracle_moe_layer.argtypes = [ctypes.POINTER(_Layer), vp, vp, i64, ci, ci, vp, vp, vp]
            L.oracle_moe_layer.restype = ci
            L.oracle_moe_layer_routed.argtypes = [ctypes.POINTER(_Layer), vp, vp, vp, i64, ci, ci, vp]
            L.oracle_moe_layer_routed.restype = ci
            L.oracle_dense_ffn.argtypes = [ci, vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, vp, i64, ci, vp]
            L.oracle_dense_ffn.restype = ci
            _lib = L
    return _lib


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ decode

def e2m1_value(code: int) -> float:
    """v(c) of a 4-bit E2M1 code (bit 3 = sign)."""
    return lib().oracle_e2m1_value(int(code))


def mx_value(code: int, e8m0: int) -> float:
    """v(c) * 2^(e-127) rounded to float32."""
    return lib().oracle_mx_value(int(code), int(e8m0))


def mx_bytes(rows: int, cols: int) -> int:
    """Bytes of an MXFP4 matrix [rows, cols]: codes plus one scale per 32 values."""
    return int(lib().oracle_mx_bytes(rows, cols))


def mx_decode(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Decode MXFP4 codes [rows, cols/2] + scales [rows, cols/32] to float32 [rows, cols]."""
    codes, scales = _c(codes, np.uint8), _c(scales, np.uint8)
    rows, cols = codes.shape[0], codes.shape[1] * 2
    assert scales.shape == (rows, cols // 32)
    out = np.empty((rows, cols), np.float32)
    rc = lib().oracle_mx_decode(_p(codes), _p(scales), rows, cols, _p(out))
    if rc != 0:
        raise ValueError("E8M0 scale 255 (NaN) in MXFP4 matrix")
    return out


def fp16_value(bits: int) -> float:
    """IEEE binary16 bit pattern to its value (double)."""
    return lib().oracle_fp16_value(int(bits))


def i4_value(q: int, z: int, scale_bits: int) -> float:
    """Group-32 INT4 weight s * (q - z) rounded to float32 (exact)."""
    return lib().oracle_i4_value(int(q), int(z), int(scale_bits))


def i4_bytes(rows: int, cols: int, zero_points: bool = True) -> int:
    """Bytes of a group-32 INT4 matrix [rows, cols]: codes, FP16 scales, zero points."""
    return int(lib().oracle_i4_bytes(rows, cols, 1 if zero_points else 0))


def i4_decode(codes: np.ndarray, scales: np.ndarray, zeros: np.ndarray | None = None) -> np.ndarray:
    """Decode group-32 INT4 codes [rows, cols/2] + FP16 scale bits [rows, cols/32]
    + zero points [rows, cols/32] (None: all 8) to float32 [rows, cols]."""
    codes, scales = _c(codes, np.uint8), _c(scales, np.uint16)
    rows, cols = codes.shape[0], codes.shape[1] * 2
    assert scales.shape == (rows, cols // 32)
    if zeros is not None:
        zeros = _c(zeros, np.uint8)
        assert zeros.shape == scales.shape
    out = np.empty((rows, cols), np.float32)
    if lib().oracle_i4_decode(_p(codes), _p(scales), _p(zeros), rows, cols, _p(out)) != 0:
        raise ValueError("non-finite FP16 scale or zero point above 15 in INT4 matrix")
    return out


def bf16_decode(bits: np.ndarray) -> np.ndarray:
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float32)
    lib().oracle_bf16_decode(_p(bits), bits.size, _p(out))
    return out


# ------------------------------------------------------------------ routing

def route(logits: np.ndarray, k: int):
    """Softmax top-k with renormalisation: returns ids int32 [T, k], w float64 [T, k]."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    lib().oracle_route(_p(logits), T, E, k, _p(ids), _p(w))
    return ids, w


def route_sigmoid(logits: np.ndarray, bias: np.ndarray | None, k: int, scale: float = 1.0):
    """Sigmoid scores, bias-adjusted top-k selection, weights normalised over the
    selected experts times scale ("Cascadia: Resident 975B MoE Inference on
    Eleven AI PCs" §3.1): returns ids int32 [T, k], w float64 [T, k]."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    if bias is not None:
        bias = _c(bias, np.float32)
        assert bias.shape == (E,)
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    lib().oracle_route_sigmoid(_p(logits), _p(bias), T, E, k, float(scale), _p(ids), _p(w))
    return ids, w


def permute(ids: np.ndarray, n_experts: int):
    """Stable counting sort of slots by expert: (off [E+1], sorted_slot [T*k], slot_pos [T*k])."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    off = np.empty(n_experts + 1, np.int32)
    ss = np.empty(T * k, np.int32)
    sp = np.empty(T * k, np.int32)
    lib().oracle_permute(_p(ids), T, k, n_experts, _p(off), _p(ss), _p(sp))
    return off, ss, sp


# ------------------------------------------------------------------ FFN / layer

def swiglu_ffn(Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray, x: np.ndarray) -> np.ndarray:
    """One SwiGLU FFN on one token in double: Wg, Wu [I, H], Wd [H, I] float32, x [H] float64."""
    Wg, Wu, Wd = _c(Wg, np.float32), _c(Wu, np.float32), _c(Wd, np.float32)
    I, H = Wg.shape
    assert Wu.shape == (I, H) and Wd.shape == (H, I)
    x = _c(x, np.float64)
    y = np.empty(H, np.float64)
    # gate and up need one common row stride: pass Wu as its own matrix with the same stride H
    lib().oracle_swiglu_ffn(_p(Wg), _p(Wu), H, _p(Wd), I, H, I, _p(x), _p(y))
    return y


class OracleWeights:
    """Host weights of an MoE layer, any subset of experts may be None.

    weight_format: "mxfp4" (codes + E8M0 scales), "bf16" (bits) or "int4g32"
    (codes + FP16 scale bits + optional zero points)."""

    def __init__(self, hidden: int, inter: int, n_experts: int, n_shared: int, weight_format: str = "mxfp4"):
        assert weight_format in _FORMATS
        self.hidden, self.inter, self.n_experts, self.n_shared = hidden, inter, n_experts, n_shared
        self.weight_format = weight_format
        n = n_experts + n_shared
        self.gu_codes = [None] * n
        self.gu_scales = [None] * n
        self.d_codes = [None] * n
        self.d_scales = [None] * n
        self.gu_zeros = [None] * n
        self.d_zeros = [None] * n

    def set_expert(self, e: int, gu_codes, gu_scales, d_codes, d_scales, gu_zeros=None, d_zeros=None):
        if self.weight_format == "bf16":
            self.gu_codes[e], self.d_codes[e] = _c(gu_codes, np.uint16), _c(d_codes, np.uint16)
            return
        sdt = np.uint16 if self.weight_format == "int4g32" else np.uint8
        self.gu_codes[e], self.gu_scales[e] = _c(gu_codes, np.uint8), _c(gu_scales, sdt)
        self.d_codes[e], self.d_scales[e] = _c(d_codes, np.uint8), _c(d_scales, sdt)
        if self.weight_format == "int4g32":
            self.gu_zeros[e] = None if gu_zeros is None else _c(gu_zeros, np.uint8)
            self.d_zeros[e] = None if d_zeros is None else _c(d_zeros, np.uint8)

    def _layer(self):
        """The C layer descriptor and the pointer arrays it refers to (keep both alive)."""
        ne = self.n_experts + self.n_shared
        arr = lambda lst: (ctypes.c_void_p * ne)(*[(None if a is None else a.ctypes.data) for a in lst])
        keep = [arr(self.gu_codes), arr(self.gu_scales), arr(self.d_codes), arr(self.d_scales), arr(self.gu_zeros),
                arr(self.d_zeros)]
        cast = lambda a: ctypes.cast(a, ctypes.POINTER(ctypes.c_void_p))
        L = _Layer(self.hidden, self.inter, self.n_experts, self.n_shared, _FORMATS[self.weight_format],
                   *(cast(a) for a in keep))
        return L, keep


def moe_layer(W: OracleWeights, x_bf16: np.ndarray, logits: np.ndarray, k: int, nthreads: int = 1):
    """The routed MoE layer on the given tokens: returns (out float64 [n, H], ids [n, k], w [n, k])."""
    x_bf16 = _c(x_bf16, np.uint16)
    logits = _c(logits, np.float32)
    n, H = x_bf16.shape
    assert H == W.hidden and logits.shape == (n, W.n_experts)
    L, _keep = W._layer()
    out = np.empty((n, H), np.float64)
    ids = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float64)
    rc = lib().oracle_moe_layer(ctypes.byref(L), _p(x_bf16), _p(logits), n, k, nthreads, _p(out), _p(ids), _p(w))
    if rc != 0:
        raise ValueError(f"oracle_moe_layer failed with {rc}")
    return out, ids, w


def moe_layer_routed(W: OracleWeights, x_bf16: np.ndarray, ids: np.ndarray, w: np.ndarray, nthreads: int = 1):
    """The MoE layer for given routing (ids [n, k] in [0, E) or -1, weights [n, k]):
    every selected and shared expert on its tokens and the weighted reduction
    ("Cascadia" §3.1, Eq. (1) of §3.3; the routing reaches it as ids and weights).
    An id of -1 is an empty slot: its term is left out of the sum, so that
    holders of disjoint expert subsets each compute their part of Eq. (1).
    Returns out float64 [n, H]."""
    x_bf16 = _c(x_bf16, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float64)
    n, H = x_bf16.shape
    k = ids.shape[1]
    assert H == W.hidden and ids.shape == (n, k) and w.shape == (n, k)
    L, _keep = W._layer()
    out = np.empty((n, H), np.float64)
    rc = lib().oracle_moe_layer_routed(ctypes.byref(L), _p(x_bf16), _p(ids), _p(w), n, k, nthreads, _p(out))
    if rc != 0:
        raise ValueError(f"oracle_moe_layer_routed failed with {rc}")
    return out


def dense_ffn(weights, x_bf16: np.ndarray, n_slices: int = 0, weight_format: str = "mxfp4") -> np.ndarray:
    """Dense SwiGLU FFN on the given tokens, unsliced (n_slices=0) or as a sum of slices.

    weights: MXFP4 ((g_codes, g_scales), (u_codes, u_scales), (d_codes, d_scales)),
    BF16 bits (W_g [I, H], W_u [I, H], W_d [H, I]), or group-32 INT4
    ((g_codes, g_scales, g_zeros), (u_...), (d_...)) with FP16 scale bits and
    zero points (None: all 8).
    """
    x_bf16 = _c(x_bf16, np.uint16)
    n, H = x_bf16.shape
    gz = uz = dz = None
    if weight_format == "bf16":
        g, u, d = (_c(a, np.uint16) for a in weights)
        gs = us = ds = None
    elif weight_format == "int4g32":
        (g, gs, gz), (u, us, uz), (d, ds, dz) = (
            (_c(a, np.uint8), _c(b, np.uint16), None if z is None else _c(z, np.uint8)) for a, b, z in weights)
    else:
        (g, gs), (u, us), (d, ds) = ((_c(a, np.uint8), _c(b, np.uint8)) for a, b in weights)
    I = g.shape[0]
    out = np.empty((n, H), np.float64)
    rc = lib().oracle_dense_ffn(_FORMATS[weight_format], _p(g), _p(gs), _p(gz), _p(u), _p(us), _p(uz), _p(d), _p(ds),
                                _p(dz), H, I, n_slices, _p(x_bf16), n, 1, _p(out))
    if rc != 0:
        raise ValueError(f"oracle_dense_ffn failed with {rc}")
    return out
