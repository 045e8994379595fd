"""CPU oracle for the MoE layer hot path -- test infrastructure only.

The oracle is the plain C++17 program in ``moe_oracle.cpp`` (FP64 sums,
one BF16 round-to-nearest-even at each store boundary), loaded here through
ctypes over numpy arrays.  BF16 tensors travel as ``numpy.uint16`` bit patterns.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library never calls it and
shares no code with it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

ACT_SWIGLU = 0
ACT_RELU2 = 1

ST_OK = 0
ST_INVALID_ARG = 1
ST_INVALID_ROUTE = 2
ST_CAPACITY = 3
ST_NONFINITE = 4


def variant(lib_path: str, src_path: str):
    """A second instance of this module bound to another build of the oracle
    (used by the test that plants mistakes in copies of the oracle source)."""
    import importlib.util
    spec = importlib.util.spec_from_file_location(f"oracle_variant_{abs(hash(lib_path))}", __file__)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._LIB_PATH = lib_path
    mod._SRC = src_path
    mod._lib = None
    return mod


def build(force: bool = False) -> str:
    """Compile the oracle with the host C++ compiler (no CUDA involved)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-std=c++17", "-O2", "-fPIC", "-shared",
                               "-o", tmp, _SRC])
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
            lib.oracle_bf16_from_double.restype = ctypes.c_uint16
            lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
            lib.oracle_double_from_bf16.restype = ctypes.c_double
            lib.oracle_double_from_bf16.argtypes = [ctypes.c_uint16]
            lib.oracle_route.restype = i
            lib.oracle_route.argtypes = [i, i, i, P, P, P]
            lib.oracle_route_sigmoid.restype = i
            lib.oracle_route_sigmoid.argtypes = [i, i, i, P, P, ctypes.c_float, P, P]
            lib.oracle_gate.restype = None
            lib.oracle_gate.argtypes = [i, i, i, P, P, P]
            lib.oracle_dispatch.restype = i
            lib.oracle_dispatch.argtypes = [i, i, i, i, i, P, P, P, P, P, P, P]
            lib.oracle_expert_up.restype = None
            lib.oracle_expert_up.argtypes = [i, i, i, P, P, P]
            lib.oracle_expert_down_acc.restype = None
            lib.oracle_expert_down_acc.argtypes = [i, i, P, P, P]
            lib.oracle_expert_row.restype = None
            lib.oracle_expert_row.argtypes = [i, i, i, P, P, P, P, P]
            lib.oracle_shared_row.restype = None
            lib.oracle_shared_row.argtypes = [i, i, i, i, P, P, P, P, P]
            lib.oracle_expert_ffn.restype = None
            lib.oracle_expert_ffn.argtypes = [i, i, i, i, i, i, i] + [P] * 11
            lib.oracle_combine_row.restype = None
            lib.oracle_combine_row.argtypes = [i, i, P, P, P, P, P, P]
            lib.oracle_combine.restype = None
            lib.oracle_combine.argtypes = [i, i, i, P, P, P, P, P, P]
            lib.oracle_layer.restype = i
            lib.oracle_layer.argtypes = [i] * 9 + [P] * 20
            lib.oracle_fp8_e4m3_decode.restype = None
            lib.oracle_fp8_e4m3_decode.argtypes = [i, P, P]
            lib.oracle_expert_ffn_fp8.restype = None
            lib.oracle_expert_ffn_fp8.argtypes = [i, i, i, i] + [P] * 8
            lib.oracle_layer_fp8.restype = i
            lib.oracle_layer_fp8.argtypes = [i] * 7 + [P] * 19
            lib.oracle_fp4_e2m1_decode.restype = None
            lib.oracle_fp4_e2m1_decode.argtypes = [i, P, P]
            lib.oracle_expert_ffn_nvfp4.restype = None
            lib.oracle_expert_ffn_nvfp4.argtypes = [i, i, i, i] + [P] * 10
            lib.oracle_layer_nvfp4.restype = i
            lib.oracle_layer_nvfp4.argtypes = [i] * 7 + [P] * 21
            _lib = lib
    return _lib


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "oracle wants C-contiguous numpy arrays"
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- scalar helpers -------------------------------------------------------
def bf16_from_double(d: float) -> int:
    return int(_load().oracle_bf16_from_double(float(d)))


def double_from_bf16(b: int) -> float:
    return float(_load().oracle_double_from_bf16(int(b)))


def up(act):
    return 2 if act == ACT_SWIGLU else 1


# ---- the five calls -------------------------------------------------------
def route(logits: np.ndarray, k: int):
    """-> (status, ids int32 [T,k], w float32 [T,k])."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    st = _load().oracle_route(T, E, k, _p(logits), _p(ids), _p(w))
    return st, ids, w


def route_sigmoid(logits: np.ndarray, k: int, bias=None, route_scale: float = 1.0):
    """Sigmoid routing with a selection-only bias -> (status, ids, w)."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    b = None if bias is None else _c(bias, np.float32)
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    st = _load().oracle_route_sigmoid(T, E, k, _p(logits), _p(b), float(route_scale), _p(ids), _p(w))
    return st, ids, w


def gate(x: np.ndarray, wg: np.ndarray) -> np.ndarray:
    """logits f32 [T,E] = x [T,H] . Wg [E,H]^T (BF16 bits in)."""
    x = _c(x, np.uint16)
    wg = _c(wg, np.uint16)
    T, H = x.shape
    E = wg.shape[0]
    out = np.zeros((T, E), np.float32)
    _load().oracle_gate(T, H, E, _p(x), _p(wg), _p(out))
    return out


def dispatch(ids: np.ndarray, x: np.ndarray, E: int, capacity: int):
    """-> (status, counts, offsets, dest, sorted_pair, x_perm).  Unwritten
    entries of dest / sorted_pair / x_perm keep the fill value -7 / -7 / 0."""
    ids = _c(ids, np.int32)
    x = _c(x, np.uint16)
    T, k = ids.shape
    H = x.shape[1]
    R = T * k
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    dest = np.full(R, -7, np.int32)
    sorted_pair = np.full(R, -7, np.int32)
    x_perm = np.zeros((R, H), np.uint16)
    st = _load().oracle_dispatch(T, E, k, H, capacity, _p(ids), _p(x), _p(counts), _p(offsets),
                                 _p(dest), _p(sorted_pair), _p(x_perm))
    return st, counts, offsets, dest, sorted_pair, x_perm


def expert_ffn(x_perm, offsets, w13, w2, act, x=None, ws13=None, ws2=None, S=0, Is=0):
    """-> (h [R,I], y_perm [R,H], h_shared [T,S*Is] or None, y_shared [T,H] or None)."""
    x_perm = _c(x_perm, np.uint16)
    offsets = _c(offsets, np.int32)
    w13 = _c(w13, np.uint16)
    w2 = _c(w2, np.uint16)
    E, H, I = w2.shape
    R = x_perm.shape[0]
    h = np.zeros((R, I), np.uint16)
    y = np.zeros((R, H), np.uint16)
    T = 0
    hs = ys = None
    if S > 0:
        x = _c(x, np.uint16)
        ws13 = _c(ws13, np.uint16)
        ws2 = _c(ws2, np.uint16)
        T = x.shape[0]
        hs = np.zeros((T, S * Is), np.uint16)
        ys = np.zeros((T, H), np.uint16)
    _load().oracle_expert_ffn(T, H, E, I, act, S, Is, _p(x_perm), _p(offsets), _p(w13), _p(w2),
                              _p(x), _p(ws13), _p(ws2), _p(h), _p(y), _p(hs), _p(ys))
    return h, y, hs, ys


def expert_row(x_row, w13_e, w2_e, act):
    """One routed row: -> (h_row [I], y_row [H])."""
    x_row = _c(x_row, np.uint16)
    w13_e = _c(w13_e, np.uint16)
    w2_e = _c(w2_e, np.uint16)
    H, I = w2_e.shape
    h = np.zeros(I, np.uint16)
    y = np.zeros(H, np.uint16)
    _load().oracle_expert_row(H, I, act, _p(x_row), _p(w13_e), _p(w2_e), _p(h), _p(y))
    return h, y


def shared_row(x_row, ws13, ws2, act):
    """Shared experts on one token row: -> (h_shared_row [S*Is], y_shared_row [H])."""
    x_row = _c(x_row, np.uint16)
    ws13 = _c(ws13, np.uint16)
    ws2 = _c(ws2, np.uint16)
    S, H, Is = ws2.shape
    h = np.zeros(S * Is, np.uint16)
    y = np.zeros(H, np.uint16)
    _load().oracle_shared_row(H, Is, S, act, _p(x_row), _p(ws13), _p(ws2), _p(h), _p(y))
    return h, y


def combine(y_perm, dest, w, y_shared=None, residual=None):
    y_perm = _c(y_perm, np.uint16)
    dest = _c(dest, np.int32).reshape(-1)
    w = _c(w, np.float32)
    T, k = w.shape
    H = y_perm.shape[1]
    out = np.zeros((T, H), np.uint16)
    ys = None if y_shared is None else _c(y_shared, np.uint16)
    res = None if residual is None else _c(residual, np.uint16)
    _load().oracle_combine(T, k, H, _p(y_perm), _p(dest), _p(w), _p(ys), _p(res), _p(out))
    return out


def combine_row(y_perm, dest_t, w_t, y_shared_t=None, residual_t=None):
    y_perm = _c(y_perm, np.uint16)
    dest_t = _c(dest_t, np.int32)
    w_t = _c(w_t, np.float32)
    H = y_perm.shape[1]
    out = np.zeros(H, np.uint16)
    ys = None if y_shared_t is None else _c(y_shared_t, np.uint16)
    res = None if residual_t is None else _c(residual_t, np.uint16)
    _load().oracle_combine_row(len(w_t), H, _p(y_perm), _p(dest_t), _p(w_t), _p(ys), _p(res), _p(out))
    return out


def layer(x, w13, w2, act, k, capacity, logits=None, ids_in=None, w_in=None,
          ws13=None, ws2=None, residual=None):
    """The whole layer; returns a dict with every intermediate and 'status'."""
    x = _c(x, np.uint16)
    w13 = _c(w13, np.uint16)
    w2 = _c(w2, np.uint16)
    T, H = x.shape
    E, _, I = w2.shape
    S = Is = 0
    if ws2 is not None:
        ws13 = _c(ws13, np.uint16)
        ws2 = _c(ws2, np.uint16)
        S, _, Is = ws2.shape
    R = T * k
    o = dict(ids=np.zeros((T, k), np.int32), w=np.zeros((T, k), np.float32),
             counts=np.zeros(E, np.int32), offsets=np.zeros(E + 1, np.int32),
             dest=np.full(R, -7, np.int32), sorted_pair=np.full(R, -7, np.int32),
             x_perm=np.zeros((R, H), np.uint16), h=np.zeros((R, I), np.uint16),
             y_perm=np.zeros((R, H), np.uint16),
             h_shared=np.zeros((T, max(S * Is, 1)), np.uint16),
             y_shared=np.zeros((T, H), np.uint16), out=np.zeros((T, H), np.uint16))
    lg = None if logits is None else _c(logits, np.float32)
    ii = None if ids_in is None else _c(ids_in, np.int32)
    wi = None if w_in is None else _c(w_in, np.float32)
    res = None if residual is None else _c(residual, np.uint16)
    st = _load().oracle_layer(T, H, E, k, I, act, S, Is, capacity, _p(lg), _p(ii), _p(wi), _p(x),
                              _p(w13), _p(w2), _p(ws13), _p(ws2), _p(res), _p(o["ids"]), _p(o["w"]),
                              _p(o["counts"]), _p(o["offsets"]), _p(o["dest"]), _p(o["sorted_pair"]),
                              _p(o["x_perm"]), _p(o["h"]), _p(o["y_perm"]), _p(o["h_shared"]),
                              _p(o["y_shared"]), _p(o["out"]))
    o["status"] = st
    return o


# ---- FP8 E4M3 expert weights ----------------------------------------------
def fp8_e4m3_decode(codes):
    """E4M3 codes (uint8) -> float64 values (NaN for the two NaN codes)."""
    c = _c(codes, np.uint8)
    out = np.zeros(c.shape, np.float64)
    _load().oracle_fp8_e4m3_decode(int(c.size), _p(c), _p(out))
    return out


def expert_ffn_fp8(x_perm, offsets, w13, s13, w2, s2, act):
    """Routed experts with FP8 E4M3 weights and one FP32 scale per weight row:
    w13 uint8 [E, up, H], s13 float32 [E, up], w2 uint8 [E, H, I], s2 float32 [E, H].
    -> (h [R, I], y_perm [R, H]) as BF16 bits."""
    x_perm = _c(x_perm, np.uint16)
    offsets = _c(offsets, np.int32)
    w13 = _c(w13, np.uint8)
    w2 = _c(w2, np.uint8)
    s13 = _c(s13, np.float32)
    s2 = _c(s2, np.float32)
    E, H, I = w2.shape
    R = x_perm.shape[0]
    h = np.zeros((R, I), np.uint16)
    y = np.zeros((R, H), np.uint16)
    _load().oracle_expert_ffn_fp8(H, E, I, act, _p(x_perm), _p(offsets), _p(w13), _p(s13), _p(w2), _p(s2),
                                  _p(h), _p(y))
    return h, y


def layer_fp8(x, w13, s13, w2, s2, act, k, capacity, logits=None, ids_in=None, w_in=None, residual=None):
    """The whole layer with FP8 E4M3 expert weights (no shared experts)."""
    x = _c(x, np.uint16)
    w13 = _c(w13, np.uint8)
    w2 = _c(w2, np.uint8)
    s13 = _c(s13, np.float32)
    s2 = _c(s2, np.float32)
    T, H = x.shape
    E, _, I = w2.shape
    R = T * k
    o = dict(ids=np.zeros((T, k), np.int32), w=np.zeros((T, k), np.float32),
             counts=np.zeros(E, np.int32), offsets=np.zeros(E + 1, np.int32),
             dest=np.full(R, -7, np.int32), sorted_pair=np.full(R, -7, np.int32),
             x_perm=np.zeros((R, H), np.uint16), h=np.zeros((R, I), np.uint16),
             y_perm=np.zeros((R, H), np.uint16), out=np.zeros((T, H), np.uint16))
    lg = None if logits is None else _c(logits, np.float32)
    ii = None if ids_in is None else _c(ids_in, np.int32)
    wi = None if w_in is None else _c(w_in, np.float32)
    res = None if residual is None else _c(residual, np.uint16)
    st = _load().oracle_layer_fp8(T, H, E, k, I, act, capacity, _p(lg), _p(ii), _p(wi), _p(x), _p(w13), _p(s13),
                                  _p(w2), _p(s2), _p(res), _p(o["ids"]), _p(o["w"]), _p(o["counts"]),
                                  _p(o["offsets"]), _p(o["dest"]), _p(o["sorted_pair"]), _p(o["x_perm"]),
                                  _p(o["h"]), _p(o["y_perm"]), _p(o["out"]))
    o["status"] = st
    return o


# ---- NVFP4 expert weights ---------------------------------------------------
def fp4_e2m1_decode(codes):
    """E2M1 codes (uint8, low 4 bits) -> float64 values."""
    c = _c(codes, np.uint8)
    out = np.zeros(c.shape, np.float64)
    _load().oracle_fp4_e2m1_decode(int(c.size), _p(c), _p(out))
    return out


def expert_ffn_nvfp4(x_perm, offsets, w13, b13, s13, w2, b2, s2, act):
    """Routed experts with NVFP4 weights: w13 uint8 [E, up, H/2] (two E2M1 per
    byte, low nibble first), b13 uint8 [E, up, 16*ceil(H/256)] E4M3 block
    scales (byte j scales elements 16j..16j+15; the rest is padding), s13
    float32 [E, up] row scales; w2 [E, H, I/2], b2 [E, H, 16*ceil(I/256)],
    s2 [E, H].  -> (h [R, I], y_perm [R, H]) as BF16 bits."""
    x_perm = _c(x_perm, np.uint16)
    offsets = _c(offsets, np.int32)
    w13, b13, w2, b2 = (_c(a, np.uint8) for a in (w13, b13, w2, b2))
    s13 = _c(s13, np.float32)
    s2 = _c(s2, np.float32)
    E, H, I2 = w2.shape
    I = 2 * I2
    R = x_perm.shape[0]
    h = np.zeros((R, I), np.uint16)
    y = np.zeros((R, H), np.uint16)
    _load().oracle_expert_ffn_nvfp4(H, E, I, act, _p(x_perm), _p(offsets), _p(w13), _p(b13), _p(s13), _p(w2),
                                    _p(b2), _p(s2), _p(h), _p(y))
    return h, y


def layer_nvfp4(x, w13, b13, s13, w2, b2, s2, act, k, capacity, logits=None, ids_in=None, w_in=None,
                residual=None):
    """The whole layer with NVFP4 expert weights (no shared experts)."""
    x = _c(x, np.uint16)
    w13, b13, w2, b2 = (_c(a, np.uint8) for a in (w13, b13, w2, b2))
    s13 = _c(s13, np.float32)
    s2 = _c(s2, np.float32)
    T, H = x.shape
    E, _, I2 = w2.shape
    I = 2 * I2
    R = T * k
    o = dict(ids=np.zeros((T, k), np.int32), w=np.zeros((T, k), np.float32),
             counts=np.zeros(E, np.int32), offsets=np.zeros(E + 1, np.int32),
             dest=np.full(R, -7, np.int32), sorted_pair=np.full(R, -7, np.int32),
             x_perm=np.zeros((R, H), np.uint16), h=np.zeros((R, I), np.uint16),
             y_perm=np.zeros((R, H), np.uint16), out=np.zeros((T, H), np.uint16))
    lg = None if logits is None else _c(logits, np.float32)
    ii = None if ids_in is None else _c(ids_in, np.int32)
    wi = None if w_in is None else _c(w_in, np.float32)
    res = None if residual is None else _c(residual, np.uint16)
    st = _load().oracle_layer_nvfp4(T, H, E, k, I, act, capacity, _p(lg), _p(ii), _p(wi), _p(x), _p(w13),
                                    _p(b13), _p(s13), _p(w2), _p(b2), _p(s2), _p(res), _p(o["ids"]), _p(o["w"]),
                                    _p(o["counts"]), _p(o["offsets"]), _p(o["dest"]), _p(o["sorted_pair"]),
                                    _p(o["x_perm"]), _p(o["h"]), _p(o["y_perm"]), _p(o["out"]))
    o["status"] = st
    return o
