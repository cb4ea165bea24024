"""CPU oracle of the routed-expert block -- TEST INFRASTRUCTURE ONLY.

The oracle is the slow, plain C++ double-precision checker (``smoe_oracle.cpp``) that the CUDA library is compared
against.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline / reference legs may import
this package.  The product path never routes through it; it shares no code with the CUDA library.

Every function here only marshals numpy arrays into the C++ functions; the arithmetic lives in the C++ file, whose
header lists the page passages it follows and the readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "smoe_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

def build(force: bool = False) -> str:
    """Compile the oracle with g++ (no fused multiply-add contraction, so the fp32 q8 rule is exact IEEE)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread",
               "-o", tmp, _SRC]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _P(t):
    return ctypes.POINTER(t)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            i64, i32, c_int = ctypes.c_int64, ctypes.c_int32, ctypes.c_int
            vp = ctypes.c_void_p
            L.oracle_f2h.argtypes = [ctypes.c_float]
            L.oracle_f2h.restype = ctypes.c_uint16
            L.oracle_h2f.argtypes = [ctypes.c_uint16]
            L.oracle_h2f.restype = ctypes.c_float
            L.oracle_route.argtypes = [vp, i64, c_int, c_int, vp, vp, c_int]
            L.oracle_group.argtypes = [vp, i64, c_int, c_int, vp, vp, vp, vp]
            L.oracle_group.restype = c_int
            L.oracle_quantize_q8.argtypes = [vp, i64, i64, vp, vp, c_int]
            L.oracle_gateup.argtypes = [vp, vp, vp, vp, c_int, vp, vp, c_int, c_int, vp, c_int]
            L.oracle_swiglu_requant.argtypes = [vp, i64, c_int, vp, vp, c_int]
            L.oracle_swiglu_requant_f32.argtypes = [vp, i64, c_int, vp, vp, c_int]
            L.oracle_down.argtypes = [vp, vp, vp, c_int, vp, vp, c_int, c_int, vp, c_int]
            L.oracle_combine.argtypes = [vp, vp, vp, i64, c_int, c_int, vp, c_int]
            L.oracle_layer.argtypes = [vp, vp, i64, c_int, c_int, c_int, c_int, vp, vp, vp, vp, vp, c_int]
            L.oracle_layer.restype = c_int
            L.oracle_layer_tokens.argtypes = [vp, vp, vp, i64, c_int, c_int, c_int, c_int, vp, vp, vp, vp, vp, vp,
                                              vp, c_int]
            L.oracle_layer_tokens_h.argtypes = [vp, vp, vp, i64, c_int, c_int, c_int, c_int, vp, vp, vp, vp, vp, vp,
                                                vp, vp, vp, vp, c_int]
            L.oracle_layer_bruteforce.argtypes = [vp, vp, i64, c_int, c_int, c_int, c_int, vp, vp, vp, vp, vp, c_int]
            L.oracle_bf16_split.argtypes = [vp, i64, vp, vp]
            L.oracle_router_logits.argtypes = [vp, vp, i64, c_int, c_int, vp, c_int]
            L.oracle_router_route.argtypes = [vp, vp, i64, c_int, c_int, c_int, vp, vp, vp, c_int]
            L.oracle_shared_gate.argtypes = [vp, vp, i64, c_int, vp, c_int]
            L.oracle_shared_expert.argtypes = [vp, i64, c_int, c_int, vp, vp, vp, vp, vp, c_int]
            L.oracle_combine_shared.argtypes = [vp, vp, vp, vp, vp, i64, c_int, c_int, vp, c_int]
            L.oracle_layer_shared.argtypes = [vp, vp, i64, c_int, c_int, c_int, c_int, vp, vp, vp, vp, vp, vp, vp, vp,
                                              vp, vp, c_int]
            L.oracle_layer_shared.restype = c_int
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------------------------------------- fp16 helpers
def f2h(x: float) -> int:
    return int(lib().oracle_f2h(float(x)))


def h2f(h: int) -> float:
    return float(lib().oracle_h2f(int(h)))


# ----------------------------------------------------------------------------------------------- the seven steps
def route(logits: np.ndarray, K: int, nthreads: int = 0):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float64)
    lib().oracle_route(_ptr(logits), T, E, K, _ptr(ids), _ptr(w), nthreads)
    return ids, w


def group(ids: np.ndarray, E: int):
    ids = _c(ids, np.int32)
    T, K = ids.shape
    n = T * K
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    src = np.empty(n, np.int32)
    slot = np.empty(n, np.int32)
    rc = lib().oracle_group(_ptr(ids), T, K, E, _ptr(counts), _ptr(offsets), _ptr(src), _ptr(slot))
    if rc != 0:
        raise ValueError("routed id out of range")
    return dict(counts=counts, offsets=offsets, src=src, slot=slot)


def quantize_q8(x: np.ndarray, nthreads: int = 0):
    x = _c(x, np.float32)
    rows, cols = x.shape
    assert cols % 32 == 0
    codes = np.empty((rows, cols), np.int8)
    scales = np.empty((rows, cols // 32), np.uint16)
    lib().oracle_quantize_q8(_ptr(x), rows, cols, _ptr(codes), _ptr(scales), nthreads)
    return codes, scales


def gateup(xc, xs, src, offsets, wgu_c, wgu_s, H: int, F: int, nthreads: int = 0):
    xc, xs, src, offsets = _c(xc, np.int8), _c(xs, np.uint16), _c(src, np.int32), _c(offsets, np.int32)
    wgu_c, wgu_s = _c(wgu_c, np.uint8), _c(wgu_s, np.uint16)
    E = offsets.shape[0] - 1
    n = int(offsets[-1])
    gu = np.empty((n, 2 * F), np.float64)
    lib().oracle_gateup(_ptr(xc), _ptr(xs), _ptr(src), _ptr(offsets), E, _ptr(wgu_c), _ptr(wgu_s), H, F, _ptr(gu),
                        nthreads)
    return gu


def swiglu_requant(gu: np.ndarray, F: int, nthreads: int = 0):
    n = gu.shape[0]
    hc = np.empty((n, F), np.int8)
    hs = np.empty((n, F // 32), np.uint16)
    if gu.dtype == np.float32:
        gu = _c(gu, np.float32)
        lib().oracle_swiglu_requant_f32(_ptr(gu), n, F, _ptr(hc), _ptr(hs), nthreads)
    else:
        gu = _c(gu, np.float64)
        lib().oracle_swiglu_requant(_ptr(gu), n, F, _ptr(hc), _ptr(hs), nthreads)
    return hc, hs


def down(hc, hs, offsets, wd_c, wd_s, H: int, F: int, nthreads: int = 0):
    hc, hs, offsets = _c(hc, np.int8), _c(hs, np.uint16), _c(offsets, np.int32)
    wd_c, wd_s = _c(wd_c, np.uint8), _c(wd_s, np.uint16)
    E = offsets.shape[0] - 1
    n = int(offsets[-1])
    dm = np.empty((n, H), np.float64)
    lib().oracle_down(_ptr(hc), _ptr(hs), _ptr(offsets), E, _ptr(wd_c), _ptr(wd_s), H, F, _ptr(dm), nthreads)
    return dm


def combine(dm, slot, w, T: int, K: int, H: int, nthreads: int = 0):
    dm, slot, w = _c(dm, np.float64), _c(slot, np.int32), _c(w, np.float64)
    y = np.empty((T, H), np.float64)
    lib().oracle_combine(_ptr(dm), _ptr(slot), _ptr(w), T, K, H, _ptr(y), nthreads)
    return y


# ----------------------------------------------------------------------------------------------- whole block
def _weights(layer):
    return (_c(layer["wgu_c"], np.uint8), _c(layer["wgu_s"], np.uint16), _c(layer["wd_c"], np.uint8),
            _c(layer["wd_s"], np.uint16))


def layer(inp: dict, nthreads: int = 0) -> np.ndarray:
    """The whole block on one chunk; `inp` as made by the package's synthetic-input module."""
    logits, x = _c(inp["logits"], np.float32), _c(inp["x"], np.float32)
    T, H = x.shape
    E, K, F = inp["E"], inp["K"], inp["F"]
    a, b, c, d = _weights(inp)
    y = np.empty((T, H), np.float64)
    rc = lib().oracle_layer(_ptr(logits), _ptr(x), T, H, E, K, F, _ptr(a), _ptr(b), _ptr(c), _ptr(d), _ptr(y),
                            nthreads)
    if rc != 0:
        raise ValueError("routed id out of range")
    return y


def layer_tokens(inp: dict, tokens, nthreads: int = 0):
    """The block for the listed tokens only (one token at a time); returns (y [ntok][H], ids, w)."""
    logits, x = _c(inp["logits"], np.float32), _c(inp["x"], np.float32)
    H = x.shape[1]
    E, K, F = inp["E"], inp["K"], inp["F"]
    tokens = _c(tokens, np.int64)
    ntok = tokens.shape[0]
    a, b, c, d = _weights(inp)
    y = np.empty((ntok, H), np.float64)
    ids = np.empty((ntok, K), np.int32)
    w = np.empty((ntok, K), np.float64)
    lib().oracle_layer_tokens(_ptr(logits), _ptr(x), _ptr(tokens), ntok, H, E, K, F, _ptr(a), _ptr(b), _ptr(c),
                              _ptr(d), _ptr(y), _ptr(ids), _ptr(w), nthreads)
    return y, ids, w


def layer_tokens_h(inp: dict, tokens, nthreads: int = 0):
    """layer_tokens plus each listed token's step-5 intermediates per slot k: returns (y [ntok][H], ids, w,
    h fp32 [ntok][K][F], hc int8 [ntok][K][F], hs fp16 bits [ntok][K][F/32])."""
    logits, x = _c(inp["logits"], np.float32), _c(inp["x"], np.float32)
    H = x.shape[1]
    E, K, F = inp["E"], inp["K"], inp["F"]
    tokens = _c(tokens, np.int64)
    ntok = tokens.shape[0]
    a, b, c, d = _weights(inp)
    y = np.empty((ntok, H), np.float64)
    ids = np.empty((ntok, K), np.int32)
    w = np.empty((ntok, K), np.float64)
    h = np.empty((ntok, K, F), np.float32)
    hc = np.empty((ntok, K, F), np.int8)
    hs = np.empty((ntok, K, F // 32), np.uint16)
    lib().oracle_layer_tokens_h(_ptr(logits), _ptr(x), _ptr(tokens), ntok, H, E, K, F, _ptr(a), _ptr(b), _ptr(c),
                                _ptr(d), _ptr(y), _ptr(ids), _ptr(w), _ptr(h), _ptr(hc), _ptr(hs), nthreads)
    return y, ids, w, h, hc, hs


def layer_bruteforce(inp: dict, nthreads: int = 0) -> np.ndarray:
    logits, x = _c(inp["logits"], np.float32), _c(inp["x"], np.float32)
    T, H = x.shape
    E, K, F = inp["E"], inp["K"], inp["F"]
    a, b, c, d = _weights(inp)
    y = np.empty((T, H), np.float64)
    lib().oracle_layer_bruteforce(_ptr(logits), _ptr(x), T, H, E, K, F, _ptr(a), _ptr(b), _ptr(c), _ptr(d), _ptr(y),
                                  nthreads)
    return y


# ----------------------------------------------------------------------------------------------- shared expert
def _shared_weights(inp):
    return (_c(inp["sgu_c"], np.uint8), _c(inp["sgu_s"], np.uint16), _c(inp["sd_c"], np.uint8),
            _c(inp["sd_s"], np.uint16))


def shared_gate(x: np.ndarray, wsg: np.ndarray, nthreads: int = 0) -> np.ndarray:
    """sg [T] = sigmoid(x . w_sg) per token, in double."""
    x, wsg = _c(x, np.float32), _c(wsg, np.float32)
    T, H = x.shape
    sg = np.empty(T, np.float64)
    lib().oracle_shared_gate(_ptr(x), _ptr(wsg), T, H, _ptr(sg), nthreads)
    return sg


def shared_expert(x: np.ndarray, sgu_c, sgu_s, sd_c, sd_s, F: int, nthreads: int = 0) -> np.ndarray:
    """The shared expert's rows S [T][H] (every token through the one shared expert)."""
    x = _c(x, np.float32)
    T, H = x.shape
    a, b, c, d = _c(sgu_c, np.uint8), _c(sgu_s, np.uint16), _c(sd_c, np.uint8), _c(sd_s, np.uint16)
    out = np.empty((T, H), np.float64)
    lib().oracle_shared_expert(_ptr(x), T, H, F, _ptr(a), _ptr(b), _ptr(c), _ptr(d), _ptr(out), nthreads)
    return out


def combine_shared(dm, slot, w, shared, sg, T: int, K: int, H: int, nthreads: int = 0) -> np.ndarray:
    dm, slot, w = _c(dm, np.float64), _c(slot, np.int32), _c(w, np.float64)
    shared, sg = _c(shared, np.float64), _c(sg, np.float64)
    y = np.empty((T, H), np.float64)
    lib().oracle_combine_shared(_ptr(dm), _ptr(slot), _ptr(w), _ptr(shared), _ptr(sg), T, K, H, _ptr(y), nthreads)
    return y


def layer_shared(inp: dict, nthreads: int = 0) -> np.ndarray:
    """The whole block with the shared expert; `inp` also holds the shared weights and the gate row."""
    logits, x = _c(inp["logits"], np.float32), _c(inp["x"], np.float32)
    T, H = x.shape
    E, K, F = inp["E"], inp["K"], inp["F"]
    a, b, c, d = _weights(inp)
    sa, sb, sc, sd = _shared_weights(inp)
    wsg = _c(inp["wsg"], np.float32)
    y = np.empty((T, H), np.float64)
    rc = lib().oracle_layer_shared(_ptr(logits), _ptr(x), T, H, E, K, F, _ptr(a), _ptr(b), _ptr(c), _ptr(d), _ptr(sa),
                                   _ptr(sb), _ptr(sc), _ptr(sd), _ptr(wsg), _ptr(y), nthreads)
    if rc != 0:
        raise ValueError("routed id out of range")
    return y


def layer_tokens_shared(inp: dict, tokens, nthreads: int = 0):
    """The block with the shared expert for the listed tokens only; returns (y [ntok][H], ids, w)."""
    y, ids, w = layer_tokens(inp, tokens, nthreads)
    xs = _c(np.asarray(inp["x"], np.float32)[np.asarray(tokens, np.int64)], np.float32)
    sa, sb, sc, sd = _shared_weights(inp)
    y = y + shared_gate(xs, inp["wsg"], nthreads)[:, None] * shared_expert(xs, sa, sb, sc, sd, inp["F"], nthreads)
    return y, ids, w


# ----------------------------------------------------------------------------------------------- router projection
def bf16_split(x: np.ndarray):
    """(xh, xl) bf16 bits (uint16) of fp32 x: xh = bf16_rne(x), xl = bf16_rne(x - xh)."""
    x = _c(x, np.float32)
    xh = np.empty(x.shape, np.uint16)
    xl = np.empty(x.shape, np.uint16)
    lib().oracle_bf16_split(_ptr(x), x.size, _ptr(xh), _ptr(xl))
    return xh, xl


def router_logits(x: np.ndarray, wr: np.ndarray, nthreads: int = 0) -> np.ndarray:
    """logits double [T][E] = wr (bf16 bits [E][H]) . (xh + xl)."""
    x, wr = _c(x, np.float32), _c(wr, np.uint16)
    T, H = x.shape
    E = wr.shape[0]
    out = np.empty((T, E), np.float64)
    lib().oracle_router_logits(_ptr(x), _ptr(wr), T, H, E, _ptr(out), nthreads)
    return out


def router_route(x: np.ndarray, wr: np.ndarray, K: int, nthreads: int = 0):
    """Step 1 from the hidden state: (ids [T][K], w double [T][K], logits double [T][E])."""
    x, wr = _c(x, np.float32), _c(wr, np.uint16)
    T, H = x.shape
    E = wr.shape[0]
    ids = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float64)
    lg = np.empty((T, E), np.float64)
    lib().oracle_router_route(_ptr(x), _ptr(wr), T, H, E, K, _ptr(ids), _ptr(w), _ptr(lg), nthreads)
    return ids, w, lg
