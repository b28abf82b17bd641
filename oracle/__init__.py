"""CPU oracle of the reduced-vocabulary draft head (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the CUDA library and
its Python binding) never does.

The arithmetic lives in ``oracle_dh.c`` (plain C11, compiled here with gcc,
``-ffp-contract=off``); this module compiles it on first use and wraps it with
numpy arrays. It shares no code with the CUDA library.

Parity-unpinned reading: the operation order inside the NVFP4 quantiser
(``or_nvfp4_quantize``) beyond the recipe the pages state.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_dh.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle_dh.so")
_lock = threading.Lock()
_lib = None

FMT_NVFP4, FMT_FP8, FMT_BF16 = 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library (gcc, no fast-math, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(
            ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            lib = C.CDLL(build())
            P = C.c_void_p
            i, f = C.c_int, C.c_float
            lib.or_e2m1_decode.argtypes = [i]
            lib.or_e2m1_decode.restype = C.c_double
            lib.or_e4m3_decode.argtypes = [i]
            lib.or_e4m3_decode.restype = C.c_double
            lib.or_e2m1_encode.argtypes = [f]
            lib.or_e2m1_encode.restype = i
            lib.or_e4m3_encode.argtypes = [f]
            lib.or_e4m3_encode.restype = i
            lib.or_build_index.argtypes = [P, i, P, i, P, P]
            lib.or_nvfp4_quantize.argtypes = [P, i, i, P, i, P, P, P]
            lib.or_fp8_quantize.argtypes = [P, i, i, P, i, P, P]
            lib.or_gemv.argtypes = [i, P, P, f, i, i, P, i, P, P]
            lib.or_fp8_act_quantize.argtypes = [P, i, i, P, P]
            lib.or_gemv_w8a8.argtypes = [P, f, i, i, P, P, i, P, P]
            lib.or_argmax.argtypes = [P, i]
            lib.or_top_tokens.argtypes = [P, i, i, P, P, P]
            lib.or_scatter_logits.argtypes = [P, i, i, P, i, i, P]
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data_as(C.c_void_p)


class OracleError(RuntimeError):
    pass


def _ok(st: int, what: str):
    if st != 0:
        raise OracleError(f"{what}: oracle status {st}")


# ---- number formats -------------------------------------------------------

def e2m1_decode(code: int) -> float:
    return _L().or_e2m1_decode(int(code))


def e4m3_decode(byte: int) -> float:
    return _L().or_e4m3_decode(int(byte))


def e2m1_encode(x: float) -> int:
    return _L().or_e2m1_encode(float(x))


def e4m3_encode(x: float) -> int:
    return _L().or_e4m3_encode(float(x))


# ---- head build -----------------------------------------------------------

def build_index(keep: np.ndarray):
    """(idx int32[N], n_kept) from a uint8 keep mask; raises on an empty mask."""
    keep = np.ascontiguousarray(keep, dtype=np.uint8)
    V = keep.size
    cap = V + 64
    idx = np.empty(cap, dtype=np.int32)
    nk, N = C.c_int(), C.c_int()
    _ok(_L().or_build_index(_p(keep), V, _p(idx), cap, C.byref(nk), C.byref(N)), "build_index")
    return idx[: N.value].copy(), nk.value


def nvfp4_quantize(W: np.ndarray, idx: np.ndarray):
    """(q uint8[N, K/2], sf uint8[N, K/16], g float32) of the rows W[idx]."""
    W = np.ascontiguousarray(W, dtype=np.uint16)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    V, K = W.shape
    N = idx.size
    q = np.empty((N, K // 2), dtype=np.uint8)
    sf = np.empty((N, K // 16), dtype=np.uint8)
    g = C.c_float()
    _ok(_L().or_nvfp4_quantize(_p(W), V, K, _p(idx), N, _p(q), _p(sf), C.byref(g)), "nvfp4_quantize")
    return q, sf, np.float32(g.value)


def fp8_quantize(W: np.ndarray, idx: np.ndarray):
    """(q uint8[N, K], scale float32) of the rows W[idx]."""
    W = np.ascontiguousarray(W, dtype=np.uint16)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    V, K = W.shape
    N = idx.size
    q = np.empty((N, K), dtype=np.uint8)
    s = C.c_float()
    _ok(_L().or_fp8_quantize(_p(W), V, K, _p(idx), N, _p(q), C.byref(s)), "fp8_quantize")
    return q, np.float32(s.value)


def fp8_act_quantize(h: np.ndarray):
    """(qx uint8[M, K], sx float32[M]): per-token E4M3 codes and scales of the
    BF16 hidden states h (uint16 bits [M, K])."""
    h = np.ascontiguousarray(np.atleast_2d(h), dtype=np.uint16)
    M, K = h.shape
    qx = np.empty((M, K), dtype=np.uint8)
    sx = np.empty(M, dtype=np.float32)
    _ok(_L().or_fp8_act_quantize(_p(h), M, K, _p(qx), _p(sx)), "fp8_act_quantize")
    return qx, sx


# ---- draft step -----------------------------------------------------------

def gemv_w8a8(q: np.ndarray, scale, qx: np.ndarray, sx: np.ndarray, want_abs: bool = True):
    """(y float64[M, N], A float64[M, N] or None): W8A8 FP8 logits of every head
    row from the per-token activation codes qx [M, K] and scales sx [M]."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    qx = np.ascontiguousarray(np.atleast_2d(qx), dtype=np.uint8)
    sx = np.ascontiguousarray(sx, dtype=np.float32)
    N, K = q.shape
    M = qx.shape[0]
    assert qx.shape[1] == K and sx.size == M
    y = np.empty((M, N), dtype=np.float64)
    A = np.empty((M, N), dtype=np.float64) if want_abs else None
    _ok(_L().or_gemv_w8a8(_p(q), float(scale), N, K, _p(qx), _p(sx), M, _p(y),
                          _p(A) if want_abs else None), "gemv_w8a8")
    return y, A


def gemv(fmt: int, q: np.ndarray, sf, scale, h: np.ndarray, want_abs: bool = True):
    """(y float64[M, N], A float64[M, N] or None): fp64 logits of every head row."""
    q = np.ascontiguousarray(q)
    N = q.shape[0]
    h = np.ascontiguousarray(np.atleast_2d(h), dtype=np.uint16)
    M, K = h.shape
    if fmt == FMT_BF16:
        q = np.ascontiguousarray(q, dtype=np.uint16)
        assert q.shape == (N, K)
    sfp = None
    if fmt == FMT_NVFP4:
        sf = np.ascontiguousarray(sf, dtype=np.uint8)
        sfp = _p(sf)
    y = np.empty((M, N), dtype=np.float64)
    A = np.empty((M, N), dtype=np.float64) if want_abs else None
    _ok(_L().or_gemv(fmt, _p(q), sfp, float(scale or 0.0), N, K, _p(h), M, _p(y),
                     _p(A) if want_abs else None), "gemv")
    return y, A


def top_tokens(y: np.ndarray, idx):
    """(ids int32[M], rows int32[M]): first-max row of each y row and its id."""
    y = np.ascontiguousarray(np.atleast_2d(y), dtype=np.float64)
    M, N = y.shape
    ids = np.empty(M, dtype=np.int32)
    rows = np.empty(M, dtype=np.int32)
    ip = None
    if idx is not None:
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        ip = _p(idx)
    _ok(_L().or_top_tokens(_p(y), M, N, ip, _p(ids), _p(rows)), "top_tokens")
    return ids, rows


def scatter_logits(y: np.ndarray, idx: np.ndarray, n_kept: int, V: int) -> np.ndarray:
    """float32[M, V]: -inf everywhere except out[m, idx[n]] = y[m, n] for n < n_kept."""
    y = np.ascontiguousarray(np.atleast_2d(y), dtype=np.float64)
    M, N = y.shape
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    out = np.empty((M, V), dtype=np.float32)
    _ok(_L().or_scatter_logits(_p(y), M, N, _p(idx), int(n_kept), V, _p(out)), "scatter_logits")
    return out


def dequant_nvfp4(q: np.ndarray, sf: np.ndarray, g) -> np.ndarray:
    """float64[N, K] dequantised NVFP4 head, through the oracle's own decoders."""
    e2 = np.array([e2m1_decode(c) for c in range(16)])
    e4 = np.array([e4m3_decode(b) for b in range(256)])
    N, Kh = q.shape
    codes = np.empty((N, 2 * Kh), dtype=np.uint8)
    codes[:, 0::2] = q & 15
    codes[:, 1::2] = q >> 4
    return e2[codes] * np.repeat(e4[sf], 16, axis=1) * float(g)
