"""Oracle for the routed-expert MoE block -- TEST INFRASTRUCTURE ONLY.

ctypes wrapper over ``strata_oracle.c`` (plain C, double precision).  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import this package; the
CUDA library never links or calls it.  See ``strata_oracle.h`` for what each function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libstrata_oracle.so")
_lib = None

_c_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_c_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_c_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_c_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_c_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")


def build(cc: str = "gcc", wait: bool = True):
    """Compile the oracle (plain C, no contraction of a*b+c so every host rounds the same)."""
    cmd = [cc, "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", "-o", LIB_PATH, os.path.join(_HERE, "strata_oracle.c"), "-lm"]
    p = subprocess.Popen(cmd)
    if wait:
        if p.wait() != 0:
            raise RuntimeError("oracle build failed")
        return None
    return p


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            build()
        L = ctypes.CDLL(LIB_PATH)
        L.oracle_fp16_to_double.restype = ctypes.c_double
        L.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_double.restype = ctypes.c_double
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_q2_code.restype = ctypes.c_int
        L.oracle_q2_code.argtypes = [_c_u8p, ctypes.c_int]
        L.oracle_dequant_blocks.restype = None
        L.oracle_dequant_blocks.argtypes = [_c_u8p, ctypes.c_int64, ctypes.c_int, _c_f64p]
        L.oracle_dequant_blob.restype = ctypes.c_int
        L.oracle_dequant_blob.argtypes = [_c_u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          _c_f64p, _c_f64p, _c_f64p]
        L.oracle_router_logits.restype = None
        L.oracle_router_logits.argtypes = [_c_f64p, ctypes.c_int, ctypes.c_int, _c_u16p,
                                           ctypes.c_void_p, _c_f64p]
        L.oracle_top_k.restype = None
        L.oracle_top_k.argtypes = [_c_f64p, ctypes.c_int, ctypes.c_int, _c_i32p, _c_f64p,
                                   ctypes.c_void_p]
        L.oracle_weights_for_ids.restype = None
        L.oracle_weights_for_ids.argtypes = [_c_f64p, ctypes.c_int, ctypes.c_int, _c_i32p, _c_f64p]
        L.oracle_group.restype = None
        L.oracle_group.argtypes = [_c_i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _c_i32p,
                                   _c_i32p, _c_i32p, _c_i32p]
        L.oracle_expert.restype = None
        L.oracle_expert.argtypes = [_c_u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _c_f64p,
                                    _c_f64p]
        L.oracle_rmsnorm.restype = None
        L.oracle_rmsnorm.argtypes = [_c_f64p, ctypes.c_int, ctypes.c_double, _c_f64p]
        L.oracle_route_tokens.restype = ctypes.c_int
        L.oracle_route_tokens.argtypes = [_c_f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          _c_u16p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        L.oracle_moe_layer.restype = ctypes.c_int
        L.oracle_moe_layer.argtypes = [
            _c_f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _c_u16p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, _c_f64p,
            ctypes.c_int, ctypes.c_void_p]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def fp16_to_double(bits: int) -> float:
    return lib().oracle_fp16_to_double(bits)


def bf16_to_double(bits: int) -> float:
    return lib().oracle_bf16_to_double(bits)


def q2_codes(codes16: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(codes16, dtype=np.uint8)
    return np.array([lib().oracle_q2_code(c, i) for i in range(64)], dtype=np.int32)


def dequant_blocks(blocks: np.ndarray, q2_offset: int) -> np.ndarray:
    b = np.ascontiguousarray(blocks, dtype=np.uint8)
    n = b.size // 18
    w = np.empty(64 * n, dtype=np.float64)
    lib().oracle_dequant_blocks(b, n, q2_offset, w)
    return w


def dequant_blob(blob: np.ndarray, H: int, FF: int, q2_offset: int):
    b = np.ascontiguousarray(blob, dtype=np.uint8)
    g = np.empty((FF, H)); u = np.empty((FF, H)); d = np.empty((H, FF))
    if lib().oracle_dequant_blob(b, H, FF, q2_offset, g, u, d):
        raise ValueError("H*FF must be a multiple of 64")
    return g, u, d


def router_logits(xn: np.ndarray, w_router: np.ndarray, bias=None) -> np.ndarray:
    E, H = w_router.shape
    xn = np.ascontiguousarray(xn, dtype=np.float64)
    out = np.empty(E, dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    lib().oracle_router_logits(xn, H, E, np.ascontiguousarray(w_router, dtype=np.uint16), _ptr(b), out)
    return out


def top_k(logits: np.ndarray, K: int):
    l = np.ascontiguousarray(logits, dtype=np.float64)
    E = l.size
    ids = np.empty(K, dtype=np.int32)
    w = np.empty(K, dtype=np.float64)
    p = np.empty(E, dtype=np.float64)
    lib().oracle_top_k(l, E, K, ids, w, _ptr(p))
    return ids, w, p


def weights_for_ids(logits: np.ndarray, ids: np.ndarray) -> np.ndarray:
    l = np.ascontiguousarray(logits, dtype=np.float64)
    i = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.empty(i.size, dtype=np.float64)
    lib().oracle_weights_for_ids(l, l.size, i.size, i, w)
    return w


def group(ids: np.ndarray, E: int):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, K = ids.shape
    off = np.empty(E + 1, dtype=np.int32)
    pair = np.empty(T * K, dtype=np.int32)
    active = np.empty(E, dtype=np.int32)
    na = np.empty(1, dtype=np.int32)
    lib().oracle_group(ids, T, K, E, off, pair, active, na)
    return off, pair, active[: int(na[0])]


def expert(blob: np.ndarray, H: int, FF: int, q2_offset: int, x: np.ndarray) -> np.ndarray:
    y = np.empty(H, dtype=np.float64)
    lib().oracle_expert(np.ascontiguousarray(blob, dtype=np.uint8), H, FF, q2_offset,
                        np.ascontiguousarray(x, dtype=np.float64), y)
    return y


def rmsnorm(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    lib().oracle_rmsnorm(x, x.size, eps, out)
    return out


def route(x, w_router, bias=None, residual=False, K=10, n_threads=None):
    """Steps 1-2 for x fp32[T][H]: dict(ids [T][K], w [T][K], logits [T][E])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    T, H = x.shape
    E = w_router.shape[0]
    ids = np.empty((T, K), dtype=np.int32)
    w = np.empty((T, K), dtype=np.float64)
    logits = np.empty((T, E), dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    nt = n_threads if n_threads else max(1, min(os.cpu_count() or 1, T))
    rc = lib().oracle_route_tokens(x, T, H, E, K, np.ascontiguousarray(w_router, dtype=np.uint16), _ptr(b),
                                   1 if residual else 0, _ptr(ids), _ptr(w), _ptr(logits), nt)
    if rc:
        raise ValueError("oracle_route_tokens: bad argument")
    return dict(ids=ids, w=w, logits=logits)


def moe_layer(x, w_router, bias, blobs, q2_offset=1, residual=False, ids_in=None, H=None, FF=None,
              K=10, want_parts=False, n_threads=None, shared=None):
    """One MoE layer for x fp32[T][H]. blobs: list of E canonical blobs (None where unused); shared:
    the layer's shared expert (canonical blob) or None.

    Returns dict(out, ids, w, logits[, parts])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    T, Hx = x.shape
    H = Hx if H is None else H
    E = w_router.shape[0]
    FF = FF if FF is not None else (blobs_ff(blobs, H))
    keep = [None if b is None else np.ascontiguousarray(b, dtype=np.uint8) for b in blobs]
    arr = (ctypes.c_void_p * E)(*[None if b is None else b.ctypes.data for b in keep])
    ids = np.empty((T, K), dtype=np.int32)
    w = np.empty((T, K), dtype=np.float64)
    logits = np.empty((T, E), dtype=np.float64)
    parts = np.empty((T, K, H), dtype=np.float64) if want_parts else None
    out = np.empty((T, H), dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    ii = None if ids_in is None else np.ascontiguousarray(ids_in, dtype=np.int32)
    nt = n_threads if n_threads else max(1, min(os.cpu_count() or 1, T))
    sh = None if shared is None else np.ascontiguousarray(shared, dtype=np.uint8)
    rc = lib().oracle_moe_layer(x, T, H, FF, E, K, np.ascontiguousarray(w_router, dtype=np.uint16),
                                _ptr(b), ctypes.cast(arr, ctypes.c_void_p), q2_offset,
                                1 if residual else 0, _ptr(ii), _ptr(ids), _ptr(w), _ptr(logits),
                                _ptr(parts), out, nt, _ptr(sh))
    if rc:
        raise ValueError("oracle_moe_layer: bad argument or a routed expert has no blob")
    res = dict(out=out, ids=ids, w=w, logits=logits)
    if want_parts:
        res["parts"] = parts
    return res


def blobs_ff(blobs, H):
    for b in blobs:
        if b is not None:
            return (b.size // 18) * 64 // (3 * H)
    raise ValueError("no blob given")
