"""Seeded synthetic inputs for the routed-expert MoE block (shared by the oracle and the GPU path).

This module holds no arithmetic of the method: it only draws random numbers and writes them in
the storage formats the method reads (fp32 activations, bf16 router rows, canonical Q2_0 expert
blobs).  Both sides of every parity check take their inputs from here; neither side's results
feed back into it.

Random numbers come from Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers:
as easy as 1, 2, 3", SC'11), restated here from that definition.  Every value is addressed by
(seed, stream tag) as the key and an index tuple as the counter, so any single expert blob can
be regenerated alone (the 33,973,862,400-byte arena of 48 x 512 blobs never has to exist on the
host).  ``gen_device.cu`` is the same generator for the expert blobs on the GPU; it uses only
integer arithmetic plus the fp16 scale table built here, so the two sides agree bit for bit.

Stream tags (key word 1) and counters:
  TAG_CODES  (1): block b of blob (layer l, expert e): counter (b, 0, l, e) -> the block's 16 code bytes
  TAG_SCALES (2): counter (b >> 3, 0, l, e) -> eight 16-bit uniforms; the (b & 7)-th picks the block's
                  scale from SCALE_TABLE (half-normal quantiles x 0.02, rounded to fp16)
  TAG_X      (3): activation x[t][h]: counter (h >> 2, 0, t, 0), Box-Muller, 4 normals per counter
  TAG_WR     (4): router row e of layer l: counter (h >> 2, 0, e, l), N(0, 0.02) rounded to bf16 via fp32
  TAG_PERM   (5): Zipf permutation keys for layer l: counter (i, 0, l, 0)
  TAG_NOISE  (6): verify-window noise for token j: counter (h >> 2, 0, j, 0)
"""
from __future__ import annotations

import ctypes
import os
import statistics

import numpy as np

H = 2560
FF = 640
E = 512
K = 10
QK = 64
BLOCK_BYTES = 18  # fp16 scale + 16 bytes of 2-bit codes

TAG_CODES, TAG_SCALES, TAG_X, TAG_WR, TAG_PERM, TAG_NOISE = 1, 2, 3, 4, 5, 6

_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32 with 10 rounds; counters are uint32 arrays (broadcast), key is two uint32 ints."""
    c0, c1, c2, c3 = np.broadcast_arrays(*(np.asarray(c, dtype=np.uint32) for c in (c0, c1, c2, c3)))
    c0, c1, c2, c3 = (c.copy() for c in (c0, c1, c2, c3))
    k0 = int(k0) & 0xFFFFFFFF
    k1 = int(k1) & 0xFFFFFFFF
    for r in range(10):
        if r:
            k0 = (k0 + _W0) & 0xFFFFFFFF
            k1 = (k1 + _W1) & 0xFFFFFFFF
        p0 = c0.astype(np.uint64) * _M0
        p1 = c2.astype(np.uint64) * _M1
        hi0 = (p0 >> np.uint64(32)).astype(np.uint32)
        lo0 = (p0 & _MASK32).astype(np.uint32)
        hi1 = (p1 >> np.uint64(32)).astype(np.uint32)
        lo1 = (p1 & _MASK32).astype(np.uint32)
        c0, c1, c2, c3 = hi1 ^ c1 ^ np.uint32(k0), lo1, hi0 ^ c3 ^ np.uint32(k1), lo0
    return c0, c1, c2, c3


def _normals(seed, tag, n, a, b):
    """n standard normals (n % 4 == 0) from counters (i, 0, a, b), i = 0 .. n/4-1, via Box-Muller."""
    i = np.arange(n // 4, dtype=np.uint32)
    w = philox4x32_10(i, 0, a, b, seed, tag)
    u = [(x.astype(np.float64) + 0.5) * 2.0 ** -32 for x in w]
    r01 = np.sqrt(-2.0 * np.log(u[0]))
    r23 = np.sqrt(-2.0 * np.log(u[2]))
    z = np.empty((n // 4, 4), dtype=np.float64)
    z[:, 0] = r01 * np.cos(2.0 * np.pi * u[1])
    z[:, 1] = r01 * np.sin(2.0 * np.pi * u[1])
    z[:, 2] = r23 * np.cos(2.0 * np.pi * u[3])
    z[:, 3] = r23 * np.sin(2.0 * np.pi * u[3])
    return z.reshape(-1)


def _build_scale_table():
    nd = statistics.NormalDist()
    q = (np.arange(65536, dtype=np.float64) + 0.5) / 131072.0 + 0.5
    z = np.array([nd.inv_cdf(v) for v in q], dtype=np.float64)
    return (0.02 * z).astype(np.float16)


SCALE_TABLE = _build_scale_table()  # fp16[65536], |N(0, 0.02)| quantiles


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def blob_blocks(H_=H, FF_=FF):
    return 3 * H_ * FF_ // QK


def blob_bytes(H_=H, FF_=FF):
    return blob_blocks(H_, FF_) * BLOCK_BYTES


def canonical_blob(seed: int, layer: int, expert: int, H_: int = H, FF_: int = FF) -> np.ndarray:
    """One expert as a canonical Q2_0 blob: gate, up, down; each block = {fp16 d, 16 code bytes}."""
    nb = blob_blocks(H_, FF_)
    b = np.arange(nb, dtype=np.uint32)
    w = philox4x32_10(b, 0, layer, expert, seed, TAG_CODES)
    codes = np.stack(w, axis=1).astype("<u4").view(np.uint8).reshape(nb, 16)
    s = philox4x32_10(np.arange((nb + 7) // 8, dtype=np.uint32), 0, layer, expert, seed, TAG_SCALES)
    u16 = np.stack(s, axis=1).astype("<u4").view("<u2").reshape(-1)[:nb]
    d = SCALE_TABLE[u16]
    out = np.empty((nb, BLOCK_BYTES), dtype=np.uint8)
    out[:, 0:2] = d.astype("<f2").view(np.uint8).reshape(nb, 2)
    out[:, 2:] = codes
    return out.reshape(-1)


def activations(seed: int, T: int, H_: int = H) -> np.ndarray:
    """x[t] ~ N(0, 1), fp32[T][H]."""
    x = np.empty((T, H_), dtype=np.float32)
    for t in range(T):
        x[t] = _normals(seed, TAG_X, H_, t, 0).astype(np.float32)
    return x


def activations_fast(seed: int, T: int, H_: int = H) -> np.ndarray:
    """Same values as ``activations`` (one Philox call over all tokens at once)."""
    i = np.tile(np.arange(H_ // 4, dtype=np.uint32), T)
    t = np.repeat(np.arange(T, dtype=np.uint32), H_ // 4)
    w = philox4x32_10(i, 0, t, 0, seed, TAG_X)
    u = [(v.astype(np.float64) + 0.5) * 2.0 ** -32 for v in w]
    r01 = np.sqrt(-2.0 * np.log(u[0]))
    r23 = np.sqrt(-2.0 * np.log(u[2]))
    z = np.empty((T * H_ // 4, 4), dtype=np.float64)
    z[:, 0] = r01 * np.cos(2.0 * np.pi * u[1])
    z[:, 1] = r01 * np.sin(2.0 * np.pi * u[1])
    z[:, 2] = r23 * np.cos(2.0 * np.pi * u[3])
    z[:, 3] = r23 * np.sin(2.0 * np.pi * u[3])
    return z.reshape(T, H_).astype(np.float32)


def verify_window(seed: int, T: int = 4, H_: int = H) -> np.ndarray:
    """Correlated verify window: x_0 ~ N(0,1); x_j = x_0 + 0.3 N(0,1) for j >= 1."""
    x0 = _normals(seed, TAG_X, H_, 0, 0)
    x = np.empty((T, H_), dtype=np.float32)
    x[0] = x0.astype(np.float32)
    for j in range(1, T):
        x[j] = (x0 + 0.3 * _normals(seed, TAG_NOISE, H_, j, 0)).astype(np.float32)
    return x


def router_weights(seed: int, layer: int, E_: int = E, H_: int = H) -> np.ndarray:
    """Router rows W[e][h] ~ N(0, 0.02), as bf16 bit patterns uint16[E][H]."""
    i = np.tile(np.arange(H_ // 4, dtype=np.uint32), E_)
    e = np.repeat(np.arange(E_, dtype=np.uint32), H_ // 4)
    w = philox4x32_10(i, 0, e, layer, seed, TAG_WR)
    u = [(v.astype(np.float64) + 0.5) * 2.0 ** -32 for v in w]
    r01 = np.sqrt(-2.0 * np.log(u[0]))
    r23 = np.sqrt(-2.0 * np.log(u[2]))
    z = np.empty((E_ * H_ // 4, 4), dtype=np.float64)
    z[:, 0] = r01 * np.cos(2.0 * np.pi * u[1])
    z[:, 1] = r01 * np.sin(2.0 * np.pi * u[1])
    z[:, 2] = r23 * np.cos(2.0 * np.pi * u[3])
    z[:, 3] = r23 * np.sin(2.0 * np.pi * u[3])
    return f32_to_bf16_bits((0.02 * z).astype(np.float32)).reshape(E_, H_)


def zipf_bias(seed: int, layer: int, E_: int = E, s: float = 1.1) -> np.ndarray:
    """Per-expert logit bias -s*ln(1 + rank(e)), rank from a seeded permutation (prior ~ rank^-s)."""
    w = philox4x32_10(np.arange(E_ // 4, dtype=np.uint32), 0, layer, 0, seed, TAG_PERM)
    keys = np.stack(w, axis=1).reshape(-1)[:E_]
    order = np.argsort(keys, kind="stable")
    rank = np.empty(E_, dtype=np.int64)
    rank[order] = np.arange(E_)
    return (-s * np.log1p(rank.astype(np.float64))).astype(np.float32)


# ----------------------------------------------------------------------------------------------
# The five benchmark workloads (seed 0) and their input recipes.
# ----------------------------------------------------------------------------------------------
CONFIGS = {
    0: dict(name="decode_1tok_1layer", T=1, L=1, bias=False, residual=False, window=False),
    1: dict(name="verify_4tok_1layer", T=4, L=1, bias=False, residual=False, window=True),
    2: dict(name="decode_1tok_48layer_stack", T=1, L=48, bias="shared", residual=True, window=False),
    3: dict(name="prefill_2048tok_1layer", T=2048, L=1, bias="shared", residual=False, window=False),
    4: dict(name="prefill_8192tok_48layer_stack", T=8192, L=48, bias="per_layer", residual=True, window=False),
}


def config_inputs(cfg: int, seed: int = 0, T: int | None = None, L: int | None = None):
    """x, per-layer router rows and biases for a workload (expert blobs are drawn per expert)."""
    c = CONFIGS[cfg]
    T = c["T"] if T is None else T
    L = c["L"] if L is None else L
    x = verify_window(seed, T) if c["window"] else activations_fast(seed, T)
    wr = [router_weights(seed, l) for l in range(L)]
    if c["bias"] == "shared":
        b = zipf_bias(seed, 0)
        bias = [b for _ in range(L)]
    elif c["bias"] == "per_layer":
        bias = [zipf_bias(seed, l) for l in range(L)]
    else:
        bias = [None for _ in range(L)]
    return dict(x=x, wr=wr, bias=bias, T=T, L=L, residual=c["residual"], name=c["name"])


# ----------------------------------------------------------------------------------------------
# Device generator (gen_device.cu): fills canonical blobs for whole layers on the GPU.
# ----------------------------------------------------------------------------------------------
_HERE = os.path.dirname(os.path.abspath(__file__))
_DEV_LIB = os.path.join(_HERE, "libstrata_gen.so")
_dev = None


def build_device(nvcc="nvcc"):
    import subprocess
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
           "-Xcompiler", "-fPIC", "-shared", "-o", _DEV_LIB, os.path.join(_HERE, "gen_device.cu")]
    return subprocess.Popen(cmd)


def device_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(_DEV_LIB):
            raise RuntimeError("gen/libstrata_gen.so is missing: run __graft_entry__.build()")
        lib = ctypes.CDLL(_DEV_LIB)
        lib.strata_gen_canonical_blobs.restype = ctypes.c_int
        lib.strata_gen_canonical_blobs.argtypes = [
            ctypes.c_uint32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        _dev = lib
    return _dev


def device_canonical_blobs(seed, layer, e0, n, table_dev_ptr, out_ptr, blob_stride, stream_ptr=0):
    """Generate canonical blobs (layer, e0..e0+n-1) into device memory at out_ptr."""
    rc = device_lib().strata_gen_canonical_blobs(seed, layer, e0, n, table_dev_ptr, out_ptr,
                                                 blob_stride, stream_ptr)
    if rc != 0:
        raise RuntimeError(f"strata_gen_canonical_blobs failed: {rc}")
