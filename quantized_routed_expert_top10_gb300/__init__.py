"""Python binding of the GB300 routed-expert MoE block (C ABI in include/strata_moe.h).

Argument marshalling only: every function has the name of the C entry point it calls, accepts
torch tensors (device tensors for device pointers), raw integer addresses or None, and raises
``StrataError`` when the call returns a status other than STRATA_OK.  All computation runs in
the CUDA library ``libstrata_moe.so``; importing a function of this module fails loudly when
the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libstrata_moe.so")

H = 2560
FF = 640
E_MAX = 512
K = 10
QK = 64
BLOB_BYTES = 1382400
T_MAX = 8192
RESIDUAL_RMSNORM = 1
GROUP_NOALLOC_SCRATCH_BYTES = 256 * 1024

STATUS = {
    0: "STRATA_OK",
    -1: "STRATA_E_INVAL",
    -2: "STRATA_E_ALIGN",
    -3: "STRATA_E_UNSUPPORTED",
    -4: "STRATA_E_CUDA",
    -5: "STRATA_E_TIMEOUT",
    -6: "STRATA_E_WORKSPACE",
    -7: "STRATA_E_CORRUPT",
}

# Every symbol include/strata_moe.h declares.
EXPORTS = (
    "strata_moe_workspace_bytes", "strata_moe_workspace_init", "strata_moe_route", "strata_moe_group",
    "strata_moe_group_noalloc",
    "strata_moe_experts", "strata_moe_combine", "strata_moe_layer", "strata_moe_stack",
    "strata_moe_layer_host", "strata_moe_stack_host", "strata_moe_wait_selftest", "strata_blob_crc32",
    "strata_blob_crc32_device",
    "strata_pack_q2_0", "strata_unpack_q2_0", "strata_pack_q2_0_device", "strata_poll_status",
    "strata_clear_status", "strata_status_str", "strata_moe_launch_count", "strata_moe_profile_arm",
    "strata_moe_profile_recorded",
)


class StrataError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} -> {STATUS.get(status, status)}")


class strata_experts_t(ctypes.Structure):
    _fields_ = [("blobs", ctypes.c_void_p), ("blob_stride", ctypes.c_int64),
                ("n_expert", ctypes.c_int32), ("q2_offset", ctypes.c_int32), ("shared_blob", ctypes.c_void_p)]


_lib = None
_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t


def lib():
    """The loaded CUDA library; raises if it is missing (there is no fallback path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA extension {LIB_PATH} is missing: run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "strata_moe_workspace_bytes": (_sz, [_i32]),
            "strata_moe_workspace_init": (ctypes.c_int, [_vp, _sz, _vp]),
            "strata_moe_route": (ctypes.c_int, [_vp, _i32, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _sz, _vp]),
            "strata_moe_group": (ctypes.c_int, [_vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
            "strata_moe_group_noalloc": (ctypes.c_int, [_vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp]),
            "strata_moe_experts": (ctypes.c_int, [ctypes.POINTER(strata_experts_t), _vp, _i32, _vp, _vp, _vp,
                                                  _vp, _vp, _vp, _sz, _vp]),
            "strata_moe_combine": (ctypes.c_int, [_vp, _vp, _i32, _vp, _vp, _vp]),
            "strata_moe_layer": (ctypes.c_int, [ctypes.POINTER(strata_experts_t), _vp, _vp, _vp, _i32, _i32,
                                                _vp, _vp, _vp, _vp, _sz, _vp]),
            "strata_moe_stack": (ctypes.c_int, [ctypes.POINTER(strata_experts_t), _vp, _vp, _i32, _vp, _i32,
                                                _vp, _vp, _vp, _sz, _vp]),
            "strata_moe_layer_host": (ctypes.c_int, [ctypes.POINTER(strata_experts_t), _vp, _vp, _vp, _i32, _i32,
                                                     _vp, _vp, _vp, _vp, _sz, _vp]),
            "strata_moe_stack_host": (ctypes.c_int, [ctypes.POINTER(strata_experts_t), _vp, _vp, _i32, _vp, _i32,
                                                     _vp, _vp, _vp, _sz, _vp]),
            "strata_moe_wait_selftest": (ctypes.c_int, [_vp, _sz, ctypes.c_uint64, _vp]),
            "strata_blob_crc32": (ctypes.c_int, [_vp, _i64, _i64, _vp]),
            "strata_blob_crc32_device": (ctypes.c_int, [_vp, _i64, _i64, _vp, _vp]),
            "strata_pack_q2_0": (ctypes.c_int, [_vp, _vp, _i64]),
            "strata_unpack_q2_0": (ctypes.c_int, [_vp, _vp, _i64]),
            "strata_pack_q2_0_device": (ctypes.c_int, [_vp, _i64, _vp, _i64, _i64, _vp]),
            "strata_poll_status": (ctypes.c_int, [_vp, _vp]),
            "strata_clear_status": (ctypes.c_int, [_vp, _vp]),
            "strata_status_str": (ctypes.c_char_p, [ctypes.c_int]),
            "strata_moe_launch_count": (ctypes.c_uint64, []),
            "strata_moe_profile_arm": (ctypes.c_int, [_i32, _i32, _vp, _vp, _i32]),
            "strata_moe_profile_recorded": (_i32, [_i32]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _p(a):
    """Address of a tensor / numpy array / int, or None."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if hasattr(a, "data_ptr"):
        return a.data_ptr()
    if hasattr(a, "ctypes"):
        return a.ctypes.data
    raise TypeError(f"cannot take the address of {type(a)}")


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _nbytes(ws, ws_bytes):
    if ws_bytes is not None:
        return ws_bytes
    return ws.numel() * ws.element_size()


def _check(fn, rc):
    if rc != 0:
        raise StrataError(fn, rc)


def experts(blobs, n_expert: int = E_MAX, q2_offset: int = 1, blob_stride: int = BLOB_BYTES,
            shared=None) -> strata_experts_t:
    """A strata_experts_t for packed blobs at a device tensor (or address); shared: the layer's shared
    expert (a packed blob, device tensor or address) or None."""
    return strata_experts_t(_p(blobs), blob_stride, n_expert, q2_offset, _p(shared))


def strata_moe_workspace_bytes(T: int) -> int:
    return lib().strata_moe_workspace_bytes(T)


def strata_moe_workspace_init(ws, ws_bytes=None, stream=None):
    _check("strata_moe_workspace_init", lib().strata_moe_workspace_init(_p(ws), _nbytes(ws, ws_bytes), _s(stream)))


def strata_moe_route(x, T, w_router, bias, n_expert, ids, weights, logits, ws, ws_bytes=None, stream=None):
    _check("strata_moe_route", lib().strata_moe_route(_p(x), T, _p(w_router), _p(bias), n_expert, _p(ids),
                                                      _p(weights), _p(logits), _p(ws), _nbytes(ws, ws_bytes),
                                                      _s(stream)))


def strata_moe_group(ids, T, n_expert, expert_off, pair, active, n_active, ws, ws_bytes=None, stream=None):
    _check("strata_moe_group", lib().strata_moe_group(_p(ids), T, n_expert, _p(expert_off), _p(pair), _p(active),
                                                      _p(n_active), _p(ws), _nbytes(ws, ws_bytes), _s(stream)))


def strata_moe_group_noalloc(ids, T, n_expert, expert_off, pair, active, n_active, stream=None):
    """Grouping with the library's own fixed device scratch: for callers that cannot allocate."""
    _check("strata_moe_group_noalloc", lib().strata_moe_group_noalloc(_p(ids), T, n_expert, _p(expert_off), _p(pair),
                                                                      _p(active), _p(n_active), _s(stream)))


def strata_moe_experts(ex, x, T, expert_off, pair, active, n_active, parts, ws, ws_bytes=None, stream=None):
    _check("strata_moe_experts", lib().strata_moe_experts(ctypes.byref(ex), _p(x), T, _p(expert_off), _p(pair),
                                                          _p(active), _p(n_active), _p(parts), _p(ws),
                                                          _nbytes(ws, ws_bytes), _s(stream)))


def strata_moe_combine(parts, weights, T, residual, out, stream=None):
    _check("strata_moe_combine", lib().strata_moe_combine(_p(parts), _p(weights), T, _p(residual), _p(out),
                                                          _s(stream)))


def strata_moe_layer(ex, w_router, bias, x, T, flags, out, ids, weights, ws, ws_bytes=None, stream=None):
    _check("strata_moe_layer", lib().strata_moe_layer(ctypes.byref(ex), _p(w_router), _p(bias), _p(x), T, flags,
                                                      _p(out), _p(ids), _p(weights), _p(ws),
                                                      _nbytes(ws, ws_bytes), _s(stream)))


def strata_moe_stack(ex_layers, w_router, bias, n_layers, x, T, ids, weights, ws, ws_bytes=None, stream=None):
    arr = (strata_experts_t * max(1, n_layers))(*ex_layers)
    _check("strata_moe_stack", lib().strata_moe_stack(arr, _p(w_router), _p(bias), n_layers, _p(x), T, _p(ids),
                                                      _p(weights), _p(ws), _nbytes(ws, ws_bytes), _s(stream)))


def strata_moe_layer_host(ex, w_router, bias, x_host, T, flags, out_host, ids, weights, ws, ws_bytes=None,
                          stream=None):
    """x_host / out_host: host arrays (CPU tensors or numpy, fp32 [T][2560]); returns with out_host written."""
    _check("strata_moe_layer_host", lib().strata_moe_layer_host(ctypes.byref(ex), _p(w_router), _p(bias), _p(x_host),
                                                                T, flags, _p(out_host), _p(ids), _p(weights), _p(ws),
                                                                _nbytes(ws, ws_bytes), _s(stream)))


def strata_moe_stack_host(ex_layers, w_router, bias, n_layers, x_host, T, ids, weights, ws, ws_bytes=None,
                          stream=None):
    """x_host: host array (fp32 [T][2560]) updated in place; returns with the result in it."""
    arr = (strata_experts_t * max(1, n_layers))(*ex_layers)
    _check("strata_moe_stack_host", lib().strata_moe_stack_host(arr, _p(w_router), _p(bias), n_layers, _p(x_host), T,
                                                                _p(ids), _p(weights), _p(ws), _nbytes(ws, ws_bytes),
                                                                _s(stream)))


class _PreparedCall:
    """A C-ABI call with its arguments marshalled once; calling the object repeats the call (the arrays
    it points at are kept alive here and may change contents between calls)."""

    def __init__(self, name, keep, args):
        self._name = name
        self._keep = keep
        self._f = getattr(lib(), name)
        self._args = args

    def __call__(self):
        rc = self._f(*self._args)
        if rc != 0:
            raise StrataError(self._name, rc)


def prepare_layer_host(ex, w_router, bias, x_host, T, flags, out_host, ids, weights, ws, ws_bytes=None, stream=None):
    """strata_moe_layer_host with fixed arguments, for a serving loop that refills x_host every step."""
    return _PreparedCall("strata_moe_layer_host", (ex, w_router, bias, x_host, out_host, ids, weights, ws, stream),
                         (ctypes.byref(ex), _p(w_router), _p(bias), _p(x_host), T, flags, _p(out_host), _p(ids),
                          _p(weights), _p(ws), _nbytes(ws, ws_bytes), _s(stream)))


def prepare_stack_host(ex_layers, w_router, bias, n_layers, x_host, T, ids, weights, ws, ws_bytes=None, stream=None):
    """strata_moe_stack_host with fixed arguments."""
    arr = (strata_experts_t * max(1, n_layers))(*ex_layers)
    return _PreparedCall("strata_moe_stack_host", (arr, w_router, bias, x_host, ids, weights, ws, stream),
                         (arr, _p(w_router), _p(bias), n_layers, _p(x_host), T, _p(ids), _p(weights), _p(ws),
                          _nbytes(ws, ws_bytes), _s(stream)))


def strata_moe_wait_selftest(ws, limit_ns, ws_bytes=None, stream=None):
    """Run the bounded waits on conditions that never hold (see the header); poll the status after."""
    _check("strata_moe_wait_selftest", lib().strata_moe_wait_selftest(_p(ws), _nbytes(ws, ws_bytes), limit_ns,
                                                                      _s(stream)))


def strata_blob_crc32(blobs, n_blobs, crc, stride=BLOB_BYTES):
    """CRC-32 (zlib's) of each packed blob in host memory into crc (host uint32 [n_blobs])."""
    _check("strata_blob_crc32", lib().strata_blob_crc32(_p(blobs), stride, n_blobs, _p(crc)))


def strata_blob_crc32_device(blobs, n_blobs, crc, stride=BLOB_BYTES, stream=None):
    """The same checksums of blobs in device memory into crc (device uint32 [n_blobs]), enqueued."""
    _check("strata_blob_crc32_device", lib().strata_blob_crc32_device(_p(blobs), stride, n_blobs, _p(crc),
                                                                      _s(stream)))


def strata_pack_q2_0(canonical, packed, n_blobs):
    _check("strata_pack_q2_0", lib().strata_pack_q2_0(_p(canonical), _p(packed), n_blobs))


def strata_unpack_q2_0(packed, canonical, n_blobs):
    _check("strata_unpack_q2_0", lib().strata_unpack_q2_0(_p(packed), _p(canonical), n_blobs))


def strata_pack_q2_0_device(canonical, src_stride, packed, dst_stride, n_blobs, stream=None):
    _check("strata_pack_q2_0_device", lib().strata_pack_q2_0_device(_p(canonical), src_stride, _p(packed),
                                                                    dst_stride, n_blobs, _s(stream)))


def strata_poll_status(ws, stream=None) -> int:
    """Synchronise and return the workspace status (0 = STRATA_OK); does not raise."""
    return lib().strata_poll_status(_p(ws), _s(stream))


def strata_clear_status(ws, stream=None):
    _check("strata_clear_status", lib().strata_clear_status(_p(ws), _s(stream)))


def strata_status_str(status: int) -> str:
    return lib().strata_status_str(status).decode()


# kernel ids of strata_moe_profile_arm (STRATA_KERNEL_* of the header)
KERNELS = ("DECODE_LAYER", "ROUTE_DECODE", "ROUTER_PREP", "ROUTER_TC", "TOP_K", "GROUP_HIST", "GROUP_SCAN",
           "GROUP_SCATTER", "TC_PREPARE", "TC_GATHER",
           "TC_GATEUP", "TC_DOWN", "COMBINE", "PACK", "HOST_COPY", "WAIT_SELFTEST", "BLOB_CRC32")
KERNEL_ID = {name: i for i, name in enumerate(KERNELS)}


def strata_moe_launch_count() -> int:
    return int(lib().strata_moe_launch_count())


def strata_moe_profile_arm(kernel, start_events, stop_events, skip=0):
    """Arm event timing of `kernel` (name or id) for this thread with lists of torch.cuda.Event (or raw
    cudaEvent_t handles), after `skip` unrecorded launches; returns the ctypes arrays, which the caller
    must keep alive while armed.  Empty lists disarm."""
    kid = KERNEL_ID[kernel] if isinstance(kernel, str) else int(kernel)
    n = len(start_events)
    if len(stop_events) != n:
        raise ValueError("start and stop event lists differ in length")

    def handle(ev):
        h = ev if isinstance(ev, int) else ev.cuda_event
        if not h:
            raise ValueError("event has no CUDA handle yet (torch creates it on its first record())")
        return h

    arr_t = ctypes.c_void_p * max(n, 1)
    a = arr_t(*[handle(e) for e in start_events])
    b = arr_t(*[handle(e) for e in stop_events])
    _check("strata_moe_profile_arm", lib().strata_moe_profile_arm(kid, skip, a if n else None, b if n else None, n))
    return a, b


def strata_moe_profile_recorded(kernel) -> int:
    kid = KERNEL_ID[kernel] if isinstance(kernel, str) else int(kernel)
    return int(lib().strata_moe_profile_recorded(kid))
