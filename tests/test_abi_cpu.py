"""C ABI checks that need no GPU: the library loads and exports every symbol the header declares,
the host packer is a byte permutation that matches the layout the header documents, and host-side
argument checks reject bad calls before anything is enqueued."""
import ctypes
import os
import re

import numpy as np
import pytest

import gen
import quantized_routed_expert_top10_gb300 as qre
from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "strata_moe.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(strata_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(qre.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return qre.lib()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) == 23
    assert sorted(names) == sorted(qre.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_prepared_calls_marshal_and_report_errors(lib):
    """The binding's prepared host calls pass their fixed arguments on every call; a call the library
    rejects before touching the device raises each time it is repeated."""
    A = 1 << 20
    ex = qre.experts(A, 512, 1)
    hx = np.zeros((4, 2560), dtype=np.float32)
    ho = np.zeros((4, 2560), dtype=np.float32)
    ws_big = qre.strata_moe_workspace_bytes(4)
    bad = qre.prepare_layer_host(ex, A, None, hx, 4, 2, ho, None, None, A, ws_bytes=ws_big, stream=0)  # flags
    for _ in range(2):
        with pytest.raises(qre.StrataError) as e:
            bad()
        assert e.value.status == -1
    empty = qre.prepare_layer_host(ex, A, None, hx, 0, 0, ho, None, None, A, ws_bytes=ws_big, stream=0)
    empty()  # T = 0: valid, nothing enqueued
    bad_stack = qre.prepare_stack_host([ex, qre.experts(A, 100, 1)], A, None, 2, hx, 4, None, None, A,
                                       ws_bytes=ws_big, stream=0)
    with pytest.raises(qre.StrataError):
        bad_stack()


def test_status_strings(lib):
    for code, name in qre.STATUS.items():
        assert qre.strata_status_str(code).startswith(name)
    assert "unknown" in qre.strata_status_str(42)


def test_workspace_sizes(lib):
    assert qre.strata_moe_workspace_bytes(-1) == 0
    assert qre.strata_moe_workspace_bytes(8193) == 0
    sizes = [qre.strata_moe_workspace_bytes(t) for t in (0, 1, 4, 8, 9, 2048, 8192)]
    assert sizes[0] == 12288
    assert all(b > a for a, b in zip(sizes, sizes[1:]))
    assert all(s % 256 == 0 for s in sizes)


def test_pack_round_trip_and_documented_layout(lib):
    n = 2
    canon = np.concatenate([gen.canonical_blob(3, 1, e) for e in range(n)])
    packed = np.zeros_like(canon)
    qre.strata_pack_q2_0(canon, packed, n)
    assert not np.array_equal(packed, canon)
    assert np.array_equal(np.sort(packed), np.sort(canon))
    back = np.zeros_like(canon)
    qre.strata_unpack_q2_0(packed, back, n)
    np.testing.assert_array_equal(back, canon)
    # Spot checks against the layout in strata_moe.h.
    B = qre.BLOB_BYTES
    for j in range(n):
        c = canon[j * B:(j + 1) * B].reshape(-1, 18)
        p = packed[j * B:(j + 1) * B]
        for (r, kb) in ((0, 0), (129, 7), (639, 39)):
            blk = c[r * 40 + kb]                   # gate row r, k-block kb
            piece = ((r // 16) * 40 + kb) * 576
            rr = r % 16
            np.testing.assert_array_equal(p[piece + 16 * rr: piece + 16 * rr + 16], blk[2:])
            np.testing.assert_array_equal(p[piece + 512 + 4 * rr: piece + 512 + 4 * rr + 2], blk[:2])
            blk = c[25600 + r * 40 + kb]           # up
            np.testing.assert_array_equal(p[piece + 256 + 16 * rr: piece + 256 + 16 * rr + 16], blk[2:])
            np.testing.assert_array_equal(p[piece + 512 + 4 * rr + 2: piece + 512 + 4 * rr + 4], blk[:2])
        for (nr, kb) in ((0, 0), (1000, 3), (2559, 9)):
            blk = c[51200 + nr * 10 + kb]          # down row nr, k-block kb
            chunk = 921600 + ((nr // 128) * 10 + kb) * 2304
            np.testing.assert_array_equal(p[chunk + 16 * (nr % 128): chunk + 16 * (nr % 128) + 16], blk[2:])
            np.testing.assert_array_equal(p[chunk + 2048 + 2 * (nr % 128): chunk + 2048 + 2 * (nr % 128) + 2], blk[:2])


def test_blob_crc32_host_is_zlibs(lib):
    import zlib
    n, stride = 3, qre.BLOB_BYTES + 256
    buf = np.random.default_rng(5).integers(0, 256, n * stride, dtype=np.uint8)
    crc = np.zeros(n, dtype=np.uint32)
    qre.strata_blob_crc32(buf, n, crc, stride=stride)
    for j in range(n):
        assert int(crc[j]) == zlib.crc32(buf[j * stride: j * stride + qre.BLOB_BYTES].tobytes())
    buf[stride + 12345] ^= 1  # one flipped bit in blob 1 changes only its checksum
    crc2 = np.zeros(n, dtype=np.uint32)
    qre.strata_blob_crc32(buf, n, crc2, stride=stride)
    assert crc2[0] == crc[0] and crc2[2] == crc[2] and crc2[1] != crc[1]


def test_pack_rejects_overlap_and_null(lib):
    buf = np.zeros(2 * qre.BLOB_BYTES, dtype=np.uint8)
    with pytest.raises(qre.StrataError):
        qre.strata_pack_q2_0(buf, buf[1000:], 1)
    assert lib.strata_pack_q2_0(None, buf.ctypes.data, 1) == -1
    assert lib.strata_unpack_q2_0(buf.ctypes.data, None, 1) == -1


def _rc(fn, *args):
    return fn(*args)


def test_host_argument_checks(lib):
    """Every rejected call returns before touching the device (no GPU here)."""
    A = 1 << 20  # fake, 256-aligned addresses: never dereferenced because the checks fail first
    ws_big = qre.strata_moe_workspace_bytes(16)
    # T out of range / null pointers / bad E
    assert lib.strata_moe_route(A, -1, A, None, 512, A, A, None, A, ws_big, None) == -1
    assert lib.strata_moe_route(A, 8193, A, None, 512, A, A, None, A, ws_big, None) == -1
    assert lib.strata_moe_route(None, 4, A, None, 512, A, A, None, A, ws_big, None) == -1
    assert lib.strata_moe_route(A, 4, A, None, 500, A, A, None, A, ws_big, None) == -1
    assert lib.strata_moe_route(A, 4, A, None, 1024, A, A, None, A, ws_big, None) == -1
    # misaligned x / ws
    assert lib.strata_moe_route(A + 4, 4, A, None, 512, A, A, None, A, ws_big, None) == -2
    assert lib.strata_moe_route(A, 4, A, None, 512, A, A, None, A + 16, ws_big, None) == -2
    # workspace too small
    assert lib.strata_moe_route(A, 16, A, None, 512, A, A, None, A, 4096, None) == -6
    # experts struct checks
    ex = qre.experts(A, 512, 1)
    bad_off = qre.experts(A, 512, 3)
    bad_stride = qre.experts(A, 512, 1, qre.BLOB_BYTES + 16)
    bad_e = qre.experts(A, 100, 1)
    bad_align = qre.experts(A + 128, 512, 1)
    for e, want in ((bad_off, -1), (bad_stride, -2), (bad_e, -1), (bad_align, -2)):
        assert lib.strata_moe_layer(ctypes.byref(e), A, None, A, 4, 0, A, None, None, A, ws_big, None) == want
    assert lib.strata_moe_layer(ctypes.byref(ex), A, None, A, 4, 2, A, None, None, A, ws_big, None) == -1
    assert lib.strata_moe_layer(None, A, None, A, 4, 0, A, None, None, A, ws_big, None) == -1
    assert lib.strata_moe_combine(None, A, 4, None, A, None) == -1
    assert lib.strata_moe_combine(A, A, 4, None, A + 8, None) == -2
    assert lib.strata_moe_group(A, 4, 512, None, A, A, A, A, ws_big, None) == -1
    assert lib.strata_moe_experts(ctypes.byref(ex), A, 9000, A, A, A, A, A, A, ws_big, None) == -1
    assert lib.strata_moe_stack(None, A, None, 2, A, 4, None, None, A, ws_big, None) == -1
    assert lib.strata_moe_group_noalloc(A, -1, 512, A, A, A, A, None) == -1
    assert lib.strata_moe_group_noalloc(A, 8193, 512, A, A, A, A, None) == -1
    assert lib.strata_moe_group_noalloc(A, 4, 512, A + 2, A, A, A, None) == -2
    assert lib.strata_moe_group_noalloc(A, 4, 512, None, A, A, A, None) == -1
    assert lib.strata_moe_group_noalloc(A, 0, 512, A, A, A, A, None) == 0
    assert lib.strata_pack_q2_0_device(A, qre.BLOB_BYTES, A + 16, qre.BLOB_BYTES, 1, None) == -2
    assert lib.strata_moe_workspace_init(A + 8, 4096, None) == -2
    assert lib.strata_moe_workspace_init(A, 100, None) == -6
    # host-buffer calls: the same checks, made before the device is touched
    hx = np.zeros((4, 2560), dtype=np.float32)
    ho = np.zeros((4, 2560), dtype=np.float32)
    xp, op = hx.ctypes.data, ho.ctypes.data
    lh, sh = lib.strata_moe_layer_host, lib.strata_moe_stack_host
    assert lh(ctypes.byref(ex), A, None, xp, -1, 0, op, None, None, A, ws_big, None) == -1
    assert lh(ctypes.byref(ex), A, None, None, 4, 0, op, None, None, A, ws_big, None) == -1
    assert lh(ctypes.byref(ex), A, None, xp, 4, 0, None, None, None, A, ws_big, None) == -1
    assert lh(ctypes.byref(ex), A, None, xp, 4, 0, xp + 4096, None, None, A, ws_big, None) == -1  # overlap
    assert lh(ctypes.byref(ex), A, None, xp, 4, 2, op, None, None, A, ws_big, None) == -1         # flags
    assert lh(ctypes.byref(bad_off), A, None, xp, 4, 0, op, None, None, A, ws_big, None) == -1
    assert lh(ctypes.byref(bad_align), A, None, xp, 4, 0, op, None, None, A, ws_big, None) == -2
    assert lh(ctypes.byref(ex), A + 2, None, xp, 4, 0, op, None, None, A, ws_big, None) == -2
    assert lh(ctypes.byref(ex), A, None, xp, 16, 0, op, None, None, A, 4096, None) == -6
    assert lh(ctypes.byref(ex), A, None, xp, 0, 0, op, None, None, A, ws_big, None) == 0
    exs = (qre.strata_experts_t * 2)(ex, bad_e)
    assert sh(exs, A, None, 2, xp, 4, None, None, A, ws_big, None) == -1
    assert sh(exs, A, None, -1, xp, 4, None, None, A, ws_big, None) == -1
    assert sh(exs, A, None, 1, None, 4, None, None, A, ws_big, None) == -1
    assert sh(exs, A, None, 1, xp, 4, None, None, A, 1024, None) == -6
    assert sh(exs, A, None, 0, xp, 4, None, None, A, ws_big, None) == 0
    # the wait self-test: workspace and limit checked before the device is touched
    ws1 = qre.strata_moe_workspace_bytes(1)
    assert lib.strata_moe_wait_selftest(None, ws1, 10000, None) == -1
    assert lib.strata_moe_wait_selftest(A + 16, ws1, 10000, None) == -2
    assert lib.strata_moe_wait_selftest(A, 1024, 10000, None) == -6
    assert lib.strata_moe_wait_selftest(A, ws1, 999, None) == -1
    assert lib.strata_moe_wait_selftest(A, ws1, 2000000001, None) == -1
    # blob checksums: sizes, pointers and alignment checked first
    assert lib.strata_blob_crc32(None, qre.BLOB_BYTES, 1, A) == -1
    assert lib.strata_blob_crc32(A, qre.BLOB_BYTES - 1, 1, A) == -1
    assert lib.strata_blob_crc32(A, qre.BLOB_BYTES, -1, A) == -1
    assert lib.strata_blob_crc32(None, qre.BLOB_BYTES, 0, None) == 0
    assert lib.strata_blob_crc32_device(A, qre.BLOB_BYTES, -1, A, None) == -1
    assert lib.strata_blob_crc32_device(None, qre.BLOB_BYTES, 2, A, None) == -1
    assert lib.strata_blob_crc32_device(A + 16, qre.BLOB_BYTES, 2, A, None) == -2
    assert lib.strata_blob_crc32_device(A, qre.BLOB_BYTES + 16, 2, A, None) == -2
    assert lib.strata_blob_crc32_device(A, qre.BLOB_BYTES, 2, A + 2, None) == -2
    assert lib.strata_blob_crc32_device(A, qre.BLOB_BYTES, 0, A, None) == 0
    # empty calls are valid and enqueue nothing
    assert lib.strata_moe_route(A, 0, A, None, 512, A, A, None, A, ws_big, None) == 0
    assert lib.strata_moe_layer(ctypes.byref(ex), A, None, A, 0, 0, A, None, None, A, ws_big, None) == 0
    assert lib.strata_moe_combine(A, A, 0, None, A, None) == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(qre, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(qre, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        qre.lib()


def test_profile_arm_argument_checks(lib):
    assert lib.strata_moe_profile_arm(-1, 0, None, None, 0) == -1
    assert lib.strata_moe_profile_arm(qre.KERNEL_ID["TC_GATEUP"], 0, None, None, 2) == -1
    assert lib.strata_moe_profile_arm(qre.KERNEL_ID["TC_GATEUP"], -1, None, None, 0) == -1
    assert lib.strata_moe_profile_arm(qre.KERNEL_ID["TC_GATEUP"], 0, None, None, 0) == 0
    assert lib.strata_moe_profile_recorded(qre.KERNEL_ID["TC_GATEUP"]) == 0
    assert lib.strata_moe_profile_recorded(len(qre.KERNELS)) == -1
    assert lib.strata_moe_launch_count() >= 0


def test_kernel_ids_match_header():
    src = open(HEADER).read()
    ids = dict((m.group(1), int(m.group(2))) for m in re.finditer(r"#define STRATA_KERNEL_([A-Z0-9_]+) (\d+)", src))
    assert ids.pop("COUNT") == len(qre.KERNELS)
    assert ids == qre.KERNEL_ID
