"""Blob checksums on the device (strata_blob_crc32_device) against zlib's CRC-32 of the same bytes
on the host: a device pack of a whole layer, a padded stride, and a single flipped bit."""
import zlib

import numpy as np
import pytest
import torch

import quantized_routed_expert_top10_gb300 as qre
from gpu_common import DEV, device_packed_layer

pytestmark = pytest.mark.gpu
B = qre.BLOB_BYTES


def device_crc(blobs, n, stride=B):
    crc = torch.zeros(n, dtype=torch.int32, device=DEV)
    qre.strata_blob_crc32_device(blobs, n, crc, stride=stride)
    torch.cuda.synchronize()
    return crc.cpu().numpy().view(np.uint32)


def test_device_pack_of_a_layer_matches_the_host():
    """All 512 experts of a layer packed on the device: device checksums = zlib over the bytes read
    back = the host call's checksums."""
    blobs = device_packed_layer(0, 0)
    got = device_crc(blobs, 512)
    host = blobs.cpu().numpy()
    want = np.array([zlib.crc32(host[j * B:(j + 1) * B].tobytes()) for j in range(512)], dtype=np.uint32)
    np.testing.assert_array_equal(got, want)
    hc = np.zeros(512, dtype=np.uint32)
    qre.strata_blob_crc32(host, 512, hc)
    np.testing.assert_array_equal(hc, want)
    del blobs
    torch.cuda.empty_cache()


def test_padded_stride_and_a_flipped_bit():
    n, stride = 5, B + 512
    host = np.random.default_rng(7).integers(0, 256, n * stride, dtype=np.uint8)
    dev = torch.from_numpy(host).to(DEV)
    want = np.array([zlib.crc32(host[j * stride: j * stride + B].tobytes()) for j in range(n)], dtype=np.uint32)
    np.testing.assert_array_equal(device_crc(dev, n, stride), want)
    dev[3 * stride + B - 1] ^= 0x80  # last byte of blob 3
    got = device_crc(dev, n, stride)
    assert got[3] != want[3]
    np.testing.assert_array_equal(np.delete(got, 3), np.delete(want, 3))
