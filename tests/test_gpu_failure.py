"""Failure detection on the GPU without a fault: the library's bounded waits, run on conditions that
never hold (a tag nothing writes, an mbarrier phase nothing completes) with a short limit, expire,
report STRATA_E_TIMEOUT through the workspace's status word, and leave the context usable."""
import time

import numpy as np
import pytest
import torch

import gen
import quantized_routed_expert_top10_gb300 as qre
from gpu_common import device_packed_layer, run_layer, workspace

pytestmark = pytest.mark.gpu

TIMEOUT = -5  # STRATA_E_TIMEOUT


@pytest.mark.parametrize("limit_ns", [20_000, 1_000_000])
def test_expired_waits_report_timeout(limit_ns):
    ws = workspace(1)
    assert qre.strata_poll_status(ws) == 0
    t0 = time.perf_counter()
    qre.strata_moe_wait_selftest(ws, limit_ns)
    st = qre.strata_poll_status(ws)  # synchronises
    elapsed = time.perf_counter() - t0
    assert st == TIMEOUT
    assert elapsed < 1.0  # both waits gave up near their limit: nothing hung
    qre.strata_clear_status(ws)
    assert qre.strata_poll_status(ws) == 0


def test_context_usable_after_a_timeout():
    """After an expired wait and a cleared status, the same workspace runs a layer that matches a
    layer run on a fresh workspace bit for bit."""
    blobs = device_packed_layer(0, 0)
    x = gen.verify_window(0, 4)
    wr = gen.router_weights(0, 0)
    ws = workspace(4)
    qre.strata_moe_wait_selftest(ws, 50_000)
    assert qre.strata_poll_status(ws) == TIMEOUT
    qre.strata_clear_status(ws)
    out, ids, w = run_layer(blobs, wr, None, x, ws=ws)
    ref_out, ref_ids, ref_w = run_layer(blobs, wr, None, x)
    np.testing.assert_array_equal(ids, ref_ids)
    np.testing.assert_array_equal(out, ref_out)
    del blobs
    torch.cuda.empty_cache()
