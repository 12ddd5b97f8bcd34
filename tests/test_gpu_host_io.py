"""GPU tests of the host-buffer calls (strata_moe_layer_host / strata_moe_stack_host): the same results as
the device-buffer calls on the same inputs (bit for bit for decode; for prefill up to the order of the
fused combine's fp32 additions), through the graph path (page-locked buffers
on a side stream, first call captured, later calls replayed) and the direct path (pageable buffers or
the default stream), with the kernel copies (page-locked buffers) and the copy engines (pageable); and
the oracle on the host path's output."""
import numpy as np
import pytest
import torch

import gen
import oracle
import quantized_routed_expert_top10_gb300 as qre
from gpu_common import (DEV, BlobCache, assert_equal_up_to_sum_order, check_close, check_routing,
                        device_packed_layer, to_dev, workspace)


def assert_same_result(got, want, T, what, layers=1):
    """Decode (T <= 8) results repeat bit for bit; prefill results up to the fused combine's order."""
    if T <= 8:
        np.testing.assert_array_equal(got, want)
    else:
        assert_equal_up_to_sum_order(got, want, 10 * layers * np.abs(want).max(), what)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def layers():
    """Seed-0 experts of layers 0-2 packed on the device, and the host blob cache for the oracle."""
    blobs = [device_packed_layer(0, l) for l in range(3)]
    yield blobs, BlobCache(0)
    del blobs
    torch.cuda.empty_cache()


def device_call(ex, wr, bias, x, flags, ws, stream):
    out = torch.empty(x.shape, dtype=torch.float32, device=DEV)
    with torch.cuda.stream(stream):
        qre.strata_moe_layer(ex, wr, bias, to_dev(x), x.shape[0], flags, out, None, None, ws, stream=stream)
    stream.synchronize()
    return out.cpu().numpy()


def host_buffers(T, pinned):
    if pinned:
        return (torch.empty(T, qre.H, dtype=torch.float32).pin_memory(),
                torch.empty(T, qre.H, dtype=torch.float32).pin_memory())
    return np.empty((T, qre.H), dtype=np.float32), np.empty((T, qre.H), dtype=np.float32)


def fill(buf, x):
    if isinstance(buf, torch.Tensor):
        buf.copy_(torch.from_numpy(x))
    else:
        buf[...] = x


def as_np(buf):
    return buf.numpy().copy() if isinstance(buf, torch.Tensor) else buf.copy()


@pytest.mark.parametrize("T,flags,pinned", [(1, 0, True), (4, 0, True), (4, 1, False), (8, 1, True),
                                            (64, 0, True), (300, 1, False), (500, 0, True)])
def test_layer_host_matches_device_call(layers, T, flags, pinned):
    blobs, _ = layers
    ex = qre.experts(blobs[0])
    wr = to_dev(gen.router_weights(0, 0))
    bias = to_dev(gen.zipf_bias(0, 0))
    ws = workspace(T)
    s = torch.cuda.Stream()
    hx, ho = host_buffers(T, pinned)
    # page-locked activations: one copy kernel in; a decode layer writes out_host directly, a prefill
    # layer's output is copied out by a second copy kernel
    extra = (1 if T <= 8 else 2) if pinned else 0
    for it in range(3):  # the first call captures, the next two replay (pinned); new x every call
        x = (gen.activations_fast(40 + it, T) * (2.0 if flags else 1.0)).astype(np.float32)
        fill(hx, x)
        n0 = qre.strata_moe_launch_count()
        qre.strata_moe_layer_host(ex, wr, bias, hx, T, flags, ho, None, None, ws, stream=s)
        n1 = qre.strata_moe_launch_count()
        got = as_np(ho)
        want = device_call(ex, wr, bias, x, flags, ws, s)
        n2 = qre.strata_moe_launch_count()
        assert_same_result(got, want, T, "host layer call")
        assert n2 - n1 >= 1
        assert n1 - n0 == n2 - n1 + extra  # replays count the graph's kernels
    assert qre.strata_poll_status(ws) == 0


def test_layer_host_at_the_largest_chunk(layers):
    """T = 8,192 (the ABI's maximum): page-locked buffers of 84 MB each way through the mapped path."""
    blobs, _ = layers
    T = 8192
    ex = qre.experts(blobs[1])
    wr = to_dev(gen.router_weights(0, 1))
    bias = to_dev(gen.zipf_bias(0, 1))
    ws = workspace(T)
    s = torch.cuda.Stream()
    hx, ho = host_buffers(T, True)
    x = gen.activations_fast(90, T)
    fill(hx, x)
    for _ in range(2):
        qre.strata_moe_layer_host(ex, wr, bias, hx, T, 1, ho, None, None, ws, stream=s)
    assert_same_result(as_np(ho), device_call(ex, wr, bias, x, 1, ws, s), T, "largest chunk")
    assert qre.strata_poll_status(ws) == 0
    del ws
    torch.cuda.empty_cache()


def test_prepared_calls_repeat_the_call(layers):
    blobs, _ = layers
    T = 4
    ex = qre.experts(blobs[0])
    wr = to_dev(gen.router_weights(0, 0))
    ws = workspace(T)
    s = torch.cuda.Stream()
    hx, ho = host_buffers(T, True)
    call = qre.prepare_layer_host(ex, wr, None, hx, T, 0, ho, None, None, ws, stream=s)
    for it in range(3):
        x = gen.activations_fast(70 + it, T)
        fill(hx, x)
        call()
        np.testing.assert_array_equal(as_np(ho), device_call(ex, wr, None, x, 0, ws, s))
    L = 2
    exs = [qre.experts(b) for b in blobs[:L]]
    wrs = to_dev(np.concatenate([gen.router_weights(0, l) for l in range(L)]))
    stack = qre.prepare_stack_host(exs, wrs, None, L, hx, T, None, None, ws, stream=s)
    x = gen.activations_fast(80, T)
    fill(hx, x)
    stack()
    xd = to_dev(x)
    with torch.cuda.stream(s):
        qre.strata_moe_stack(exs, wrs, None, L, xd, T, None, None, ws, stream=s)
    s.synchronize()
    np.testing.assert_array_equal(as_np(hx), xd.cpu().numpy())


def test_layer_host_on_default_stream(layers):
    blobs, _ = layers
    ex = qre.experts(blobs[0])
    wr = to_dev(gen.router_weights(0, 0))
    T = 4
    ws = workspace(T)
    hx, ho = host_buffers(T, True)
    x = gen.verify_window(0, T)
    fill(hx, x)
    qre.strata_moe_layer_host(ex, wr, None, hx, T, 0, ho, None, None, ws, stream=0)
    np.testing.assert_array_equal(as_np(ho), device_call(ex, wr, None, x, 0, ws, torch.cuda.Stream()))


def test_layer_host_parity_with_oracle(layers):
    """The verify window through the host path against the oracle (routing up to ties, outputs to 2e-3)."""
    blobs, cache = layers
    T = 4
    x = gen.verify_window(0, T)
    wr_h = gen.router_weights(0, 0)
    ws = workspace(T)
    ids = torch.empty(T, qre.K, dtype=torch.int32, device=DEV)
    hx, ho = host_buffers(T, True)
    fill(hx, x)
    s = torch.cuda.Stream()
    for _ in range(2):
        qre.strata_moe_layer_host(qre.experts(blobs[0]), to_dev(wr_h), None, hx, T, 0, ho, ids, None, ws, stream=s)
    ids_h = ids.cpu().numpy()
    ref_r = oracle.route(x, wr_h, None, residual=False)
    check_routing(ids_h, ref_r["ids"], ref_r["logits"])
    ref = oracle.moe_layer(x, wr_h, None, cache.layer_list(0, ids_h, 512), ids_in=ids_h)
    check_close(as_np(ho), ref["out"], "host-buffer layer output")


@pytest.mark.parametrize("T,pinned", [(1, True), (4, False), (20, True)])
def test_stack_host_matches_device_call(layers, T, pinned):
    blobs, _ = layers
    L = 3
    exs = [qre.experts(b) for b in blobs]
    wr = to_dev(np.concatenate([gen.router_weights(0, l) for l in range(L)]))
    bias = to_dev(np.concatenate([gen.zipf_bias(0, l) for l in range(L)]))
    ws = workspace(T)
    s = torch.cuda.Stream()
    hx, _ = host_buffers(T, pinned)
    for it in range(2):
        x = gen.activations_fast(60 + it, T)
        fill(hx, x)
        qre.strata_moe_stack_host(exs, wr, bias, L, hx, T, None, None, ws, stream=s)
        xd = to_dev(x)
        with torch.cuda.stream(s):
            qre.strata_moe_stack(exs, wr, bias, L, xd, T, None, None, ws, stream=s)
        s.synchronize()
        assert_same_result(as_np(hx), xd.cpu().numpy(), T, "host stack call", layers=L)
    assert qre.strata_poll_status(ws) == 0


def test_host_call_refused_inside_capture(layers):
    blobs, _ = layers
    T = 4
    ws = workspace(T)
    hx, ho = host_buffers(T, True)
    ex = qre.experts(blobs[0])
    wr = to_dev(gen.router_weights(0, 0))
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with pytest.raises(qre.StrataError):
        with torch.cuda.graph(g, stream=s):
            qre.strata_moe_layer_host(ex, wr, None, hx, T, 0, ho, None, None, ws, stream=s)
