"""GPU parity of strata_moe_layer (steps 1-5 through the C ABI) against the oracle."""
import numpy as np
import pytest
import torch

import gen
import oracle
import quantized_routed_expert_top10_gb300 as qre
from gpu_common import (W_TOL, DEV, BlobCache, assert_equal_up_to_sum_order, check_close, check_routing,
                        device_packed_layer, run_layer, to_dev, workspace)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def layer0():
    """Seed-0 layer-0 experts packed on the device, and the host blob cache for the oracle."""
    blobs = device_packed_layer(0, 0)
    yield blobs, BlobCache(0)
    del blobs
    torch.cuda.empty_cache()


def parity(layer0, x, wr, bias, flags=0, q2_offset=1, E=512):
    blobs, cache = layer0
    out, ids, w = run_layer(blobs, wr, bias, x, flags, q2_offset, E=E)
    ref_r = oracle.route(x, wr, bias, residual=bool(flags))
    ties = check_routing(ids, ref_r["ids"], ref_r["logits"])
    ref = oracle.moe_layer(x, wr, bias, cache.layer_list(0, ids, E), q2_offset=q2_offset, residual=bool(flags),
                           ids_in=ids)
    np.testing.assert_allclose(w, ref["w"], rtol=0, atol=W_TOL)
    if flags:
        check_close(out - x, ref["out"] - x.astype(np.float64), "moe part of residual layer")
    else:
        check_close(out, ref["out"], "layer output")
    return ties


@pytest.mark.parametrize("q2_offset", [1, 2])
def test_config0_decode_one_token(layer0, q2_offset):
    parity(layer0, gen.activations_fast(0, 1), gen.router_weights(0, 0), None, q2_offset=q2_offset)


def test_config1_verify_window(layer0):
    parity(layer0, gen.verify_window(0, 4), gen.router_weights(0, 0), None)


@pytest.mark.parametrize("T", [2, 3, 5, 8, 9, 37, 300])
def test_ragged_token_counts_with_zipf_bias(layer0, T):
    parity(layer0, gen.activations_fast(11, T), gen.router_weights(0, 0), gen.zipf_bias(0, 0))


@pytest.mark.parametrize("E,T", [(256, 1), (256, 4), (256, 8), (256, 300), (32, 4), (32, 64)])
def test_smaller_expert_counts(layer0, E, T):
    """The 256-expert variant (and the smallest E the ABI takes): routing over the first E experts of
    the layer, decode (T <= 8) and prefill paths."""
    parity(layer0, gen.activations_fast(13, T), gen.router_weights(0, 0, E_=E), None, E=E)


@pytest.mark.parametrize("T", [1, 3, 20])
def test_residual_rmsnorm_layer(layer0, T):
    x = 3.0 * gen.activations_fast(5, T)
    parity(layer0, x.astype(np.float32), gen.router_weights(0, 0), gen.zipf_bias(0, 0), flags=1)


def test_every_token_on_the_same_ten_experts(layer0):
    """Degenerate routing: 64 tokens all pick the same ten experts (groups of 64, several tiles)."""
    bias = np.zeros(512, dtype=np.float32)
    hot = [5, 17, 99, 130, 255, 256, 300, 411, 500, 511]
    bias[hot] = 50.0
    blobs, cache = layer0
    x = gen.activations_fast(2, 64)
    wr = gen.router_weights(0, 0)
    out, ids, w = run_layer(blobs, wr, bias, x)
    assert np.all(np.sort(ids, axis=1) == np.array(hot))
    parity(layer0, x, wr, bias)


@pytest.mark.parametrize("T", [1, 20])
def test_equal_logits_pick_lowest_ids(layer0, T):
    blobs, cache = layer0
    wr = np.zeros((512, 2560), dtype=np.uint16)
    x = gen.activations_fast(4, T)
    out, ids, w = run_layer(blobs, wr, None, x)
    assert np.all(ids == np.arange(10)) and np.all(w == np.float32(0.1))
    ref = oracle.moe_layer(x, wr, None, cache.layer_list(0, ids), ids_in=ids)
    check_close(out, ref["out"], "equal-logit layer")


def test_empty_call_is_a_no_op(layer0):
    blobs, _ = layer0
    ws = workspace(1)
    out = torch.full((1, qre.H), 7.0, device=DEV)
    x = torch.zeros(1, qre.H, device=DEV)
    wr = torch.zeros(512, qre.H, dtype=torch.int16, device=DEV)
    qre.strata_moe_layer(qre.experts(blobs), wr, None, x, 0, 0, out, None, None, ws)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)


def test_out_may_alias_x(layer0):
    blobs, cache = layer0
    T = 4
    x = gen.activations_fast(9, T)
    wr = gen.router_weights(0, 0)
    ref_out, _, _ = run_layer(blobs, wr, None, x, flags=1)
    xd = to_dev(x)
    ws = workspace(T)
    qre.strata_moe_layer(qre.experts(blobs), to_dev(wr), None, xd, T, 1, xd, None, None, ws)
    assert qre.strata_poll_status(ws) == 0
    np.testing.assert_array_equal(xd.cpu().numpy(), ref_out)


@pytest.mark.parametrize("T", [4, 300])
def test_repeat_calls(layer0, T):
    """Decode layers (T <= 8) repeat bit for bit.  Prefill layers repeat their routing bit for bit and
    their outputs up to the order of the fused combine's fp32 additions."""
    blobs, _ = layer0
    x = gen.activations_fast(6, T)
    wr = gen.router_weights(0, 0)
    bias = gen.zipf_bias(0, 0)
    a = run_layer(blobs, wr, bias, x)
    b = run_layer(blobs, wr, bias, x)
    np.testing.assert_array_equal(a[1], b[1])
    np.testing.assert_array_equal(a[2], b[2])
    if T <= 8:
        np.testing.assert_array_equal(a[0], b[0])
    else:
        assert_equal_up_to_sum_order(a[0], b[0], np.abs(b[0]).max(), "repeat prefill layer")


def test_epoch_wrap_clears_the_exchange_area(layer0):
    """The decode layer tags its exchange words with a call epoch kept in the workspace header (the
    int32 at byte 4096 + 4 * 32).  The call that takes the last tag, 0xFFFFFFFF, counts its CTAs out,
    clears the exchange area and restarts the epoch from 0; results stay the same throughout."""
    blobs, _ = layer0
    T = 4
    x = gen.verify_window(0, T)
    wr = gen.router_weights(0, 0)
    ref_out, ref_ids, _ = run_layer(blobs, wr, None, x)
    ws = workspace(T)
    epoch = ws[4224:4228]
    epoch.copy_(torch.tensor(np.array([0xFFFFFFFE], dtype=np.uint32).view(np.uint8), device=DEV))
    out, ids, _ = run_layer(blobs, wr, None, x, ws=ws)
    np.testing.assert_array_equal(out, ref_out)
    np.testing.assert_array_equal(ids, ref_ids)
    assert int(epoch.cpu().numpy().view(np.uint32)[0]) == 0
    area = ws[12288:12288 + 16 * 8 * 512 * 8]  # router words: cleared with the rest of the area
    assert int(torch.count_nonzero(area)) == 0
    out, ids, _ = run_layer(blobs, wr, None, x, ws=ws)
    np.testing.assert_array_equal(out, ref_out)
    assert int(epoch.cpu().numpy().view(np.uint32)[0]) == 1


@pytest.mark.parametrize("T", [4, 300])
def test_layers_interleaved_with_other_kernels_on_the_stream(layer0, T):
    """A layer call, a PyTorch kernel that rewrites its output on the same stream, then a second layer
    call on that: the second call must see the rewritten values (the prefill chain's kernels overlap
    one another's prologues, never the caller's work).  Each call is checked against the oracle on
    the input it was given."""
    blobs, cache = layer0
    wr = gen.router_weights(0, 0)
    bias = gen.zipf_bias(0, 0)
    x = gen.activations_fast(21, T)
    ws = workspace(T)
    ex = qre.experts(blobs)
    wr_d, bias_d = to_dev(wr), to_dev(bias)
    xd = to_dev(x)
    out1 = torch.empty(T, qre.H, dtype=torch.float32, device=DEV)
    out2 = torch.empty_like(out1)
    ids1 = torch.empty(T, qre.K, dtype=torch.int32, device=DEV)
    ids2 = torch.empty_like(ids1)
    w1 = torch.empty(T, qre.K, dtype=torch.float32, device=DEV)
    w2 = torch.empty_like(w1)
    qre.strata_moe_layer(ex, wr_d, bias_d, xd, T, 1, out1, ids1, w1, ws)
    first = out1.clone()  # a kernel reading the first call's output
    y = out1.mul_(0.5).add_(xd)  # in place on the layer's output, same stream, no synchronisation
    qre.strata_moe_layer(ex, wr_d, bias_d, y, T, 1, out2, ids2, w2, ws)
    torch.cuda.synchronize()
    assert qre.strata_poll_status(ws) == 0
    y_h = y.cpu().numpy()
    for inp, ids, w, out, what in ((x, ids1, w1, first, "first"), (y_h, ids2, w2, out2, "second")):
        ids_h = ids.cpu().numpy()
        ref_r = oracle.route(inp, wr, bias, residual=True)
        check_routing(ids_h, ref_r["ids"], ref_r["logits"])
        ref = oracle.moe_layer(inp, wr, bias, cache.layer_list(0, ids_h), residual=True, ids_in=ids_h)
        np.testing.assert_allclose(w.cpu().numpy(), ref["w"], rtol=0, atol=W_TOL)
        check_close(out.cpu().numpy() - inp, ref["out"] - inp.astype(np.float64), f"{what} layer's moe part")
