"""Decode stacks of one to four tokens: strata_moe_stack runs the layers as a chain of one-layer
launches that look one layer ahead (the next router on this layer's input names the experts the next
launch prefetches) and alternate between x and a workspace buffer.  The lookahead is a hint, so the
stack must equal the same layers run one strata_moe_layer call at a time bit for bit (ids, weights and
activations), for every token count, for stacks of any length and across the exchange area's epoch
wrap; the stack's last layer is also checked against the oracle on the input the GPU gave it."""
import numpy as np
import pytest
import torch

import gen
import oracle
import quantized_routed_expert_top10_gb300 as qre
from gpu_common import DEV, B, BlobCache, check_close, check_routing, device_packed_layer, to_dev, workspace

pytestmark = pytest.mark.gpu
E = 512
NL = 4  # distinct layers of blobs and routers; longer stacks cycle through them
K = qre.K


@pytest.fixture(scope="module")
def layers():
    blobs = [device_packed_layer(0, l) for l in range(NL)]
    wr = np.stack([gen.router_weights(0, l) for l in range(NL)])
    bias = np.stack([gen.zipf_bias(0, l) for l in range(NL)])
    yield blobs, wr, bias
    del blobs
    torch.cuda.empty_cache()


def tokens(T, seed=40):
    return gen.verify_window(seed, T) if T > 1 else gen.activations_fast(seed, 1)


def run_chain(exs, wr_d, bias_d, x, T, ws):
    """The layers one strata_moe_layer call at a time: (inputs, ids, weights, final x)."""
    xl = to_dev(x)
    ins, ids, wts = [], [], []
    idl = torch.empty(T, K, dtype=torch.int32, device=DEV)
    wl = torch.empty(T, K, dtype=torch.float32, device=DEV)
    for l in range(len(exs)):
        ins.append(xl.cpu().numpy())
        qre.strata_moe_layer(exs[l], wr_d[l], bias_d[l], xl, T, qre.RESIDUAL_RMSNORM, xl, idl, wl, ws)
        ids.append(idl.cpu().numpy())
        wts.append(wl.cpu().numpy())
    assert qre.strata_poll_status(ws) == 0
    return ins, np.stack(ids), np.stack(wts), xl.cpu().numpy()


def run_stack(exs, wr_d, bias_d, x, T, ws, with_outputs=True):
    n = len(exs)
    xs = to_dev(x)
    ids = torch.full((n, T, K), -1, dtype=torch.int32, device=DEV) if with_outputs else None
    wts = torch.zeros(n, T, K, dtype=torch.float32, device=DEV) if with_outputs else None
    qre.strata_moe_stack(exs, wr_d, bias_d, n, xs, T, ids, wts, ws)
    assert qre.strata_poll_status(ws) == 0
    return (ids.cpu().numpy() if with_outputs else None), (wts.cpu().numpy() if with_outputs else None), xs.cpu().numpy()


@pytest.mark.parametrize("T", [1, 2, 3, 4])
@pytest.mark.parametrize("n_layers", [2, 3, 5])
def test_stack_equals_layer_chain(layers, T, n_layers):
    blobs, wr, bias = layers
    sel = [l % NL for l in range(n_layers)]
    exs = [qre.experts(blobs[i]) for i in sel]
    wr_d, bias_d = to_dev(wr[sel]), to_dev(bias[sel])
    x = tokens(T)
    ws = workspace(T)
    ids_s, w_s, x_s = run_stack(exs, wr_d, bias_d, x, T, ws)
    ins, ids_c, w_c, x_c = run_chain(exs, wr_d, bias_d, x, T, ws)
    np.testing.assert_array_equal(ids_s, ids_c)
    np.testing.assert_array_equal(w_s, w_c)
    np.testing.assert_array_equal(x_s, x_c)
    # the last layer against the oracle, on the input the GPU gave it
    l = n_layers - 1
    r = oracle.route(ins[l], wr[sel[l]], bias[sel[l]], residual=True)
    check_routing(ids_s[l], r["ids"], r["logits"])
    ref = oracle.moe_layer(ins[l], wr[sel[l]], bias[sel[l]], BlobCache(0).layer_list(sel[l], ids_s[l]),
                           residual=True, ids_in=ids_s[l])
    check_close(x_s - ins[l], ref["out"] - ins[l].astype(np.float64), f"T={T} stack layer {l}")


@pytest.mark.parametrize("n_layers", [65, 66])
def test_long_stacks(layers, n_layers):
    """65 and 66 layers (odd and even: an odd stack ends with a copy back into x)."""
    blobs, wr, bias = layers
    T = 1
    sel = [l % NL for l in range(n_layers)]
    exs = [qre.experts(blobs[i]) for i in sel]
    wr_d, bias_d = to_dev(wr[sel]), to_dev(bias[sel])
    x = tokens(T, seed=41)
    ws = workspace(T)
    ids_s, w_s, x_s = run_stack(exs, wr_d, bias_d, x, T, ws)
    _, ids_c, w_c, x_c = run_chain(exs, wr_d, bias_d, x, T, ws)
    np.testing.assert_array_equal(ids_s, ids_c)
    np.testing.assert_array_equal(w_s, w_c)
    np.testing.assert_array_equal(x_s, x_c)


def test_stack_without_outputs(layers):
    """ids and weights are optional: the activations are the same without them."""
    blobs, wr, bias = layers
    T, n = 4, 3
    exs = [qre.experts(blobs[l]) for l in range(n)]
    wr_d, bias_d = to_dev(wr[:n]), to_dev(bias[:n])
    x = tokens(T, seed=42)
    ws = workspace(T)
    _, _, x_a = run_stack(exs, wr_d, bias_d, x, T, ws, with_outputs=False)
    _, _, x_b = run_stack(exs, wr_d, bias_d, x, T, ws)
    np.testing.assert_array_equal(x_a, x_b)


def test_stack_epoch_wrap(layers):
    """A stack across the epoch wrap (the int32 at byte 4096 + 4 * 32 of the workspace): the layer that
    takes tag 0xFFFFFFFF clears the exchange area and restarts the epoch from 0, the next layer takes
    tag 1, and the lookahead words of the layer before the wrap are not mistaken for the next's; the
    results are those of a fresh workspace."""
    blobs, wr, bias = layers
    T, n = 2, 3
    exs = [qre.experts(blobs[l]) for l in range(n)]
    wr_d, bias_d = to_dev(wr[:n]), to_dev(bias[:n])
    x = tokens(T, seed=43)
    ids_a, w_a, x_a = run_stack(exs, wr_d, bias_d, x, T, workspace(T))
    ws = workspace(T)
    epoch = ws[4224:4228]
    epoch.copy_(torch.tensor(np.array([0xFFFFFFFD], dtype=np.uint32).view(np.uint8), device=DEV))
    ids_b, w_b, x_b = run_stack(exs, wr_d, bias_d, x, T, ws)
    np.testing.assert_array_equal(ids_a, ids_b)
    np.testing.assert_array_equal(w_a, w_b)
    np.testing.assert_array_equal(x_a, x_b)
    assert int(epoch.cpu().numpy().view(np.uint32)[0]) == 1
    _, _, x_c = run_stack(exs, wr_d, bias_d, x, T, ws)
    np.testing.assert_array_equal(x_a, x_c)
    assert int(epoch.cpu().numpy().view(np.uint32)[0]) == 1 + n
