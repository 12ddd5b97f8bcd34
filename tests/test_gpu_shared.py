"""GPU parity of the layer's shared expert (strata_experts_t.shared_blob) against the oracle.

Reading (the pages name a shared expert that runs for every token but give neither its width nor a
gate): an expert of the routed experts' shape and Q2_0 format whose output on the routed experts' input
is added with weight 1 to their weighted sum, before the residual.  Decode (one kernel for T <= 8) and
prefill (the tensor-core path, T > 8) both carry it as one more expert over every token."""
import numpy as np
import pytest
import torch

import gen
import oracle
import quantized_routed_expert_top10_gb300 as qre
from gpu_common import (DEV, B, BlobCache, check_close, check_routing, device_canonical, device_packed_layer, to_dev,
                        workspace)

pytestmark = pytest.mark.gpu
SHARED_ID = 512  # the generator's expert index for a layer's shared expert (past the routed ones)


def packed_shared(layer):
    canon = device_canonical(0, layer, SHARED_ID, 1)
    out = torch.empty(B, dtype=torch.uint8, device=DEV)
    qre.strata_pack_q2_0_device(canon, B, out, B, 1)
    return out


@pytest.fixture(scope="module")
def layers():
    blobs = [device_packed_layer(0, l) for l in range(2)]
    shared = [packed_shared(l) for l in range(2)]
    yield blobs, shared, BlobCache(0)
    del blobs, shared
    torch.cuda.empty_cache()


def layer_call(blobs, shared, wr, bias, x, flags):
    T = x.shape[0]
    ws = workspace(T)
    out = torch.empty(T, qre.H, dtype=torch.float32, device=DEV)
    ids = torch.empty(T, qre.K, dtype=torch.int32, device=DEV)
    ex = qre.experts(blobs, shared=shared)
    qre.strata_moe_layer(ex, to_dev(wr), None if bias is None else to_dev(bias), to_dev(x), T, flags, out, ids, None, ws)
    assert qre.strata_poll_status(ws) == 0
    return out.cpu().numpy(), ids.cpu().numpy()


@pytest.mark.parametrize("T", [1, 4, 8, 9, 37, 300])
@pytest.mark.parametrize("flags", [0, 1])
def test_layer_with_shared_expert(layers, T, flags):
    blobs, shared, cache = layers
    x = (gen.activations_fast(50 + T, T) * (2.0 if flags else 1.0)).astype(np.float32)
    wr, bias = gen.router_weights(0, 0), gen.zipf_bias(0, 0)
    out, ids = layer_call(blobs[0], shared[0], wr, bias, x, flags)
    r = oracle.route(x, wr, bias, residual=bool(flags))
    check_routing(ids, r["ids"], r["logits"])
    ref = oracle.moe_layer(x, wr, bias, cache.layer_list(0, ids), residual=bool(flags), ids_in=ids,
                           shared=cache.get(0, SHARED_ID))
    if flags:
        check_close(out - x, ref["out"] - x.astype(np.float64), f"T={T} residual layer with shared expert")
    else:
        check_close(out, ref["out"], f"T={T} layer with shared expert")
    # and the shared expert's contribution is really there: without it the output differs by about it
    out0, _ = layer_call(blobs[0], None, wr, bias, x, flags)
    base = oracle.moe_layer(x, wr, bias, cache.layer_list(0, ids), residual=bool(flags), ids_in=ids)
    check_close(out - out0, ref["out"] - base["out"], f"T={T} shared expert's part")


@pytest.mark.parametrize("T", [1, 20])
def test_stack_with_shared_experts(layers, T):
    """Two residual layers, each with its own shared expert, in one strata_moe_stack call: every layer
    against the oracle with the GPU's own layer input (the layers run one call at a time for that)."""
    blobs, shared, cache = layers
    L = 2
    wr = np.stack([gen.router_weights(0, l) for l in range(L)])
    bias = np.stack([gen.zipf_bias(0, l) for l in range(L)])
    exs = [qre.experts(blobs[l], shared=shared[l]) for l in range(L)]
    x = gen.activations_fast(70, T)
    ws = workspace(T)
    xs = to_dev(x)
    qre.strata_moe_stack(exs, to_dev(wr), to_dev(bias), L, xs, T, None, None, ws)
    assert qre.strata_poll_status(ws) == 0
    xl = to_dev(x)
    idl = torch.empty(T, qre.K, dtype=torch.int32, device=DEV)
    for l in range(L):
        x_in = xl.cpu().numpy()
        qre.strata_moe_layer(exs[l], to_dev(wr[l]), to_dev(bias[l]), xl, T, qre.RESIDUAL_RMSNORM, xl, idl, None, ws)
        ids = idl.cpu().numpy()
        ref = oracle.moe_layer(x_in, wr[l], bias[l], cache.layer_list(l, ids), residual=True, ids_in=ids,
                               shared=cache.get(l, SHARED_ID))
        check_close(xl.cpu().numpy() - x_in, ref["out"] - x_in.astype(np.float64), f"layer {l}")
    assert qre.strata_poll_status(ws) == 0
    got, want = xs.cpu().numpy(), xl.cpu().numpy()
    scale = np.abs(want - x).max()
    assert np.abs(got - want).max() <= 1e-4 * scale, "stack and layer chain disagree"


@pytest.mark.parametrize("T", [4, 64])
def test_host_call_tells_shared_from_plain(layers, T):
    """The host-buffer call's graph cache keys on the descriptor's shared expert too: the same buffers
    with and without it give the two different results."""
    blobs, shared, _ = layers
    wr = to_dev(gen.router_weights(0, 0))
    ws = workspace(T)
    s = torch.cuda.Stream()
    hx = torch.from_numpy(gen.activations_fast(80, T)).pin_memory()
    ho = torch.empty_like(hx).pin_memory()
    res = []
    for sh in (shared[0], None, shared[0]):
        qre.strata_moe_layer_host(qre.experts(blobs[0], shared=sh), wr, None, hx, T, 0, ho, None, None, ws, stream=s)
        res.append(ho.numpy().copy())
    xd = hx.to(DEV)
    want = []
    for sh in (shared[0], None):
        out = torch.empty_like(xd)
        qre.strata_moe_layer(qre.experts(blobs[0], shared=sh), wr, None, xd, T, 0, out, None, None, ws)
        want.append(out.cpu().numpy())
    tol = 1e-5 * np.abs(want[0]).max()
    assert np.abs(res[0] - want[0]).max() <= tol and np.abs(res[2] - want[0]).max() <= tol
    assert np.abs(res[1] - want[1]).max() <= tol
    assert np.abs(res[0] - res[1]).max() > 100 * tol
