"""GPU parity of the separate steps (route, group, experts, combine), the device generator and the
device packer, through the C ABI."""
import numpy as np
import pytest
import torch

import gen
import oracle
import quantized_routed_expert_top10_gb300 as qre
from gpu_common import (W_TOL, LOGIT_TOL, DEV, B, BlobCache, check_close, check_routing, device_canonical, device_packed_layer,
                        host_packed, to_dev, workspace)

pytestmark = pytest.mark.gpu


def test_device_generator_matches_host_generator():
    for layer, e in ((0, 0), (3, 77), (47, 511)):
        d = device_canonical(0, layer, e, 1).cpu().numpy()
        np.testing.assert_array_equal(d, gen.canonical_blob(0, layer, e))


def test_device_pack_matches_host_pack():
    canon = [gen.canonical_blob(1, 0, e) for e in range(3)]
    host = host_packed(canon).cpu().numpy()
    src = to_dev(np.concatenate(canon))
    dst = torch.empty_like(src)
    qre.strata_pack_q2_0_device(src, B, dst, B, 3)
    np.testing.assert_array_equal(dst.cpu().numpy(), host)


@pytest.mark.parametrize("T", [1, 4, 8, 64, 1000])
def test_route_step(T):
    x = gen.activations_fast(21, T)
    wr = gen.router_weights(0, 0)
    bias = gen.zipf_bias(0, 0) if T > 4 else None
    ws = workspace(T)
    ids = torch.empty(T, 10, dtype=torch.int32, device=DEV)
    w = torch.empty(T, 10, dtype=torch.float32, device=DEV)
    logits = torch.empty(T, 512, dtype=torch.float32, device=DEV)
    qre.strata_moe_route(to_dev(x), T, to_dev(wr), None if bias is None else to_dev(bias), 512, ids, w, logits, ws)
    assert qre.strata_poll_status(ws) == 0
    ref = oracle.route(x, wr, bias)
    # decode GEMV: fp32 FFMA; prefill: tensor-core GEMM with bf16 hi/lo parts of x (see gpu_common)
    np.testing.assert_allclose(logits.cpu().numpy(), ref["logits"], rtol=0, atol=2e-5 if T <= 8 else LOGIT_TOL)
    ids_h = ids.cpu().numpy()
    check_routing(ids_h, ref["ids"], ref["logits"])
    wref = np.stack([oracle.weights_for_ids(ref["logits"][t], ids_h[t]) for t in range(T)])
    np.testing.assert_allclose(w.cpu().numpy(), wref, rtol=0, atol=W_TOL)


@pytest.mark.parametrize("E", [32, 256])
def test_route_smaller_expert_counts(E):
    T = 6
    x = gen.activations_fast(22, T)
    wr = gen.router_weights(0, 0, E_=E)
    ws = workspace(T)
    ids = torch.empty(T, 10, dtype=torch.int32, device=DEV)
    w = torch.empty(T, 10, dtype=torch.float32, device=DEV)
    qre.strata_moe_route(to_dev(x), T, to_dev(wr), None, E, ids, w, None, ws)
    ref = oracle.route(x, wr)
    check_routing(ids.cpu().numpy(), ref["ids"], ref["logits"])


def _random_ids(T, seed, skew=True):
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, 513) ** 1.1 if skew else np.ones(512)
    p /= p.sum()
    return np.stack([rng.choice(512, 10, replace=False, p=p) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T", [1, 4, 8, 100, 2048, 8192])
def test_group_step_bit_exact(T):
    ids = _random_ids(T, T)
    ws = workspace(T)
    off = torch.empty(513, dtype=torch.int32, device=DEV)
    pair = torch.empty(T * 10, dtype=torch.int32, device=DEV)
    active = torch.empty(512, dtype=torch.int32, device=DEV)
    na = torch.empty(1, dtype=torch.int32, device=DEV)
    qre.strata_moe_group(to_dev(ids), T, 512, off, pair, active, na, ws)
    assert qre.strata_poll_status(ws) == 0
    r_off, r_pair, r_active = oracle.group(ids, 512)
    np.testing.assert_array_equal(off.cpu().numpy(), r_off)
    np.testing.assert_array_equal(pair.cpu().numpy(), r_pair)
    n = int(na.item())
    assert n == r_active.size
    np.testing.assert_array_equal(active.cpu().numpy()[:n], r_active)


def test_group_invalid_id_sets_corrupt_status():
    T = 4
    ids = _random_ids(T, 1)
    ids[2, 3] = 700
    ws = workspace(T)
    off = torch.empty(513, dtype=torch.int32, device=DEV)
    pair = torch.empty(T * 10, dtype=torch.int32, device=DEV)
    active = torch.empty(512, dtype=torch.int32, device=DEV)
    na = torch.empty(1, dtype=torch.int32, device=DEV)
    qre.strata_moe_group(to_dev(ids), T, 512, off, pair, active, na, ws)
    assert qre.strata_poll_status(ws) == -7
    assert int(off[512].item()) == T * 10 - 1  # the bad pair is dropped
    qre.strata_clear_status(ws)
    assert qre.strata_poll_status(ws) == 0


@pytest.fixture(scope="module")
def layer0():
    blobs = device_packed_layer(0, 0)
    yield blobs, BlobCache(0)
    del blobs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("bad", ["duplicate_active", "overlapping_ranges", "descending_active"])
def test_experts_reject_inconsistent_grouping(layer0, bad):
    """A caller's grouping whose active list repeats an expert, runs backwards, or whose slot ranges
    overlap would make the tile list run past the workspace's padded rows: the device check finds it
    before any expert work, sets STRATA_E_CORRUPT and the call leaves parts untouched."""
    blobs, _ = layer0
    T = 12
    ids = _random_ids(T, 7, skew=False)
    off, pair, active = oracle.group(ids, 512)
    off, active = off.copy(), active.copy()
    na = active.size
    if bad == "duplicate_active":
        active = np.concatenate([active[:1], active])[:512].astype(np.int32)
        na = min(na + 1, 512)
    elif bad == "descending_active":
        active = active[::-1].copy()
    else:  # an active expert's range is stretched into the next active expert's
        i = int(np.flatnonzero(np.diff(active) > 1)[0])
        off[int(active[i]) + 1] = off[int(active[i + 1])] + 1
    ws = workspace(T)
    parts = torch.full((T, 10, qre.H), 3.5, dtype=torch.float32, device=DEV)
    act = torch.zeros(512, dtype=torch.int32, device=DEV)
    act[:active.size] = to_dev(active.astype(np.int32))
    qre.strata_moe_experts(qre.experts(blobs), to_dev(gen.activations_fast(3, T)), T, to_dev(off), to_dev(pair), act,
                           to_dev(np.array([na], dtype=np.int32)), parts, ws)
    assert qre.strata_poll_status(ws) == -7
    assert bool(torch.all(parts == 3.5))
    qre.strata_clear_status(ws)
    assert qre.strata_poll_status(ws) == 0


@pytest.mark.parametrize("T", [4, 37])
def test_experts_and_combine_steps(layer0, T):
    blobs, cache = layer0
    x = gen.activations_fast(31, T)
    wr = gen.router_weights(0, 0)
    bias = gen.zipf_bias(0, 0)
    ws = workspace(T)
    xd = to_dev(x)
    ids = torch.empty(T, 10, dtype=torch.int32, device=DEV)
    w = torch.empty(T, 10, dtype=torch.float32, device=DEV)
    qre.strata_moe_route(xd, T, to_dev(wr), to_dev(bias), 512, ids, w, None, ws)
    off = torch.empty(513, dtype=torch.int32, device=DEV)
    pair = torch.empty(T * 10, dtype=torch.int32, device=DEV)
    active = torch.empty(512, dtype=torch.int32, device=DEV)
    na = torch.empty(1, dtype=torch.int32, device=DEV)
    qre.strata_moe_group(ids, T, 512, off, pair, active, na, ws)
    parts = torch.empty(T, 10, qre.H, dtype=torch.float32, device=DEV)
    qre.strata_moe_experts(qre.experts(blobs), xd, T, off, pair, active, na, parts, ws)
    assert qre.strata_poll_status(ws) == 0
    ids_h = ids.cpu().numpy()
    ref = oracle.moe_layer(x, wr, bias, cache.layer_list(0, ids_h), ids_in=ids_h, want_parts=True)
    parts_h = parts.cpu().numpy()
    for t in range(T):
        for k in range(10):
            check_close(parts_h[t, k], ref["parts"][t, k], f"parts[{t}][{k}]")
    # combine fed with the oracle's parts and weights
    out = torch.empty(T, qre.H, dtype=torch.float32, device=DEV)
    qre.strata_moe_combine(to_dev(ref["parts"].astype(np.float32)), to_dev(ref["w"].astype(np.float32)), T, None, out)
    check_close(out.cpu().numpy(), ref["out"], "combine")
    # combine with a residual, in place
    res = to_dev(x)
    qre.strata_moe_combine(to_dev(ref["parts"].astype(np.float32)), to_dev(ref["w"].astype(np.float32)), T, res, res)
    check_close(res.cpu().numpy() - x, ref["out"], "combine + residual")
