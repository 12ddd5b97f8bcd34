"""Full-size workloads on the GPU, checked against the oracle on sampled outputs.

  config 2: 48 residual layers x 512 experts (33,973,862,400 bytes of blobs in HBM), 1 token,
            Zipf-biased routing: every layer checked with the GPU's own layer input (teacher forcing).
  config 3: one layer over 2,048 tokens, Zipf-biased routing: routing of all tokens, outputs of a sample.
  config 4: 48 residual layers over 8,192 tokens, the Zipf permutation reseeded per layer: routing and
            outputs of sampled tokens in every layer, with the GPU's own layer inputs.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
import quantized_routed_expert_top10_gb300 as qre
from gpu_common import (W_TOL, DEV, B, BlobCache, assert_equal_up_to_sum_order, check_close, check_routing,
                        device_packed_layer, run_layer, stratified_sample, to_dev, workspace)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
L = 48
E = 512


@pytest.fixture(scope="module")
def arena():
    """All 48 x 512 packed blobs of seed 0 in HBM, generated and packed layer by layer on the GPU."""
    a = torch.empty(L * E * B, dtype=torch.uint8, device=DEV)
    tmp = torch.empty(E * B, dtype=torch.uint8, device=DEV)
    for l in range(L):
        device_packed_layer(0, l, E, out=a[l * E * B:(l + 1) * E * B], tmp=tmp)
    del tmp
    torch.cuda.synchronize()
    yield a
    del a
    torch.cuda.empty_cache()


def layer_experts(arena, l):
    return qre.experts(arena[l * E * B:(l + 1) * E * B], E, 1)


def test_config2_decode_stack_48_layers(arena):
    cfg = gen.config_inputs(2)
    wr_all = np.stack(cfg["wr"])
    bias_all = np.stack(cfg["bias"])
    wr_d, bias_d = to_dev(wr_all), to_dev(bias_all)
    ws = workspace(1)
    exs = [layer_experts(arena, l) for l in range(L)]
    # one call for the whole stack
    xs = to_dev(cfg["x"])
    ids_all = torch.empty(L, 1, 10, dtype=torch.int32, device=DEV)
    qre.strata_moe_stack(exs, wr_d, bias_d, L, xs, 1, ids_all, None, ws)
    assert qre.strata_poll_status(ws) == 0
    # layer by layer, keeping every layer's input
    xl = to_dev(cfg["x"])
    ins, outs, ids = [], [], []
    for l in range(L):
        ins.append(xl.cpu().numpy())
        idl = torch.empty(1, 10, dtype=torch.int32, device=DEV)
        qre.strata_moe_layer(exs[l], wr_d[l], bias_d[l], xl, 1, qre.RESIDUAL_RMSNORM, xl, idl, None, ws)
        outs.append(xl.cpu().numpy())
        ids.append(idl.cpu().numpy())
    assert qre.strata_poll_status(ws) == 0
    np.testing.assert_array_equal(xs.cpu().numpy(), outs[-1])
    np.testing.assert_array_equal(ids_all.cpu().numpy(), np.stack(ids))
    cache = BlobCache(0)
    for l in range(L):
        r = oracle.route(ins[l], wr_all[l], bias_all[l], residual=True)
        check_routing(ids[l], r["ids"], r["logits"])
        ref = oracle.moe_layer(ins[l], wr_all[l], bias_all[l], cache.layer_list(l, ids[l]), residual=True,
                               ids_in=ids[l])
        check_close(outs[l] - ins[l], ref["out"] - ins[l].astype(np.float64), f"layer {l}")
    # end-to-end drift of the free-running oracle chain (reported, not gated)
    x = cfg["x"].copy()
    for l in range(L):
        r = oracle.route(x, wr_all[l], bias_all[l], residual=True)
        ref = oracle.moe_layer(x, wr_all[l], bias_all[l], cache.layer_list(l, r["ids"]), residual=True)
        x = ref["out"].astype(np.float32)
    drift = np.abs(outs[-1] - x).max() / np.abs(x).max()
    print(f"config 2: end-to-end relative drift of x_48 vs the free-running oracle: {drift:.3e}")


def test_config3_prefill_2048(arena):
    """All 2,048 tokens' routing; outputs of the first and last token of every prefill tile of every
    expert (every gate/up tile class and every down tile)."""
    cfg = gen.config_inputs(3)
    x, wr, bias = cfg["x"], cfg["wr"][0], cfg["bias"][0]
    out, ids, w = run_layer(arena[:E * B], wr, bias, x)
    r = oracle.route(x, wr, bias)
    ties = check_routing(ids, r["ids"], r["logits"])
    counts = np.bincount(ids.reshape(-1), minlength=E)
    sample, n_exp, per_cls = stratified_sample(ids)
    print(f"config 3: {ties} tie tokens; experts touched {np.count_nonzero(counts)}; "
          f"max/mean load {counts.max()}/{counts[counts > 0].mean():.1f}; outputs checked for {sample.size} tokens "
          f"covering {n_exp} experts and tiles {per_cls}")
    assert n_exp == np.count_nonzero(counts)
    cache = BlobCache(0)
    ref = oracle.moe_layer(x[sample], wr, bias, cache.layer_list(0, ids[sample]), ids_in=ids[sample])
    check_close(out[sample], ref["out"], "config 3 sampled outputs")
    np.testing.assert_allclose(w[sample], ref["w"], rtol=0, atol=W_TOL)


def test_config4_prefill_8192_stack_sampled(arena):
    """Every layer: routing of 256 random tokens, and outputs of 64 tokens chosen from the layer's own
    tiles (the first and last tile of each class, then experts in an order rotated per layer), with
    the GPU's own layer inputs."""
    T = 8192
    cfg = gen.config_inputs(4)
    rng = np.random.default_rng(4)
    route_sample = np.sort(rng.choice(T, 256, replace=False))
    rs = torch.from_numpy(route_sample).to(DEV)
    ws = workspace(T)
    xl = to_dev(cfg["x"])
    idl = torch.empty(T, 10, dtype=torch.int32, device=DEV)
    cache = BlobCache(0)
    ties, n_checked, experts_seen = 0, 0, set()
    for l in range(L):
        x_before = xl.clone()
        qre.strata_moe_layer(layer_experts(arena, l), to_dev(cfg["wr"][l]), to_dev(cfg["bias"][l]), xl, T,
                             qre.RESIDUAL_RMSNORM, xl, idl, None, ws)
        ids_all = idl.cpu().numpy()
        r = oracle.route(x_before[rs].cpu().numpy(), cfg["wr"][l], cfg["bias"][l], residual=True)
        ties += check_routing(ids_all[route_sample], r["ids"], r["logits"])
        sample, _, _ = stratified_sample(ids_all, budget=64, rotate=37 * l)
        st = torch.from_numpy(sample).to(DEV)
        x_in, x_out = x_before[st].cpu().numpy(), xl[st].cpu().numpy()
        ids = ids_all[sample]
        experts_seen.update((l, int(e)) for e in np.unique(ids))
        ref = oracle.moe_layer(x_in, cfg["wr"][l], cfg["bias"][l], cache.layer_list(l, ids), residual=True,
                               ids_in=ids)
        check_close(x_out - x_in, ref["out"] - x_in.astype(np.float64), f"layer {l}")
        n_checked += sample.size
        for key in [k for k in cache.cache if k[0] == l]:
            del cache.cache[key]
    assert qre.strata_poll_status(ws) == 0
    print(f"config 4: {ties} tie tokens among {256 * L} routed token-layers; outputs of {n_checked} token-layers "
          f"checked, {len(experts_seen)} (layer, expert) pairs")


@pytest.mark.parametrize("T,n_layers", [(300, 3), (8192, 2)])
def test_prefill_stack_equals_layer_chain(arena, T, n_layers):
    """strata_moe_stack for a prefill chunk (the call the long-prefill benchmark times) against the same
    layers run one strata_moe_layer call at a time.  The first layer's routing is bit-exact; the fused
    combine's fp32 additions may round differently in the two runs, so later layers see inputs that
    differ in the last bits: their routing may differ only where logits are that close (at most one
    token in a thousand), and the final activations of every token routed alike in every layer agree
    to the summation-order bound, scaled by the layers."""
    cfg = gen.config_inputs(4, T=T, L=n_layers)
    wr_d, bias_d = to_dev(np.stack(cfg["wr"])), to_dev(np.stack(cfg["bias"]))
    exs = [layer_experts(arena, l) for l in range(n_layers)]
    ws = workspace(T)
    xs = to_dev(cfg["x"])
    ids_s = torch.empty(n_layers, T, 10, dtype=torch.int32, device=DEV)
    qre.strata_moe_stack(exs, wr_d, bias_d, n_layers, xs, T, ids_s, None, ws)
    assert qre.strata_poll_status(ws) == 0
    xl = to_dev(cfg["x"])
    idl = torch.empty(T, 10, dtype=torch.int32, device=DEV)
    same = np.ones(T, dtype=bool)
    for l in range(n_layers):
        qre.strata_moe_layer(exs[l], wr_d[l], bias_d[l], xl, T, qre.RESIDUAL_RMSNORM, xl, idl, None, ws)
        a, b = ids_s[l].cpu().numpy(), idl.cpu().numpy()
        differ = np.any(a != b, axis=1)
        if l == 0:
            assert not differ.any(), "first layer routing differs"
        assert differ.sum() <= max(1, T // 1000), f"layer {l}: {differ.sum()} tokens routed differently"
        same &= ~differ
    assert qre.strata_poll_status(ws) == 0
    got, want = xs.cpu().numpy(), xl.cpu().numpy()
    assert_equal_up_to_sum_order(got[same], want[same], 10 * n_layers * np.abs(want).max(), "stack vs layer chain")
