"""Pins for the oracle: facts the pages fix, closed forms, library routines and brute force.

Each test would fail under a plausible mistake in the oracle (wrong bit order or offset, swapped
gate/up, transposed matrices, a dropped renormalisation, wrong tie order, a missing residual)."""
import math

import numpy as np
import pytest

import gen
import oracle
from conftest import golden_path, read_golden_kv

SIZES = read_golden_kv("format_sizes.txt")


# ---------------------------------------------------------------------------------------------
# helpers: canonical blobs with chosen codes and scales
# ---------------------------------------------------------------------------------------------
def pack_codes(flat):
    c = np.asarray(flat, dtype=np.uint8).reshape(-1, 16, 4)
    return (c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)).astype(np.uint8)


def make_blob(mats, d_bits=0x3C00):
    """mats = (gate codes [FF][H], up codes [FF][H], down codes [H][FF]), values 0..3."""
    parts = []
    for m in mats:
        flat = np.asarray(m, dtype=np.uint8).reshape(-1)
        nb = flat.size // 64
        blk = np.empty((nb, 18), dtype=np.uint8)
        blk[:, 0] = d_bits & 0xFF
        blk[:, 1] = d_bits >> 8
        blk[:, 2:] = pack_codes(flat)
        parts.append(blk.reshape(-1))
    return np.concatenate(parts)


def silu(z):
    return z / (1.0 + math.exp(-z))


def selection_blob(H, FF, off, sel_code_delta=1, d_bits=0x3C00):
    sig = [(7 * r + 3) % H for r in range(FF)]
    tau = [(11 * r + 5) % H for r in range(FF)]
    rho = [(3 * n + 1) % FF for n in range(H)]
    G = np.full((FF, H), off, np.uint8)
    U = np.full((FF, H), off, np.uint8)
    D = np.full((H, FF), off, np.uint8)
    for r in range(FF):
        G[r, sig[r]] = off + sel_code_delta
        U[r, tau[r]] = off + 1
    for n in range(H):
        D[n, rho[n]] = off + 1
    return make_blob((G, U, D), d_bits), sig, tau, rho


# ---------------------------------------------------------------------------------------------
# format
# ---------------------------------------------------------------------------------------------
def test_format_sizes_from_pages():
    assert gen.blob_bytes() == SIZES["blob_bytes"] == 3 * SIZES["H"] * SIZES["FF"] * 18 // SIZES["QK"]
    assert SIZES["layers"] * SIZES["experts"] * SIZES["blob_bytes"] == SIZES["arena_bytes"]
    assert SIZES["layers"] * SIZES["top_k"] * SIZES["blob_bytes"] == SIZES["token_expert_bytes"]
    assert 18 * 8 / 64 == SIZES["bits_per_weight"]
    assert gen.blob_bytes(64, 16) == SIZES["tiny_blob_bytes"]
    assert gen.canonical_blob(0, 0, 0).size == SIZES["blob_bytes"]
    assert gen.canonical_blob(0, 0, 0, H_=64, FF_=16).size == SIZES["tiny_blob_bytes"]


def test_q2_bit_order_worked_examples():
    with open(golden_path("q2_0_bitorder.txt")) as f:
        rows = [l for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) == 4
    for row in rows:
        hexs, codes = row.split(":")
        b = np.frombuffer(bytes.fromhex(hexs.strip()), dtype=np.uint8)
        want = np.array([int(c) for c in codes.split()], dtype=np.int32)
        np.testing.assert_array_equal(oracle.q2_codes(b), want)


@pytest.mark.parametrize("off,vals", [(1, (-1.0, 0.0, 1.0, 2.0)), (2, (-2.0, -1.0, 0.0, 1.0))])
def test_code_meaning_and_scale(off, vals):
    # d = 1.0 (fp16 0x3C00), codes 0,1,2,3 repeating -> {-1,0,1,2} (pages) or the c-2 reading.
    blk = np.concatenate([np.array([0x00, 0x3C], np.uint8), np.full(16, 0xE4, np.uint8)])
    w = oracle.dequant_blocks(blk, off)
    np.testing.assert_array_equal(w, np.tile(np.array(vals), 16))
    # d = -0.5 (0xB800) scales every weight.
    blk[0:2] = [0x00, 0xB8]
    np.testing.assert_array_equal(oracle.dequant_blocks(blk, off), -0.5 * np.tile(np.array(vals), 16))


def test_fp16_and_bf16_decode_match_ieee():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(got[finite], ref[finite])
    assert np.all(np.isnan(got[np.isnan(ref)]))
    assert oracle.fp16_to_double(0x0001) == 2.0 ** -24 and oracle.fp16_to_double(0x7BFF) == 65504.0
    rng = np.random.default_rng(1)
    for b in rng.integers(0, 65536, 2000, dtype=np.uint16):
        f = np.array([int(b) << 16], dtype=np.uint32).view(np.float32)[0]
        if np.isfinite(f):
            assert oracle.bf16_to_double(int(b)) == float(f)


def test_blob_matrix_boundaries():
    """gate occupies bytes [0, 460800), up [460800, 921600), down [921600, 1382400)."""
    H, FF = 2560, 640
    zero = make_blob((np.ones((FF, H)), np.ones((FF, H)), np.ones((H, FF))))  # all codes = off 1
    for start, which in ((0, 0), (460800, 1), (921600, 2)):
        b = zero.copy()
        b[start + 2] = 0x57  # codes (3,1,1,1): first weight of that matrix -> +2, rest stay 0
        mats = oracle.dequant_blob(b, H, FF, 1)
        for m in range(3):
            nz = np.flatnonzero(mats[m])
            if m == which:
                assert list(nz) == [0] and mats[m].flat[0] == 2.0
            else:
                assert nz.size == 0
    b = zero.copy()
    b[-1] = 0xD5  # codes (1,1,1,3): weight 63 of the last block -> down[H-1][FF-1]
    g, u, d = oracle.dequant_blob(b, H, FF, 1)
    assert d[H - 1, FF - 1] == 2.0 and np.count_nonzero(d) == 1


# ---------------------------------------------------------------------------------------------
# expert FFN
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("H,FF", [(64, 16), (2560, 640)])
@pytest.mark.parametrize("off", [1, 2])
def test_expert_selection_closed_form(H, FF, off):
    blob, sig, tau, rho = selection_blob(H, FF, off)
    x = gen.activations(7, 1, H_=H)[0].astype(np.float64)
    y = oracle.expert(blob, H, FF, off, x)
    h = [silu(x[sig[r]]) * x[tau[r]] for r in range(FF)]
    want = np.array([h[rho[n]] for n in range(H)])
    np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-15)


def test_expert_negative_codes_and_scale():
    H, FF, off = 64, 16, 1
    blob, sig, tau, rho = selection_blob(H, FF, off, sel_code_delta=-1, d_bits=0x3800)  # d = 0.5
    x = gen.activations(8, 1, H_=H)[0].astype(np.float64)
    y = oracle.expert(blob, H, FF, off, x)
    # gate weight -0.5, up +0.5, down +0.5
    h = [silu(-0.5 * x[sig[r]]) * (0.5 * x[tau[r]]) for r in range(FF)]
    want = np.array([0.5 * h[rho[n]] for n in range(H)])
    np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("off", [1, 2])
def test_expert_all_offset_codes_give_zero(off):
    H, FF = 2560, 640
    blob = make_blob((np.full((FF, H), off), np.full((FF, H), off), np.full((H, FF), off)))
    x = gen.activations(3, 1)[0].astype(np.float64)
    assert np.all(oracle.expert(blob, H, FF, off, x) == 0.0)


def _numpy_expert(blob, H, FF, off, x):
    """Independent route: np.unpackbits decode + np.matmul."""
    nb = H * FF // 64
    mats = []
    for m in range(3):
        blk = blob[18 * nb * m: 18 * nb * (m + 1)].reshape(nb, 18)
        d = blk[:, 0:2].copy().view("<f2").astype(np.float64).reshape(nb)
        bits = np.unpackbits(blk[:, 2:], axis=1, bitorder="little").reshape(nb, 64, 2)
        code = bits[..., 0].astype(np.int64) + 2 * bits[..., 1]
        mats.append((d[:, None] * (code - off)).reshape(-1))
    G = mats[0].reshape(FF, H); U = mats[1].reshape(FF, H); D = mats[2].reshape(H, FF)
    g = G @ x; u = U @ x
    return D @ (g / (1.0 + np.exp(-g)) * u)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
@pytest.mark.parametrize("off", [1, 2])
def test_expert_brute_force_tiny(seed, off):
    H, FF = 64, 16
    blob = gen.canonical_blob(seed, 0, seed, H_=H, FF_=FF)
    x = gen.activations(seed, 1, H_=H)[0].astype(np.float64)
    np.testing.assert_allclose(oracle.expert(blob, H, FF, off, x), _numpy_expert(blob, H, FF, off, x),
                               rtol=1e-12, atol=1e-14)


def test_expert_full_size_matches_numpy_route():
    H, FF = 2560, 640
    blob = gen.canonical_blob(0, 0, 17)
    x = gen.activations(0, 1)[0].astype(np.float64)
    np.testing.assert_allclose(oracle.expert(blob, H, FF, 1, x), _numpy_expert(blob, H, FF, 1, x),
                               rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------------------------------------
# router and top-k
# ---------------------------------------------------------------------------------------------
def test_router_logits_one_hot_and_bias():
    wr = gen.router_weights(0, 0, E_=64, H_=128)
    bias = gen.zipf_bias(0, 0, E_=64)
    for h in (0, 5, 127):
        x = np.zeros(128); x[h] = 1.0
        l = oracle.router_logits(x, wr, bias)
        want = gen.bf16_bits_to_f32(wr[:, h]).astype(np.float64) + bias.astype(np.float64)
        np.testing.assert_array_equal(l, want)
    x = gen.activations(0, 1, H_=128)[0].astype(np.float64)
    np.testing.assert_array_equal(oracle.router_logits(4.0 * x, wr), 4.0 * oracle.router_logits(x, wr))
    dense = gen.bf16_bits_to_f32(wr).astype(np.float64) @ x
    np.testing.assert_allclose(oracle.router_logits(x, wr), dense, rtol=1e-12, atol=1e-14)


def test_zipf_bias_is_a_rank_prior():
    b = gen.zipf_bias(0, 0).astype(np.float64)
    ranks = np.rint(np.expm1(-b / 1.1)).astype(np.int64)
    assert sorted(ranks.tolist()) == list(range(512))


def test_top_k_closed_form_log_logits():
    # logits ln(1..8): p_i = (i+1)/36; top-2 = experts 7, 6; renormalised 8/15, 7/15.
    l = np.log(np.arange(1, 9, dtype=np.float64))
    ids, w, p = oracle.top_k(l, 2)
    assert list(ids) == [7, 6]
    np.testing.assert_allclose(w, [8 / 15, 7 / 15], rtol=1e-15)
    np.testing.assert_allclose(p, np.arange(1, 9) / 36.0, rtol=1e-14)


def test_top_k_all_equal_takes_lowest_ids():
    ids, w, _ = oracle.top_k(np.full(512, 0.25), 10)
    assert list(ids) == list(range(10))
    np.testing.assert_allclose(w, 0.1, rtol=1e-15)


def test_top_k_ties_keep_lower_id_first():
    l = np.array([1.0, 3.0, 3.0, 2.0, 3.0, 0.0])
    ids, w, _ = oracle.top_k(l, 4)
    assert list(ids) == [1, 2, 4, 3]
    np.testing.assert_allclose(w[:3], w[0])


def test_top_k_dominant_logit():
    l = np.zeros(512); l[300] = 50.0
    ids, w, _ = oracle.top_k(l, 10)
    assert ids[0] == 300 and list(ids[1:]) == list(range(9))
    assert abs(w[0] - 1.0) < 1e-20 + 9 * math.exp(-50) * 1.01
    np.testing.assert_allclose(w[1:], math.exp(-50) / (1 + 9 * math.exp(-50)), rtol=1e-12)


def test_top_k_brute_force_subsets():
    import itertools
    rng = np.random.default_rng(5)
    for _ in range(200):
        l = rng.normal(size=8)
        ids, w, p = oracle.top_k(l, 2)
        best = max(itertools.combinations(range(8), 2), key=lambda s: (p[s[0]] + p[s[1]]))
        assert set(ids) == set(best)
        assert p[ids[0]] >= p[ids[1]]
        np.testing.assert_allclose(w, p[ids] / p[ids].sum(), rtol=1e-14)


def test_top_k_invariants_on_router_scale():
    wr = gen.router_weights(0, 0)
    x = gen.activations_fast(0, 16)
    for t in range(16):
        l = oracle.router_logits(x[t].astype(np.float64), wr)
        ids, w, p = oracle.top_k(l, 10)
        assert len(set(ids.tolist())) == 10
        assert np.all(w > 0) and np.all(np.diff(w) <= 0)
        assert abs(w.sum() - 1.0) < 1e-12
        assert p[ids].sum() >= 10 / 512  # the 2^-14 clamp can never bind
        assert np.all(p[ids].min() >= np.delete(p, ids))


def test_weights_for_ids_matches_top_k():
    l = np.random.default_rng(3).normal(size=512)
    ids, w, p = oracle.top_k(l, 10)
    np.testing.assert_allclose(oracle.weights_for_ids(l, ids), w, rtol=1e-15)
    perm = ids[::-1].copy()
    np.testing.assert_allclose(oracle.weights_for_ids(l, perm), w[::-1], rtol=1e-15)


def _dense_route(x, wr, bias, residual, K):
    """Independent route: rmsnorm and logits with numpy in float64, then a stable descending argsort of
    the softmax (the first K), renormalised."""
    xd = x.astype(np.float64)
    if residual:
        xd = xd / np.sqrt(np.mean(xd * xd, axis=1, keepdims=True) + 1e-6)
    l = xd @ gen.bf16_bits_to_f32(wr).astype(np.float64).T
    if bias is not None:
        l = l + bias.astype(np.float64)
    p = np.exp(l - l.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    ids = np.argsort(-p, axis=1, kind="stable")[:, :K]
    w = np.take_along_axis(p, ids, axis=1)
    return ids, w / w.sum(axis=1, keepdims=True), l


@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("H,E,K,T", [(64, 8, 2, 6), (2560, 512, 10, 2)])
def test_route_tokens_against_numpy(H, E, K, T, residual, with_bias):
    """oracle.route (the routing every GPU check compares with): rmsnorm on residual layers, the bias
    added, and the top-K of the softmax, against a dense numpy evaluation.  x is scaled by 3 so a
    dropped rmsnorm changes the logits."""
    x = (3.0 * gen.activations(H + T, T, H_=H)).astype(np.float32)
    wr = gen.router_weights(1, 0, E_=E, H_=H)
    bias = gen.zipf_bias(1, 0, E_=E) if with_bias else None
    r = oracle.route(x, wr, bias, residual=residual, K=K)
    ids, w, l = _dense_route(x, wr, bias, residual, K)
    np.testing.assert_allclose(r["logits"], l, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(r["ids"], ids)
    np.testing.assert_allclose(r["w"], w, rtol=1e-12)


@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("with_bias", [False, True])
def test_route_tokens_equal_the_layer_routing(residual, with_bias):
    """oracle.route and the routing inside oracle.moe_layer are separate code: the same bits."""
    H, E, FF, K, T = 64, 8, 16, 2, 7
    x, wr, blobs = _tiny_layer_inputs(T)
    x = (2.5 * x).astype(np.float32)
    bias = gen.zipf_bias(0, 0, E_=E) if with_bias else None
    r = oracle.route(x, wr, bias, residual=residual, K=K)
    m = oracle.moe_layer(x, wr, bias, blobs, K=K, residual=residual)
    np.testing.assert_array_equal(r["ids"], m["ids"])
    np.testing.assert_array_equal(r["w"], m["w"])
    np.testing.assert_array_equal(r["logits"], m["logits"])


def test_route_one_hot_gives_the_router_column_plus_bias():
    wr = gen.router_weights(0, 0, E_=64, H_=128)
    bias = gen.zipf_bias(0, 0, E_=64)
    x = np.zeros((3, 128), dtype=np.float32)
    cols = (0, 77, 127)
    for t, h in enumerate(cols):
        x[t, h] = 1.0
    r = oracle.route(x, wr, bias, K=10)
    for t, h in enumerate(cols):
        want = gen.bf16_bits_to_f32(wr[:, h]).astype(np.float64) + bias.astype(np.float64)
        np.testing.assert_array_equal(r["logits"][t], want)
    # residual: rmsnorm of a one-hot vector is the one-hot vector times 1/sqrt(1/H + 1e-6)
    r = oracle.route(x, wr, None, residual=True, K=10)
    s = 1.0 / math.sqrt(1.0 / 128 + 1e-6)
    for t, h in enumerate(cols):
        np.testing.assert_allclose(r["logits"][t], gen.bf16_bits_to_f32(wr[:, h]).astype(np.float64) * s,
                                   rtol=1e-14, atol=0)


# ---------------------------------------------------------------------------------------------
# grouping
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1, 4, 37, 300])
def test_group_is_stable_counting_sort(T):
    rng = np.random.default_rng(T)
    ids = np.stack([rng.choice(512, 10, replace=False) for _ in range(T)]).astype(np.int32)
    off, pair, active = oracle.group(ids, 512)
    flat = ids.reshape(-1)
    np.testing.assert_array_equal(pair, np.argsort(flat, kind="stable"))
    np.testing.assert_array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=512))]))
    np.testing.assert_array_equal(active, np.unique(flat))
    assert off[-1] == T * 10 and np.all(np.diff(off) >= 0)


# ---------------------------------------------------------------------------------------------
# layer, combine, residual stack
# ---------------------------------------------------------------------------------------------
def _tiny_layer_inputs(T, E=8, H=64, FF=16, seed=0):
    x = gen.activations(seed, T, H_=H)
    wr = gen.router_weights(seed, 0, E_=E, H_=H)
    blobs = [gen.canonical_blob(seed, 0, e, H_=H, FF_=FF) for e in range(E)]
    return x, wr, blobs


def test_layer_top1_is_the_expert_itself():
    x, wr, blobs = _tiny_layer_inputs(3)
    r = oracle.moe_layer(x, wr, None, blobs, K=1, want_parts=True)
    for t in range(3):
        e = r["ids"][t, 0]
        y = oracle.expert(blobs[e], 64, 16, 1, x[t].astype(np.float64))
        assert r["w"][t, 0] == 1.0
        np.testing.assert_array_equal(r["out"][t], y)


def test_layer_combine_is_weighted_sum_in_k_order():
    x, wr, blobs = _tiny_layer_inputs(5)
    r = oracle.moe_layer(x, wr, None, blobs, K=2, want_parts=True)
    for t in range(5):
        ys = [oracle.expert(blobs[e], 64, 16, 1, x[t].astype(np.float64)) for e in r["ids"][t]]
        np.testing.assert_array_equal(r["parts"][t, 0], ys[0])
        np.testing.assert_array_equal(r["parts"][t, 1], ys[1])
        np.testing.assert_array_equal(r["out"][t], 0.0 + r["w"][t, 0] * ys[0] + r["w"][t, 1] * ys[1])
        l = oracle.router_logits(x[t].astype(np.float64), wr)
        ids, w, _ = oracle.top_k(l, 2)
        np.testing.assert_array_equal(ids, r["ids"][t])


def test_layer_teacher_forced_one_hot_weights():
    x, wr, blobs = _tiny_layer_inputs(2)
    # Forcing the same id twice makes both weights 1/2: out = y.
    forced = np.array([[4, 4], [1, 1]], dtype=np.int32)
    r = oracle.moe_layer(x, wr, None, blobs, K=2, ids_in=forced)
    for t in range(2):
        y = oracle.expert(blobs[forced[t, 0]], 64, 16, 1, x[t].astype(np.float64))
        np.testing.assert_allclose(r["out"][t], y, rtol=1e-15, atol=1e-300)
        np.testing.assert_array_equal(r["w"][t], [0.5, 0.5])


def test_residual_with_zero_experts_is_identity():
    H, FF, E = 64, 16, 8
    x = gen.activations(2, 4, H_=H)
    wr = gen.router_weights(2, 0, E_=E, H_=H)
    zero = make_blob((np.ones((FF, H)), np.ones((FF, H)), np.ones((H, FF))))
    r = oracle.moe_layer(x, wr, None, [zero] * E, K=2, residual=True)
    np.testing.assert_array_equal(r["out"], x.astype(np.float64))


def test_residual_layer_routes_on_normalised_input():
    x, wr, blobs = _tiny_layer_inputs(3)
    r = oracle.moe_layer(3.0 * x, wr, None, blobs, K=2, residual=True)
    r1 = oracle.moe_layer(x, wr, None, blobs, K=2, residual=True)
    # rmsnorm removes the scale: routing and the MoE part are (nearly) unchanged, only x scales.
    np.testing.assert_array_equal(r["ids"], r1["ids"])
    np.testing.assert_allclose(r["out"] - 3.0 * x, r1["out"] - x, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("H,FF", [(64, 16), (2560, 640)])
def test_shared_expert_closed_form_through_the_layer(H, FF, residual):
    """Routed experts whose codes all equal the offset contribute nothing, so the layer's output is the
    shared expert alone: a selection matrix's closed form on the (normalised) input, plus x when
    residual."""
    E, K, T, off = 8, 2, 3, 1
    zero = make_blob((np.full((FF, H), off), np.full((FF, H), off), np.full((H, FF), off)))
    shared, sig, tau, rho = selection_blob(H, FF, off)
    x = (2.0 * gen.activations(11, T, H_=H)).astype(np.float32)
    wr = gen.router_weights(3, 0, E_=E, H_=H)
    r = oracle.moe_layer(x, wr, None, [zero] * E, K=K, residual=residual, shared=shared)
    for t in range(T):
        xd = x[t].astype(np.float64)
        xn = xd / math.sqrt(np.mean(xd * xd) + 1e-6) if residual else xd
        h = [silu(xn[sig[q]]) * xn[tau[q]] for q in range(FF)]
        want = np.array([h[rho[n]] for n in range(H)]) + (xd if residual else 0.0)
        np.testing.assert_allclose(r["out"][t], want, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("residual", [False, True])
def test_shared_expert_adds_its_output_with_weight_one(residual):
    """The layer with a shared expert minus the same layer without it is that expert on the routed
    experts' input (rmsnorm(x) for residual layers), unweighted; routing is unchanged."""
    T, E, H, FF = 5, 8, 64, 16
    x, wr, blobs = _tiny_layer_inputs(T)
    x = (3.0 * x).astype(np.float32)
    shared = gen.canonical_blob(9, 0, 99, H_=H, FF_=FF)
    a = oracle.moe_layer(x, wr, None, blobs, K=2, residual=residual, shared=shared)
    b = oracle.moe_layer(x, wr, None, blobs, K=2, residual=residual)
    np.testing.assert_array_equal(a["ids"], b["ids"])
    for t in range(T):
        xd = x[t].astype(np.float64)
        xn = xd / math.sqrt(np.mean(xd * xd) + 1e-6) if residual else xd
        y = _numpy_expert(shared, H, FF, 1, xn)
        np.testing.assert_allclose(a["out"][t] - b["out"][t], y, rtol=1e-9, atol=1e-12)


def test_rmsnorm_mean_square():
    x = gen.activations(4, 1)[0].astype(np.float64) * 7.0
    xn = oracle.rmsnorm(x)
    ms = np.mean(x * x)
    assert abs(np.mean(xn * xn) - ms / (ms + 1e-6)) < 1e-14
    np.testing.assert_allclose(xn / x, xn[0] / x[0], rtol=1e-14)


def test_layer_independent_of_thread_count():
    x, wr, blobs = _tiny_layer_inputs(9)
    a = oracle.moe_layer(x, wr, None, blobs, K=2, n_threads=1)
    b = oracle.moe_layer(x, wr, None, blobs, K=2, n_threads=4)
    np.testing.assert_array_equal(a["out"], b["out"])
    np.testing.assert_array_equal(a["ids"], b["ids"])


# ---------------------------------------------------------------------------------------------
# input generator (not the oracle, but both sides depend on it)
# ---------------------------------------------------------------------------------------------
def test_philox_known_answers():
    with open(golden_path("philox4x32_10_kat.txt")) as f:
        rows = [l for l in f if l.strip() and not l.startswith("#")]
    for row in rows:
        a, b = row.split(":")
        ins = [int(v, 16) for v in a.split()]
        want = [int(v, 16) for v in b.split()]
        got = gen.philox4x32_10(*ins)
        assert [int(g) for g in got] == want


def test_generator_distributions():
    x = gen.activations_fast(0, 64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    w = gen.bf16_bits_to_f32(gen.router_weights(0, 0))
    assert abs(w.std() - 0.02) < 2e-4
    b = gen.canonical_blob(0, 1, 2)
    d = b.reshape(-1, 18)[:, :2].copy().view("<f2").astype(np.float64)
    assert np.all(d >= 0) and abs(np.sqrt(np.mean(d * d)) - 0.02) < 2e-4
    codes = np.unpackbits(b.reshape(-1, 18)[:, 2:], bitorder="little")
    assert abs(codes.mean() - 0.5) < 0.01
    v = gen.verify_window(0)
    c = np.corrcoef(v)
    assert np.all(c > 0.9)
