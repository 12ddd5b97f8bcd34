"""The decode stack's lookahead (one layer ahead): after layer l, the workspace holds the distinct
experts that the next router, applied to layer l's normalised input, selects for the tokens -- the
experts the next layer's CTAs prefetch into L2.  Checked against the oracle's routing of the same
input with the next layer's router (up to the 1e-4 tie band).  The words are read from the decode
exchange area of the workspace, whose layout (right after the 12 KiB header) is: router dot products
[16][8][512], h [88][640], expert outputs [88][2560] (routed pairs, then a shared expert's), predicted logits [8][512], then the prediction
[1 + 80], all 64-bit (value bits, call tag) words."""
import numpy as np
import pytest
import torch

import gen
import oracle
import quantized_routed_expert_top10_gb300 as qre
from gpu_common import DEV, B, device_packed_layer, to_dev, workspace

pytestmark = pytest.mark.gpu

WS_HEADER = 12288
PRED_IDS = WS_HEADER + 8 * (16 * 8 * 512 + 88 * 640 + 88 * 2560 + 8 * 512)


@pytest.mark.parametrize("T", [1, 4])
def test_stack_lookahead_names_the_next_layers_experts(T):
    E, L = 512, 2
    cfg = gen.config_inputs(2)
    x = gen.verify_window(3, T) if T > 1 else cfg["x"]
    wr = np.stack(cfg["wr"][:L])
    bias = np.stack(cfg["bias"][:L])
    arena = torch.empty(L * E * B, dtype=torch.uint8, device=DEV)
    for l in range(L):
        device_packed_layer(0, l, E, out=arena[l * E * B:(l + 1) * E * B])
    exs = [qre.experts(arena[l * E * B:(l + 1) * E * B], E, 1) for l in range(L)]
    ws = workspace(T)
    xd = to_dev(x)
    qre.strata_moe_stack(exs, to_dev(wr), to_dev(bias), L, xd, T, None, None, ws)
    assert qre.strata_poll_status(ws) == 0
    words = ws[PRED_IDS:PRED_IDS + 8 * (1 + 80)].cpu().numpy().view(np.uint64)
    tags = (words >> np.uint64(32)).astype(np.uint32)
    vals = (words & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.int32)  # ids stored as int bits
    assert tags[0] == 1, "written by the stack's first layer (call tag 1 after workspace init)"
    D = int(vals[0])
    got = vals[1:1 + D]
    assert np.all(tags[1:1 + D] == 1)
    assert np.all(np.diff(got) > 0), "distinct, ascending"
    r = oracle.route(x, wr[1], bias[1], residual=True)
    want = np.unique(r["ids"])
    if not np.array_equal(got, want):
        # only experts inside a token's 1e-4 tie band at its 10th logit may differ
        for e in np.setxor1d(got, want):
            near = [abs(r["logits"][t][e] - np.sort(r["logits"][t])[-10]) < 1e-4 for t in range(T)]
            assert any(near), f"expert {e} is not a tie of any token"
