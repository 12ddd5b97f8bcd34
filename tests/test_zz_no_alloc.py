"""strata_moe_group_noalloc -- grouping for callers that cannot allocate device memory -- against
strata_moe_group, both through the C ABI, and against the oracle's grouping.

The no-alloc entry point keeps its scratch in a fixed array inside the library (no workspace
argument), for callers that cannot call cudaMalloc.  Its results must equal the workspace entry
point's bit for bit (grouping is integer work), including on back-to-back calls that reuse the
shared array.  This file is named to be collected after every other test file.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_routed_expert_top10_gb300 as qre

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _ids(T, seed):
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, 513) ** 1.1
    p /= p.sum()
    return np.stack([rng.choice(512, 10, replace=False, p=p) for _ in range(T)]).astype(np.int32)


def _outputs(T):
    return (torch.empty(513, dtype=torch.int32, device=DEV), torch.empty(T * 10, dtype=torch.int32, device=DEV),
            torch.empty(512, dtype=torch.int32, device=DEV), torch.empty(1, dtype=torch.int32, device=DEV))


def _with_workspace(ids_d, T):
    ws = torch.empty(qre.strata_moe_workspace_bytes(T), dtype=torch.uint8, device=DEV)
    qre.strata_moe_workspace_init(ws)
    off, pair, active, na = _outputs(T)
    qre.strata_moe_group(ids_d, T, 512, off, pair, active, na, ws)
    assert qre.strata_poll_status(ws) == 0
    return off, pair, active, na


def _same(a, b):
    off_a, pair_a, act_a, na_a = (t.cpu().numpy() for t in a)
    off_b, pair_b, act_b, na_b = (t.cpu().numpy() for t in b)
    np.testing.assert_array_equal(off_a, off_b)
    np.testing.assert_array_equal(pair_a, pair_b)
    assert int(na_a[0]) == int(na_b[0])
    n = int(na_a[0])
    np.testing.assert_array_equal(act_a[:n], act_b[:n])


def test_noalloc_grouping_matches_workspace_grouping_on_two_calls_in_a_row():
    cases = [(2048, 7), (4, 8)]  # a large call, then a small one over the large call's leftovers
    ids_d = [torch.from_numpy(_ids(T, s)).to(DEV) for T, s in cases]
    refs = [_with_workspace(ids_d[i], T) for i, (T, _) in enumerate(cases)]
    outs = [_outputs(T) for T, _ in cases]
    for i, (T, _) in enumerate(cases):  # back to back on the same stream, no sync in between
        qre.strata_moe_group_noalloc(ids_d[i], T, 512, *outs[i])
    torch.cuda.synchronize()
    for ref, got in zip(refs, outs):
        _same(ref, got)


def test_noalloc_grouping_limits():
    T = qre.T_MAX
    ids_d = torch.from_numpy(_ids(T, 9)).to(DEV)
    got = _outputs(T)
    qre.strata_moe_group_noalloc(ids_d, T, 512, *got)
    _same(_with_workspace(ids_d, T), got)
    with pytest.raises(qre.StrataError):
        qre.strata_moe_group_noalloc(ids_d, T + 1, 512, *got)


@pytest.mark.parametrize("T", [1, 37, 2048])
def test_noalloc_grouping_matches_the_oracle(T):
    """Bit for bit against oracle.group: expert offsets, the stable pair order within each expert, and
    the active list in ascending expert order."""
    ids = _ids(T, 100 + T)
    got = _outputs(T)
    qre.strata_moe_group_noalloc(torch.from_numpy(ids).to(DEV), T, 512, *got)
    torch.cuda.synchronize()
    off, pair, active, na = (t.cpu().numpy() for t in got)
    ref_off, ref_pair, ref_active = oracle.group(ids, 512)
    np.testing.assert_array_equal(off, ref_off)
    np.testing.assert_array_equal(pair, ref_pair)
    assert int(na[0]) == len(ref_active)
    np.testing.assert_array_equal(active[: int(na[0])], ref_active)
