"""The routing comparison rule used by the GPU parity tests, checked on the CPU: at a
tie between a kept and a dropped group (group-limited routing) another valid choice
is accepted, and a choice that no tie explains is rejected."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from moe_testutil import check_routing, fro_err


def _group_tie_case():
    # E = 8 experts in 4 groups of 2, keep 2 groups, k = 2 (group score = best expert).
    # Token 0: groups 1 and 2 tie exactly for the second place behind group 0.
    E, k, n_group, topk_group = 8, 2, 4, 2
    z = np.array([[3.0, -2.0, 1.0, -3.0, 1.0, -3.0, -4.0, -4.0],
                  [2.0, -2.0, 0.5, -3.0, -1.0, -3.0, -4.0, 1.5]], np.float64)
    x = np.eye(2, 8)  # x . w_router[i] = z[t, i] with w_router = z^T restricted
    wr = np.zeros((E, 8))
    wr[:, 0] = z[0]
    wr[:, 1] = z[1]
    ref = O.route(x, wr, np.zeros(E, np.float32), k, n_group=n_group, topk_group=topk_group)
    return ref, E, k, n_group, topk_group


def _tensors(ref, idx, E):
    idx = np.asarray(idx, np.int32)
    s = ref["s"].astype(np.float64)
    g = np.take_along_axis(s, idx.astype(np.int64), 1)
    g = g / g.sum(1, keepdims=True)
    counts = np.bincount(idx.reshape(-1), minlength=E).astype(np.int32)
    return (torch.from_numpy(idx), torch.from_numpy(g.astype(np.float32)), torch.from_numpy(counts),
            torch.from_numpy(O.offsets_from_counts(counts)))


def test_group_tie_accepts_either_group():
    ref, E, k, ng, tg = _group_tie_case()
    assert ref["group_tie"][0] and not ref["group_tie"][1]
    assert ref["idx"][0].tolist() == [0, 2]  # the lower of the tied groups
    # the other tied group is a valid choice too
    alt = ref["idx"].copy()
    alt[0] = [0, 4]
    assert check_routing(ref, *_tensors(ref, alt, E), E, ng, tg) >= 1
    assert check_routing(ref, *_tensors(ref, ref["idx"], E), E, ng, tg) >= 1


def test_group_tie_rejects_a_worse_group():
    ref, E, k, ng, tg = _group_tie_case()
    bad = ref["idx"].copy()
    bad[0] = [0, 6]  # group 3 is far behind the tied groups
    with pytest.raises(AssertionError):
        check_routing(ref, *_tensors(ref, bad, E), E, ng, tg)
    bad[0] = [0, 3]  # a kept group, but its weaker expert
    with pytest.raises(AssertionError):
        check_routing(ref, *_tensors(ref, bad, E), E, ng, tg)


def test_fro_err():
    ref = np.array([3.0, 4.0])
    assert fro_err(np.array([3.0, 4.5]), ref) == pytest.approx(0.1)


def test_fp8_gates_tell_a_flip_from_a_tile_error():
    from moe_testutil import fp8_errs, fp8_ok
    rng = np.random.default_rng(0)
    ref = rng.standard_normal((502, 2048))
    base = ref * (1 + rng.uniform(-2 ** -9, 2 ** -9, ref.shape))  # bf16-level rounding
    # one E4M3 flip of h (a step of 0.5 sigma of h): one row moves through a column of W_down
    flip = base.copy()
    w = rng.standard_normal(2048) / np.sqrt(2048)
    flip[77] += 0.5 * w
    e = fp8_errs(flip, ref)
    assert fp8_ok(e), e
    # a 2 % scale error on one 176-token x 256-feature tile: small in Frobenius, but
    # thousands of elements beyond the bf16 bound
    tile = base.copy()
    tile[176:352, 256:512] *= 1.02
    e = fp8_errs(tile, ref)
    assert e["fro"] < 5e-3 and not fp8_ok(e), e
