"""Pins for the oracle's router, dispatch tables and bias update (CPU only).

Each test ties the oracle to something other than itself: a hand-worked example,
brute force over all subsets, invariants the method guarantees, or a closed form.
"""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import moe_oracle as O


def _load(golden_dir):
    with open(os.path.join(golden_dir, "hand_4x4.json")) as f:
        return json.load(f)


def test_hand_worked_route(golden_dir):
    fx = _load(golden_dir)
    ex = fx["expected"]
    r = O.route(np.array(fx["x"]), np.array(fx["w_router"]), np.array(fx["bias"]), fx["k"])
    np.testing.assert_array_equal(r["idx"], np.array(ex["idx"]))
    np.testing.assert_allclose(r["gate"], np.array(ex["gate"]), rtol=1e-6, atol=0)
    np.testing.assert_array_equal(r["boundary_tie"], np.array(ex["boundary_tie"]))
    np.testing.assert_array_equal(r["order_tie"], np.array(ex["order_tie"]))
    p = O.permutation(r["idx"], fx["E"])
    np.testing.assert_array_equal(p["counts"], ex["counts"])
    np.testing.assert_array_equal(p["offsets"], ex["offsets"])
    np.testing.assert_array_equal(p["perm_token"], ex["perm_token"])
    np.testing.assert_array_equal(p["inv_pos"], np.array(ex["inv_pos"]))
    b = O.bias_update(np.array(fx["bias"]), p["counts"], fx["T"], fx["k"], fx["gamma"])
    np.testing.assert_array_equal(b, np.array(ex["bias_after"], dtype=np.float32))


def test_hand_worked_forward(golden_dir):
    fx = _load(golden_dir)
    res = O.forward(np.array(fx["x"]), np.array(fx["w_router"]), np.array(fx["bias"]),
                    np.array(fx["w_gate_up"]), np.array(fx["w_down"]), fx["k"], fx["S"])
    np.testing.assert_allclose(res["out"], np.array(fx["expected"]["out"]), rtol=1e-6, atol=0)


def _brute_topk(v, k):
    """Best subset by the sum of biased scores, over all C(E, k) subsets."""
    E = v.shape[0]
    best, best_set = -np.inf, None
    for c in itertools.combinations(range(E), k):
        sc = float(np.sum(v[list(c)].astype(np.float64)))
        if sc > best:
            best, best_set = sc, c
    return set(best_set)


@pytest.mark.parametrize("E,k", [(5, 1), (7, 2), (9, 3), (12, 3), (12, 2)])
def test_topk_brute_force(E, k):
    rng = np.random.default_rng(E * 10 + k)
    T, d = 40, 16
    x = rng.standard_normal((T, d)).astype(np.float32)
    w = rng.standard_normal((E, d)).astype(np.float32) * 0.3
    b = rng.uniform(-0.2, 0.2, E).astype(np.float32)
    r = O.route(x, w, b, k)
    for t in range(T):
        assert set(r["idx"][t].tolist()) == _brute_topk(r["v"][t], k)
        vv = r["v"][t][r["idx"][t]]
        assert np.all(np.diff(vv) <= 0), "chosen experts must come in descending biased score"


def test_affinity_is_sigmoid_of_dot_product():
    # z for a one-hot x is the router column itself; s(0) = 1/2, s(-z) = 1 - s(z)
    E = 6
    w = np.array([[0.0], [1.0], [-1.0], [3.0], [-3.0], [0.5]], dtype=np.float32)
    x = np.ones((1, 1), dtype=np.float32)
    z = O.router_logits(x, w)
    np.testing.assert_array_equal(z[0], w[:, 0])
    s = O.affinity(z)[0]
    assert s[0] == np.float32(0.5)
    np.testing.assert_allclose(s[1] + s[2], 1.0, rtol=0, atol=1e-7)
    np.testing.assert_allclose(s[3] + s[4], 1.0, rtol=0, atol=1e-7)
    np.testing.assert_allclose(s[1], 1 / (1 + np.e ** -1), rtol=1e-7)
    assert E == s.shape[0]


def test_logit_offset_enters_before_sigmoid():
    x = np.ones((1, 1), dtype=np.float32)
    w = np.zeros((3, 1), dtype=np.float32)
    off = np.array([0.0, 2.0, -1.0], dtype=np.float32)
    r = O.route(x, w, np.zeros(3, np.float32), 2, logit_offset=off)
    np.testing.assert_array_equal(r["idx"][0], [1, 0])
    # gates follow the offset (it moves the affinity), unlike the bias
    s1, s0 = 1 / (1 + np.exp(-2.0)), 0.5
    np.testing.assert_allclose(r["gate"][0], [s1 / (s1 + s0), s0 / (s1 + s0)], rtol=1e-6)


def test_gates_sum_to_one_and_bias_changes_selection_only():
    rng = np.random.default_rng(3)
    T, d, E, k = 200, 32, 16, 4
    x = rng.standard_normal((T, d)).astype(np.float32)
    w = (rng.standard_normal((E, d)) * 0.2).astype(np.float32)
    r0 = O.route(x, w, np.zeros(E, np.float32), k)
    np.testing.assert_allclose(r0["gate"].sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(r0["gate"] > 0)
    # a bias that changes some selections
    b = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    r1 = O.route(x, w, b, k)
    same = np.all(np.sort(r0["idx"], 1) == np.sort(r1["idx"], 1), axis=1)
    assert same.any() and (~same).any()
    # where the chosen set is unchanged, gates per expert are identical (bias not in the gate)
    for t in np.nonzero(same)[0]:
        g0 = dict(zip(r0["idx"][t].tolist(), r0["gate"][t].tolist()))
        g1 = dict(zip(r1["idx"][t].tolist(), r1["gate"][t].tolist()))
        assert g0 == g1
    # the gate of a chosen expert is its unbiased affinity over the chosen sum
    t = int(np.nonzero(~same)[0][0])
    s = r1["s"][t].astype(np.float64)
    np.testing.assert_allclose(r1["gate"][t], s[r1["idx"][t]] / s[r1["idx"][t]].sum(), rtol=1e-12)


def test_ties_go_to_lower_index():
    x = np.ones((1, 1), dtype=np.float32)
    w = np.array([[0.0], [1.0], [1.0], [1.0], [0.0]], dtype=np.float32)
    r = O.route(x, w, np.zeros(5, np.float32), 2)
    np.testing.assert_array_equal(r["idx"][0], [1, 2])
    assert r["boundary_tie"][0] and r["order_tie"][0]
    r = O.route(x, w, np.zeros(5, np.float32), 4)
    np.testing.assert_array_equal(r["idx"][0], [1, 2, 3, 0])


def test_counts_offsets_and_permutation_round_trip():
    rng = np.random.default_rng(5)
    T, d, E, k = 300, 24, 10, 3
    x = rng.standard_normal((T, d)).astype(np.float32)
    w = (rng.standard_normal((E, d)) * 0.5).astype(np.float32)
    r = O.route(x, w, np.zeros(E, np.float32), k)
    p = O.permutation(r["idx"], E)
    assert p["counts"].sum() == T * k
    assert p["offsets"][0] == 0 and p["offsets"][-1] == T * k
    assert np.all(np.diff(p["offsets"]) == p["counts"])
    # every (t, j) lands in its expert's segment, tokens ascending inside a segment
    pt, inv = p["perm_token"], p["inv_pos"]
    assert sorted(inv.reshape(-1).tolist()) == list(range(T * k))
    for t in range(T):
        for j in range(k):
            pos = inv[t, j]
            e = r["idx"][t, j]
            assert pt[pos] == t
            assert p["offsets"][e] <= pos < p["offsets"][e + 1]
    for e in range(E):
        seg = pt[p["offsets"][e]:p["offsets"][e + 1]]
        assert np.all(np.diff(seg) > 0)
    xp = x[pt]
    np.testing.assert_array_equal(xp[inv.reshape(-1)], np.repeat(x, k, axis=0))


def test_bias_update_closed_form():
    T, k, E, g = 8, 2, 4, 0.001
    # mean load is T*k/E = 4; overloaded -> down, underloaded -> up, exact mean -> unchanged
    counts = np.array([6, 2, 4, 4])
    b = O.bias_update(np.zeros(E, np.float32), counts, T, k, g)
    np.testing.assert_array_equal(b, np.array([-g, g, 0.0, 0.0], dtype=np.float32))
    assert b.dtype == np.float32
    # one step from b = 0 always lands in {-g, 0, +g}
    rng = np.random.default_rng(1)
    for _ in range(20):
        E = int(rng.integers(2, 40))
        c = rng.multinomial(T * k * 3, np.ones(E) / E)
        b = O.bias_update(np.zeros(E, np.float32), c, T * 3, k, g)
        assert set(np.unique(b).tolist()) <= {np.float32(-g), 0.0, np.float32(g)}
    # n steps with a constant sign move b by n * gamma (up to float32 rounding)
    b = np.zeros(4, np.float32)
    for _ in range(20):
        b = O.bias_update(b, counts, T, k, g)
    np.testing.assert_allclose(b, [-0.02, 0.02, 0.0, 0.0], rtol=0, atol=20 * 2 ** -24 * 0.03)


def test_bias_update_is_resumable():
    # the only state is b: 10 + 10 steps equal 20 steps bit for bit
    rng = np.random.default_rng(2)
    E, T, k = 16, 64, 4
    seq = [rng.multinomial(T * k, np.ones(E) / E) for _ in range(20)]
    b = np.zeros(E, np.float32)
    for c in seq:
        b = O.bias_update(b, c, T, k)
    b2 = np.zeros(E, np.float32)
    for c in seq[:10]:
        b2 = O.bias_update(b2, c, T, k)
    saved = b2.copy()
    b3 = saved
    for c in seq[10:]:
        b3 = O.bias_update(b3, c, T, k)
    np.testing.assert_array_equal(b, b3)


def test_max_rel_err_definition():
    ref = np.array([3.0, -4.0])  # RMS = sqrt(12.5)
    out = np.array([3.5, -4.0])
    assert abs(O.max_rel_err(out, ref) - 0.5 / np.sqrt(12.5)) < 1e-15


def _brute_grouped(v, n_group, topk_group, k):
    """All group subsets of size topk_group; the best by group score, then the best
    k-subset of the experts in the kept groups (by the sum of biased scores)."""
    E = v.shape[0]
    gsz = E // n_group
    m = -(-k // topk_group)
    gscore = []
    for g in range(n_group):
        top = sorted(v[g * gsz:(g + 1) * gsz].tolist(), reverse=True)[:m]
        acc = np.float32(0)
        for t in top:
            acc = np.float32(acc + np.float32(t))
        gscore.append(float(acc))
    best_groups = max(itertools.combinations(range(n_group), topk_group), key=lambda c: sum(gscore[g] for g in c))
    allowed = [e for g in best_groups for e in range(g * gsz, (g + 1) * gsz)]
    return set(max(itertools.combinations(allowed, k), key=lambda c: sum(float(v[e]) for e in c)))


@pytest.mark.parametrize("E,n_group,topk_group,k", [(12, 4, 2, 3), (12, 3, 1, 2), (16, 4, 2, 4), (8, 2, 2, 3)])
def test_group_limited_topk_brute_force(E, n_group, topk_group, k):
    rng = np.random.default_rng(E + 7 * n_group + k)
    T, d = 30, 16
    x = rng.standard_normal((T, d)).astype(np.float32)
    w = (rng.standard_normal((E, d)) * 0.4).astype(np.float32)
    b = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    r = O.route(x, w, b, k, n_group=n_group, topk_group=topk_group)
    s_v = O.route(x, w, b, k)["v"]  # unmasked biased scores
    gsz = E // n_group
    for t in range(T):
        assert set(r["idx"][t].tolist()) == _brute_grouped(s_v[t], n_group, topk_group, k)
        assert len({e // gsz for e in r["idx"][t].tolist()}) <= topk_group


def test_group_limit_all_groups_is_plain_topk():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((50, 8)).astype(np.float32)
    w = rng.standard_normal((16, 8)).astype(np.float32)
    b = np.zeros(16, np.float32)
    a = O.route(x, w, b, 4)
    g = O.route(x, w, b, 4, n_group=4, topk_group=4)
    np.testing.assert_array_equal(a["idx"], g["idx"])
    np.testing.assert_array_equal(a["gate"], g["gate"])


def test_group_limit_changes_selection_by_hand():
    # 4 experts in 2 groups of 2, top-2 from 1 group: scores (bias only, z = 0 -> s = 0.5)
    # group 0 = {0.9, 0.0}, group 1 = {0.8, 0.7}; group scores with m = 2: 0.9 vs 1.5
    x = np.ones((1, 1), np.float32)
    w = np.zeros((4, 1), np.float32)
    b = np.array([0.4, -0.5, 0.3, 0.2], np.float32)  # v = s + b = 0.9, 0.0, 0.8, 0.7
    plain = O.route(x, w, b, 2)
    np.testing.assert_array_equal(plain["idx"][0], [0, 2])
    grp = O.route(x, w, b, 2, n_group=2, topk_group=1)
    np.testing.assert_array_equal(grp["idx"][0], [2, 3])
    np.testing.assert_allclose(grp["gate"][0], [0.5, 0.5])  # unbiased s are all 0.5
